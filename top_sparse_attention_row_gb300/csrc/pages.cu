// Touched-page mark and masked page split ("[SM120] Only split touched SWA pages in FlashMLA
// page-split kernel", Modifications): a decode step reads only the pages its sparse indices
// reference, so a pass that re-lays the KV pool from one page size to a smaller one copies only
// those pages.
//  * page_mark_kernel: one thread per index element; every valid token slot t sets
//    mark[t / src_page_size] = 1.  Threads that mark the same page store the same byte, so no
//    atomic is needed.
//  * page_split_kernel: one CTA per source page (a fixed grid of n_src_pages, so the launch
//    shape does not depend on the indices and a captured graph replays it).  A CTA whose page is
//    unmarked returns after a one-byte load; otherwise it copies every sub-page of every section
//    with 16-byte loads and stores, four in flight per thread.
// Page layout (both pools): a page of P tokens holds its sections one after another, section k
// being P x section_bytes[k] bytes, token-major inside the section.  Destination page
// p * ratio + i holds source tokens i * dst_page_size .. (i + 1) * dst_page_size - 1 of source
// page p.  Nothing is read back to the host.
#include <cstdint>

#include "internal.h"

namespace qsa {
namespace {

constexpr int kMarkThreads = 256;
constexpr int kSplitThreads = 256;

__global__ void __launch_bounds__(kMarkThreads)
    page_mark_kernel(const int32_t* __restrict__ indices, int64_t n_indices, int32_t src_page_size,
                     int64_t n_src_pages, uint8_t* __restrict__ mark) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_indices;
       e += stride) {
    const int32_t t = __ldg(indices + e);
    if (t < 0) continue;
    const int64_t page = t / src_page_size;
    if (page < n_src_pages) mark[page] = 1;
  }
}

__global__ void __launch_bounds__(kSplitThreads)
    page_split_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                      const uint8_t* __restrict__ mark, int32_t ratio, int32_t dst_page_size,
                      PageSections sec) {
  const int64_t p = blockIdx.x;                       // source page
  if (mark != nullptr && __ldg(mark + p) == 0) return;
  const int64_t dst_page_bytes = static_cast<int64_t>(dst_page_size) * sec.token_bytes;
  const uint8_t* sp = src + p * ratio * dst_page_bytes;
  int64_t src_off = 0, dst_off = 0;
  for (int k = 0; k < sec.n; ++k) {
    const int64_t run = static_cast<int64_t>(dst_page_size) * sec.bytes[k];   // one sub-page
    const int64_t n16 = run / 16;
    for (int i = 0; i < ratio; ++i) {
      // sub-page i of section k: contiguous in both pools
      const uint4* s4 = reinterpret_cast<const uint4*>(sp + src_off + i * run);
      uint4* d4 = reinterpret_cast<uint4*>(dst + (p * ratio + i) * dst_page_bytes + dst_off);
      int64_t e = threadIdx.x;
      for (; e + 3 * kSplitThreads < n16; e += 4 * kSplitThreads) {
        const uint4 a0 = __ldg(s4 + e), a1 = __ldg(s4 + e + kSplitThreads);
        const uint4 a2 = __ldg(s4 + e + 2 * kSplitThreads), a3 = __ldg(s4 + e + 3 * kSplitThreads);
        d4[e] = a0;
        d4[e + kSplitThreads] = a1;
        d4[e + 2 * kSplitThreads] = a2;
        d4[e + 3 * kSplitThreads] = a3;
      }
      for (; e < n16; e += kSplitThreads) d4[e] = __ldg(s4 + e);
    }
    src_off += static_cast<int64_t>(ratio) * run;
    dst_off += run;
  }
}

}  // namespace

cudaError_t launch_page_mark(const int32_t* indices, int64_t n_indices, int32_t src_page_size,
                             int64_t n_src_pages, uint8_t* mark, int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(mark, 0, static_cast<size_t>(n_src_pages), stream);
  if (e != cudaSuccess || n_indices == 0) return e;
  const int64_t blocks_needed = (n_indices + kMarkThreads - 1) / kMarkThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
  page_mark_kernel<<<grid, kMarkThreads, 0, stream>>>(indices, n_indices, src_page_size, n_src_pages,
                                                      mark);
  return cudaGetLastError();
}

cudaError_t launch_page_split(const void* src, void* dst, const uint8_t* mark, int64_t n_src_pages,
                              int32_t src_page_size, int32_t dst_page_size,
                              const PageSections& sec, cudaStream_t stream) {
  const int32_t ratio = src_page_size / dst_page_size;
  const int64_t grid = n_src_pages;
  if (grid == 0) return cudaSuccess;
  page_split_kernel<<<static_cast<unsigned>(grid), kSplitThreads, 0, stream>>>(
      static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), mark, ratio, dst_page_size, sec);
  return cudaGetLastError();
}

}  // namespace qsa
