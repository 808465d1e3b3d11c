// Allocation-free variant of qsa_sparse_prefill.
//
// Union mode needs a scratch workspace (the group lists, ownership bits and list lengths).
// The plain entry point allocates it per call on the stream; this variant instead uses a
// fixed-size array in device global memory that belongs to the library.  It is for callers
// that must not allocate device memory: code whose GPU memory is entirely owned by a
// framework's pool (which forbids allocations behind its back), latency-critical loops where
// an allocator call and the device synchronisation it can cause are not acceptable, and
// plugin hosts that hand kernels no allocator at all.
//
// The array is a file-scope __device__ variable: every GPU on which the library is loaded
// holds it (kNoAllocScratchBytes) until the process exits.  In host code its name is only a
// host-side stand-in, so the device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, and the address is what the kernels get.
#include <atomic>
#include <mutex>

#include "internal.h"

namespace qsa {
namespace {

constexpr size_t kNoAllocScratchBytes = QSA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<uintptr_t> g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  uintptr_t a = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (a == 0) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    a = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (a == 0) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      a = reinterpret_cast<uintptr_t>(ptr);
      g_scratch_addr[dev].store(a, std::memory_order_release);
    }
  }
  *out = reinterpret_cast<void*>(a);
  return cudaSuccess;
}

}  // namespace
}  // namespace qsa

extern "C" qsa_status qsa_sparse_prefill_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* indices,
    const int32_t* topk_len, void* out, float* lse, int64_t n_rows, int32_t n_qheads,
    int32_t n_kvheads, int32_t head_dim, int32_t topk, float scale, int32_t union_g,
    void* stream) {
  // Shape errors come back exactly as from the other entry points.
  qsa_geometry g{};
  qsa_status st = qsa_select_geometry(n_qheads, n_kvheads, union_g, topk, head_dim,
                                      n_rows < 0 ? 0 : n_rows, 1, &g);
  if (st != QSA_OK) return st;
  if (g.union_g > 1 &&
      qsa_union_workspace_bytes(n_rows, topk, g.union_g) > qsa::kNoAllocScratchBytes)
    return QSA_ERR_WORKSPACE;   // call needs more scratch than the fixed array holds
  void* scratch = nullptr;
  if (!q || !k_cache || !v_cache || !indices || !out) return QSA_ERR_INVALID_ARG;
  // Only union calls use the array: a per-token call never looks its address up, so it
  // neither loads the array's module nor needs to come before a stream capture.
  if (n_rows > 0 && g.union_g > 1 && qsa::scratch_address(&scratch) != cudaSuccess)
    return QSA_ERR_CUDA;
  return qsa_sparse_prefill_ex(q, k_cache, v_cache, indices, topk_len, out, lse, n_rows,
                               n_qheads, n_kvheads, head_dim, topk, scale, union_g, 0, scratch,
                               qsa::kNoAllocScratchBytes, nullptr, stream);
}
