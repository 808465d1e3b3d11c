// G-token union of selected slots with per-row ownership bits, one CTA per group.
//
// "DSA prefill ... triton_sparse_mla", Modifications: G adjacent query rows share one gathered
// index set.  Each row's selection is sorted by itself and its entries are looked up (a
// lower_bound search) in the other rows' sorted lists; a slot enters the group's list through
// the first row holding it and carries one ownership bit per row that selected it.  Accuracy
// Tests on the same page give the contract: every slot appears one time, its bits are the union
// of the rows that picked it, and padding is removed.
//
// Two kernels produce the same lists, bits and lengths:
//  * union_bitmap_kernel (the hot path): slot numbers are small integers, so each row's valid
//    set is written as a bitmap over the group's slot window in shared memory -- a counting sort
//    that also drops repeats.  A row's emitted slots are its bits not set in any earlier row's
//    bitmap, its ownership bits come from one bit test per row, and popcount prefix sums give
//    every emitted slot its place.  O(G*topk + G*window/32) work, a handful of barriers.
//  * union_build_kernel (when the caller also wants each row's sorted slots with repeats, as
//    qsa_union_build can return): rows are bitonic-sorted in shared memory and every first
//    occurrence is searched (lower_bound) in the other rows, the pages' formulation.
// The canonical order is row 0's emitted slots ascending, then row 1's, and so on.  Both are
// deterministic (the bitmap kernel's atomicOr on shared words is order independent), keep
// nothing past the call and read nothing back to the host.
#include <atomic>
#include <climits>

#include "internal.h"
#include "paged.cuh"

namespace qsa {

namespace {

constexpr int kUnionThreads = 512;

__device__ __forceinline__ int lower_bound_smem(const int32_t* row, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (row[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

int next_pow2(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p < 2 ? 2 : p;
}

}  // namespace

__global__ void __launch_bounds__(kUnionThreads)
    union_build_kernel(const int32_t* __restrict__ indices, const int32_t* __restrict__ topk_len,
                       int64_t n_rows, int32_t topk, int32_t G, int32_t Kp, int64_t n_kv_slots,
                       int32_t* __restrict__ sorted_out, int32_t* __restrict__ union_idx,
                       uint8_t* __restrict__ union_bits, int32_t* __restrict__ union_len,
                       int32_t pad_outputs) {
  extern __shared__ int32_t keys[];                                   // [G][Kp]
  uint16_t* flags = reinterpret_cast<uint16_t*>(keys + G * Kp);       // [G][Kp]: bit 8 = emit
  __shared__ int32_t cnt[8];
  __shared__ int32_t warp_tot[kUnionThreads / 32];

  const int64_t group = blockIdx.x;
  const int64_t r0 = group * G;
  const int Gp = static_cast<int>(n_rows - r0 < G ? n_rows - r0 : G);
  const int E = Gp * Kp;
  const int tid = threadIdx.x;

  // 1. load + filter
  for (int e = tid; e < E; e += kUnionThreads) {
    const int u = e / Kp, j = e - u * Kp;
    const int64_t r = r0 + u;
    int Lr = topk;
    if (topk_len) Lr = min(max(topk_len[r], 0), topk);
    int32_t x = -1;
    if (j < Lr) x = indices[r * topk + j];
    const bool ok = x >= 0 && (n_kv_slots == 0 || x < n_kv_slots);
    keys[e] = ok ? x : INT_MAX;
  }
  __syncthreads();

  // 2. bitonic sort of every row segment, ascending (INT_MAX padding sorts last)
  const int half = Kp >> 1;
  for (int k = 2; k <= Kp; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int e = tid; e < Gp * half; e += kUnionThreads) {
        const int u = e / half, i = e - u * half;
        const int lo = ((i & ~(jj - 1)) << 1) | (i & (jj - 1));
        const int hi = lo + jj;
        const bool asc = (lo & k) == 0;
        int32_t* row = keys + u * Kp;
        const int32_t a = row[lo], b = row[hi];
        if ((a > b) == asc) {
          row[lo] = b;
          row[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  if (tid < Gp) cnt[tid] = lower_bound_smem(keys + tid * Kp, Kp, INT_MAX);
  __syncthreads();

  if (sorted_out) {
    for (int e = tid; e < Gp * topk; e += kUnionThreads) {
      const int u = e / topk, j = e - u * topk;
      const int32_t x = keys[u * Kp + j];
      sorted_out[(r0 + u) * topk + j] = x == INT_MAX ? -1 : x;
    }
  }

  // 3. ownership bits and emit flags for every valid first occurrence
  for (int e = tid; e < E; e += kUnionThreads) {
    const int u = e / Kp, i = e - u * Kp;
    uint16_t f = 0;
    if (i < cnt[u]) {
      const int32_t x = keys[e];
      if (i == 0 || keys[e - 1] != x) {
        uint32_t bits = 1u << u;
        bool emit = true;
        for (int v = 0; v < Gp; ++v) {
          if (v == u) continue;
          const int32_t* row = keys + v * Kp;
          const int pos = lower_bound_smem(row, cnt[v], x);
          if (pos < cnt[v] && row[pos] == x) {
            bits |= 1u << v;
            if (v < u) emit = false;
          }
        }
        f = static_cast<uint16_t>(bits | (emit ? 0x100u : 0u));
      }
    }
    flags[e] = f;
  }
  __syncthreads();

  // 4. positions: exclusive scan of emit flags over (row, rank) order, contiguous chunks
  const int chunk = (E + kUnionThreads - 1) / kUnionThreads;
  const int e0 = min(tid * chunk, E), e1 = min(e0 + chunk, E);
  int mine = 0;
  for (int e = e0; e < e1; ++e) mine += (flags[e] >> 8) & 1;
  const int lane = tid & 31, w = tid >> 5;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  int before = 0, total = 0;
  for (int i = 0; i < kUnionThreads / 32; ++i) {
    if (i < w) before += warp_tot[i];
    total += warp_tot[i];
  }
  int pos = before + incl - mine;
  const int64_t cap = static_cast<int64_t>(G) * topk;
  int32_t* out_idx = union_idx + group * cap;
  uint8_t* out_bits = union_bits + group * cap;
  for (int e = e0; e < e1; ++e) {
    const uint16_t f = flags[e];
    if (f & 0x100u) {
      out_idx[pos] = keys[e];
      out_bits[pos] = static_cast<uint8_t>(f & 0xFFu);
      ++pos;
    }
  }
  if (tid == 0) union_len[group] = total;
  if (pad_outputs) {
    for (int64_t e = total + tid; e < cap; e += kUnionThreads) {
      out_idx[e] = -1;
      out_bits[e] = 0;
    }
  }
}

namespace {

constexpr int kBmThreads = 256;
constexpr int kBmMaxWords = 4096;      // bitmap window: up to 131072 slots per pass

__device__ __forceinline__ int block_reduce_max(int v, int* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  int r = scratch[0];
  for (int i = 1; i < kBmThreads / 32; ++i) r = max(r, scratch[i]);
  return r;
}

__device__ __forceinline__ int block_reduce_min(int v, int* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  int r = scratch[0];
  for (int i = 1; i < kBmThreads / 32; ++i) r = min(r, scratch[i]);
  return r;
}

// Exclusive prefixes over the block of eight per-thread counts at once (entries t >= n are 0):
// off[t] = sum of c[t] over lower threads, tot[t] = block sum.  One barrier pair for all eight.
__device__ __forceinline__ void block_exclusive_scan8(const int (&c)[8], int (&off)[8], int (&tot)[8],
                                                      int (*scratch)[8]) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int incl[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    incl[t] = c[t];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl[t], o);
      if (lane >= o) incl[t] += y;
    }
  }
  __syncthreads();
  if (lane == 31) {
#pragma unroll
    for (int t = 0; t < 8; ++t) scratch[w][t] = incl[t];
  }
  __syncthreads();
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    int before = 0, sum = 0;
    for (int i = 0; i < kBmThreads / 32; ++i) {
      if (i < w) before += scratch[i][t];
      sum += scratch[i][t];
    }
    off[t] = before + incl[t] - c[t];
    tot[t] = sum;
  }
}

// Exclusive prefix of v over the block; *total gets the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) scratch[w] = incl;
  __syncthreads();
  int before = 0, sum = 0;
  for (int i = 0; i < kBmThreads / 32; ++i) {
    if (i < w) before += scratch[i];
    sum += scratch[i];
  }
  *total = sum;
  return before + incl - v;
}

}  // namespace

__global__ void __launch_bounds__(kBmThreads)
    union_bitmap_kernel(const int32_t* __restrict__ indices, const int32_t* __restrict__ topk_len,
                        int64_t n_rows, int32_t topk, int32_t G, int32_t W, int64_t n_kv_slots,
                        int32_t* __restrict__ union_idx, uint8_t* __restrict__ union_bits,
                        int32_t* __restrict__ union_len, int32_t pad_outputs, PagedAddr pa,
                        int32_t* __restrict__ item_counter) {
  extern __shared__ uint32_t sm_words[];
  int32_t* ent = reinterpret_cast<int32_t*>(sm_words);    // [G][topk]: valid slot or -1
  uint32_t* bm = sm_words + G * topk;                      // [G][W] bitmaps of one window
  __shared__ int scratch[kBmThreads / 32];
  __shared__ int row_total[8], row_base[8], row_done[8];
  __shared__ int32_t row_req[8], row_kvlen[8];
  __shared__ int vscratch[kBmThreads / 32][8];

  const int64_t group = blockIdx.x;
  const int64_t r0 = group * G;
  const int Gp = static_cast<int>(n_rows - r0 < G ? n_rows - r0 : G);
  const int tid = threadIdx.x;
  // the attention kernel that follows on the stream hands out its items through this counter
  if (item_counter != nullptr && group == 0 && tid == 0) *item_counter = 0;
  const int64_t cap = static_cast<int64_t>(G) * topk;
  int32_t* out_idx = union_idx + group * cap;
  uint8_t* out_bits = union_bits + group * cap;

  // 0. paged indices: every row's request and KV length (warp 0, one row at a time)
  const bool paged = pa.page_table != nullptr;
  if (paged) {
    if (tid < 32) {
      for (int u = 0; u < Gp; ++u) {
        const int32_t req = paged_request_of_row(pa, r0 + u, tid);
        if (tid == 0) {
          row_req[u] = req;
          row_kvlen[u] = paged_kv_len(pa, req);
        }
      }
    }
    __syncthreads();
  }

  // 1. valid slots of the group's rows (topk_len, negative, >= n_kv_slots filtered; logical
  //    positions translated through the page table) and their max.  Each thread has eight
  //    index loads in flight before it uses any: the build is bound by load latency.
  int my_max = -1;
  constexpr int kLoadsInFlight = 8;
  const int n_ent = Gp * topk;
  // (row, position) of element e = e0 + k * kBmThreads + tid, stepped without a division
  int eu = tid / topk, ej = tid - eu * topk;
  for (int e0 = 0; e0 < n_ent; e0 += kLoadsInFlight * kBmThreads) {
    int32_t xs[kLoadsInFlight];
    int us[kLoadsInFlight];
#pragma unroll
    for (int k = 0; k < kLoadsInFlight; ++k) {
      const int e = e0 + k * kBmThreads + tid;
      us[k] = eu;
      xs[k] = -1;
      if (e < n_ent) {
        const int64_t r = r0 + eu;
        const int Lr = topk_len ? min(max(__ldg(topk_len + r), 0), topk) : topk;
        if (ej < Lr) xs[k] = __ldg(indices + r * topk + ej);
      }
      ej += kBmThreads;
      if (ej >= topk) {          // a row boundary was crossed (at most once when topk >= 256)
        const int q = ej / topk;
        eu += q;
        ej -= q * topk;
      }
    }
#pragma unroll
    for (int k = 0; k < kLoadsInFlight; ++k) {
      const int e = e0 + k * kBmThreads + tid;
      if (e >= n_ent) break;
      int32_t x = xs[k];
      if (paged) {
        const int u = us[k];
        const int64_t slot = paged_slot(pa, row_req[u], row_kvlen[u], x);
        x = slot > static_cast<int64_t>(INT32_MAX) ? -1 : static_cast<int32_t>(slot);
      }
      if (x < 0 || (n_kv_slots > 0 && x >= n_kv_slots)) x = -1;
      ent[e] = x;
      my_max = max(my_max, x);
    }
  }
  const int gmax = block_reduce_max(my_max, scratch);
  if (tid < 8) { row_total[tid] = 0; row_done[tid] = 0; }
  __syncthreads();

  // 2. windows of W*32 slots, ascending; two passes (counts, then placement) unless one window
  //    covers every slot, in which case the bitmaps are built once.
  const int64_t span = static_cast<int64_t>(W) * 32;
  const bool one_window = gmax >= 0 && gmax < span;
  // One window: the bitmaps are built once, one vector scan gives every (thread, row) count its
  // place, and a single pass emits all rows.  Several windows: a counting pass first, because a
  // row's slots from every window precede the next row's.
  int placed = 0;
  if (one_window) {
    const int active = gmax / 32 + 1;
    for (int i = tid; i < Gp * active; i += kBmThreads) bm[(i / active) * W + i % active] = 0u;
    __syncthreads();
    for (int e = tid; e < Gp * topk; e += kBmThreads) {
      const int32_t x = ent[e];
      if (x >= 0) atomicOr(&bm[(e / topk) * W + (x >> 5)], 1u << (x & 31));
    }
    __syncthreads();
    const int wpt = (active + kBmThreads - 1) / kBmThreads;   // words per thread
    const int w0 = tid * wpt, w1 = min(w0 + wpt, active);
    int cnt[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) cnt[t] = 0;
    for (int w = w0; w < w1; ++w) {
      uint32_t earlier = 0u;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (t < Gp) {
          const uint32_t m = bm[t * W + w];
          cnt[t] += __popc(m & ~earlier);
          earlier |= m;
        }
      }
    }
    int off[8], tot[8];
    block_exclusive_scan8(cnt, off, tot, vscratch);
    int pos[8], acc = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      pos[t] = acc + off[t];
      acc += t < Gp ? tot[t] : 0;
    }
    for (int w = w0; w < w1; ++w) {
      uint32_t words[8], earlier = 0u;
#pragma unroll
      for (int t = 0; t < 8; ++t) words[t] = t < Gp ? bm[t * W + w] : 0u;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        uint32_t m = words[t] & ~earlier;
        earlier |= words[t];
        while (m) {
          const int b = __ffs(m) - 1;
          m &= m - 1u;
          uint32_t owners = 0u;
#pragma unroll
          for (int u = 0; u < 8; ++u) owners |= ((words[u] >> b) & 1u) << u;
          out_idx[pos[t]] = 32 * w + b;
          out_bits[pos[t]] = static_cast<uint8_t>(owners);
          ++pos[t];
        }
      }
    }
    placed = acc;
  }
  for (int pass = 0; pass < 2 && gmax >= 0 && !one_window; ++pass) {
    int64_t wbase = 0;
    if (pass == 1) {
      if (tid == 0) {
        int acc = 0;
        for (int t = 0; t < Gp; ++t) { row_base[t] = acc; acc += row_total[t]; }
      }
      __syncthreads();
    }
    while (wbase <= gmax) {
      const int64_t need_words = (gmax - wbase) / 32 + 1;
      const int active = static_cast<int>(need_words < W ? need_words : W);
      const int wpt = (active + kBmThreads - 1) / kBmThreads;   // words per thread
      {
        for (int i = tid; i < Gp * active; i += kBmThreads) bm[(i / active) * W + i % active] = 0u;
        __syncthreads();
        for (int e = tid; e < Gp * topk; e += kBmThreads) {
          const int32_t x = ent[e];
          if (x >= wbase && x < wbase + span) {
            const int u = e / topk;
            const int off = static_cast<int>(x - wbase);
            atomicOr(&bm[u * W + (off >> 5)], 1u << (off & 31));
          }
        }
        __syncthreads();
      }
      const int w0 = tid * wpt, w1 = min(w0 + wpt, active);
      for (int t = 0; t < Gp; ++t) {
        // this thread's emitted count for row t in its words
        int c = 0;
        for (int w = w0; w < w1; ++w) {
          uint32_t earlier = 0u;
          for (int u = 0; u < t; ++u) earlier |= bm[u * W + w];
          c += __popc(bm[t * W + w] & ~earlier);
        }
        int total = 0;
        const int off = block_exclusive_scan(c, scratch, &total);
        if (pass == 0) {
          if (tid == 0) row_total[t] += total;
        } else {
          int pos = row_base[t] + row_done[t] + off;
          for (int w = w0; w < w1; ++w) {
            uint32_t earlier = 0u;
            for (int u = 0; u < t; ++u) earlier |= bm[u * W + w];
            uint32_t m = bm[t * W + w] & ~earlier;
            while (m) {
              const int b = __ffs(m) - 1;
              m &= m - 1u;
              uint32_t owners = 0u;
              for (int u = 0; u < Gp; ++u) owners |= ((bm[u * W + w] >> b) & 1u) << u;
              out_idx[pos] = static_cast<int32_t>(wbase + 32 * w + b);
              out_bits[pos] = static_cast<uint8_t>(owners);
              ++pos;
            }
          }
          __syncthreads();
          if (tid == 0) row_done[t] += total;
        }
        __syncthreads();
      }
      // next window starts at the smallest slot past this one
      int my_next = INT_MAX;
      for (int e = tid; e < Gp * topk; e += kBmThreads) {
        const int32_t x = ent[e];
        if (x >= wbase + span) my_next = min(my_next, x);
      }
      const int nxt = block_reduce_min(my_next, scratch);
      if (nxt == INT_MAX) break;
      wbase = nxt;
    }
  }
  int total = 0;
  if (one_window) {
    total = placed;
  } else {
    for (int t = 0; t < Gp; ++t) total += row_total[t];
  }
  if (tid == 0) union_len[group] = total;
  if (pad_outputs) {
    for (int64_t e = total + tid; e < cap; e += kBmThreads) {
      out_idx[e] = -1;
      out_bits[e] = 0;
    }
  }
}

int union_bitmap_words(int32_t topk, int32_t union_g) {
  const int64_t ent = static_cast<int64_t>(union_g) * topk * 4;
  const int64_t room = static_cast<int64_t>(kUnionMaxSmem) - ent;
  if (room <= 0) return 0;
  int64_t w = room / (static_cast<int64_t>(union_g) * 4);
  w = w / kBmThreads * kBmThreads;
  return static_cast<int>(w < kBmMaxWords ? w : kBmMaxWords);
}

size_t union_build_smem_bytes(int32_t topk, int32_t union_g) {
  // shared memory of the bitmap kernel at its largest window (0 if not even 256 words fit)
  const int w = union_bitmap_words(topk, union_g);
  if (w < kBmThreads) return static_cast<size_t>(kUnionMaxSmem) + 1;
  return static_cast<size_t>(union_g) * (static_cast<size_t>(topk) + w) * 4;
}

size_t union_sort_smem_bytes(int32_t topk, int32_t union_g) {
  const size_t Kp = static_cast<size_t>(next_pow2(topk));
  return static_cast<size_t>(union_g) * Kp * (sizeof(int32_t) + sizeof(uint16_t));
}

cudaError_t launch_union_build(const int32_t* indices, const int32_t* topk_len, int64_t n_rows,
                               int32_t topk, int32_t union_g, int64_t n_kv_slots,
                               int32_t* sorted_out, int32_t* union_idx, uint8_t* union_bits,
                               int32_t* union_len, bool pad_outputs, const PagedAddr* paged,
                               cudaStream_t stream, int32_t* item_counter) {
  if (n_rows == 0) return cudaSuccess;
  // The sorted-rows kernel takes physical slots only.
  if (paged != nullptr && sorted_out != nullptr) return cudaErrorInvalidValue;
  if (item_counter != nullptr && sorted_out != nullptr) return cudaErrorInvalidValue;
  PagedAddr pa{};
  if (paged != nullptr) pa = *paged;
  const int64_t n_groups = (n_rows + union_g - 1) / union_g;
  if (sorted_out == nullptr) {
    // Window: the widest that still lets several groups share an SM (the build is latency
    // bound), no wider than the slot count when the caller gives one.
    int W = union_bitmap_words(topk, union_g);
    if (W < kBmThreads) return cudaErrorInvalidValue;
    for (int per_sm = 4; per_sm >= 2; --per_sm) {
      const int64_t budget = (227 * 1024) / per_sm - 1024;
      const int64_t w = (budget / 4 - static_cast<int64_t>(union_g) * topk) / union_g / kBmThreads * kBmThreads;
      if (w >= 1024) {
        if (w < W) W = static_cast<int>(w);
        break;
      }
    }
    if (n_kv_slots > 0) {
      const int64_t need = ((n_kv_slots + 31) / 32 + kBmThreads - 1) / kBmThreads * kBmThreads;
      if (need < W) W = static_cast<int>(need);
    }
    const size_t smem = static_cast<size_t>(union_g) * (static_cast<size_t>(topk) + W) * 4;
    static std::atomic<int> bm_opted_in[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || bm_opted_in[dev].load() < static_cast<int>(smem)) {
      e = cudaFuncSetAttribute(union_bitmap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) bm_opted_in[dev].store(static_cast<int>(smem));
    }
    union_bitmap_kernel<<<static_cast<unsigned>(n_groups), kBmThreads, smem, stream>>>(
        indices, topk_len, n_rows, topk, union_g, W, n_kv_slots, union_idx, union_bits, union_len,
        pad_outputs ? 1 : 0, pa, item_counter);
    return cudaGetLastError();
  }
  const int Kp = next_pow2(topk);
  const size_t smem = union_sort_smem_bytes(topk, union_g);
  static std::atomic<int> opted_in[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || opted_in[dev].load() < static_cast<int>(smem)) {
    e = cudaFuncSetAttribute(union_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) opted_in[dev].store(static_cast<int>(smem));
  }
  union_build_kernel<<<static_cast<unsigned>(n_groups), kUnionThreads, smem, stream>>>(
      indices, topk_len, n_rows, topk, union_g, Kp, n_kv_slots, sorted_out, union_idx, union_bits,
      union_len, pad_outputs ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace qsa
