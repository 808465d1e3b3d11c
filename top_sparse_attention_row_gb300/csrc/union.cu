// G-token union of selected slots with per-row ownership bits, one CTA per group.
//
// "DSA prefill ... triton_sparse_mla", Modifications: G adjacent query rows share one gathered
// index set; each row's selection is sorted on its own, then every entry is searched
// (lower_bound) in the other rows' sorted lists; a row emits a slot no earlier row of the group
// selected and ORs in the bit of every row that did.  Accuracy Tests on the same page give the
// contract: each slot once, bits = OR of owners, -1 dropped.
//
// Here the sort and the union build are one kernel: the group's G rows are loaded into shared
// memory (invalid entries -- beyond topk_len, negative, >= n_kv_slots -- become INT_MAX), each
// row is bitonic-sorted in place, every valid first occurrence is searched in the other rows,
// and a block-wide scan over (row, rank) order gives each emitted slot its place in the
// canonical list (row 0's emitted slots ascending, then row 1's, ...).  No atomics: the output
// is deterministic.  Nothing outlives the call and nothing is read back to the host.
#include <atomic>
#include <climits>

#include "internal.h"

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

size_t union_build_smem_bytes(int32_t topk, int32_t union_g) {
  const size_t Kp = static_cast<size_t>(next_pow2(topk));
  return static_cast<size_t>(union_g) * Kp * (sizeof(int32_t) + sizeof(uint16_t));
}

cudaError_t launch_union_build(const int32_t* indices, const int32_t* topk_len, int64_t n_rows,
                               int32_t topk, int32_t union_g, int64_t n_kv_slots,
                               int32_t* sorted_out, int32_t* union_idx, uint8_t* union_bits,
                               int32_t* union_len, bool pad_outputs, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  const int Kp = next_pow2(topk);
  const size_t smem = union_build_smem_bytes(topk, union_g);
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
  const int64_t n_groups = (n_rows + union_g - 1) / union_g;
  union_build_kernel<<<static_cast<unsigned>(n_groups), kUnionThreads, smem, stream>>>(
      indices, topk_len, n_rows, topk, union_g, Kp, n_kv_slots, sorted_out, union_idx, union_bits,
      union_len, pad_outputs ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace qsa
