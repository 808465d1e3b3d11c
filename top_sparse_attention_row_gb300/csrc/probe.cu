// Gather-ceiling probe: how fast can one GB300 SM pull random half-rows (256 B) of a KV cache
// from L2 into shared memory, with nothing else running?  It uses the same engines and shapes as
// the attention kernel's producers -- TMA tile::gather4 (4 rows x 128 B per op) or cp.async
// 16-byte copies, 32 KiB pieces of 128 rows x 256 B, 128-byte swizzled destinations, a 6-stage
// ring -- but the consumer only releases each stage, so the result bounds what the gather side
// of the kernel can approach.
//
// Each of the six producer warps owns one stage of the ring and gathers every piece that lands
// on it, so no two warps ever wait on different phases of one stage.
//
// The contention variant (qsa_probe_gather_mma) adds one more warp that keeps the tensor pipe
// busy for as long as the gather runs: batches of 16 tcgen05.mma M128 x N x K16 (bf16 -> fp32,
// the attention kernel's swap-AB shape) on a shared-memory region of its own, one commit per
// batch, at most two batches in flight.  A reads from shared memory (mode 1, as the kernel's
// operands do) or from tensor memory (mode 2).  It reports the gather rate under that load and
// the tensor pipe's time per MMA under the gather; pieces_per_cta = 0 times the MMAs alone.
#include "internal.h"
#include "ptx.cuh"

namespace qsa {
namespace {

constexpr int kProbeStages = 6;
constexpr int kProbeWarps = kProbeStages + 1;     // six owners + one releasing consumer

__device__ __forceinline__ unsigned long long probe_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ bool probe_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = probe_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (probe_ns() - t0 > 1000000000ull) {
      *abort_flag = 1;
      atomicExch(status, 1);
      return false;
    }
  }
  return true;
}

constexpr int kProbeMmaBatch = 16;     // MMAs per commit: one 256-dim K pass of the kernel
constexpr int kProbeMmaMaxN = 64;
constexpr int kProbeMmaA = 16384;      // A region: 128 rows x 128 B (SW128), four K16 steps
constexpr int kProbeMmaB = kProbeMmaMaxN * 128;

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16 (A: 128 lanes x 8 columns per K16 step).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Bounded wait that ignores the abort flag: lets work already issued finish before teardown.
__device__ void probe_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = probe_ns();
  while (!mbar_try_wait(bar, parity) && probe_ns() - t0 < 1000000000ull) {
  }
}

// MMA_MODE: 0 = gather only; 1 = plus MMAs with A in shared memory; 2 = A in tensor memory.
template <int MMA_MODE>
__global__ void __launch_bounds__(32 * (kProbeWarps + 1), 1)
    gather_probe_kernel(const __grid_constant__ CUtensorMap tm, const uint8_t* __restrict__ cache,
                        const int32_t* __restrict__ rows, int64_t n_table_pieces,
                        int32_t pieces_per_cta, int use_tma, int mma_n, int32_t mma_batches,
                        int* status, unsigned long long* mma_stats) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t ring_end = base + kProbeStages * kStageBytes;
  const uint32_t mma_a = ring_end;
  const uint32_t mma_b = ring_end + kProbeMmaA;
  const uint32_t full = ring_end + (MMA_MODE ? kProbeMmaA + kProbeMmaB : 0);
  const uint32_t empty = full + 8 * kProbeStages;
  const uint32_t mbar = empty + 8 * kProbeStages;     // two MMA batch barriers (MMA modes)
  __shared__ int abort_flag;
  __shared__ int gather_done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kProbeStages; ++s) {
      // engine 2 (mixed): even stages TMA, odd stages cp.async
      const bool stage_tma = use_tma == 1 || (use_tma == 2 && (s & 1) == 0);
      mbar_init(full + 8 * s, stage_tma ? 1 : 32);
      mbar_init(empty + 8 * s, 1);
    }
    if (MMA_MODE) {
      mbar_init(mbar, 1);
      mbar_init(mbar + 8, 1);
    }
    abort_flag = 0;
    gather_done = 0;
    fence_mbar_init();
  }
  if constexpr (MMA_MODE != 0) {
    if (warp == kProbeWarps) {
      tmem_alloc(smem_u32(&tmem_slot), 128);
      tmem_relinquish();
    }
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (MMA_MODE != 0) tc_fence_after();
  volatile int* ab = &abort_flag;
  if (warp < kProbeStages) {
    const int st = warp;
    const bool warp_tma = use_tma == 1 || (use_tma == 2 && (st & 1) == 0);
    int last = -1;   // newest piece this warp issued
    for (int p = st; p < pieces_per_cta; p += kProbeStages) {
      const uint32_t par = ((p / kProbeStages) & 1) ^ 1;
      if (!__all_sync(0xffffffffu, probe_wait(empty + 8 * st, par, ab, status))) break;
      const int32_t* prow = rows + ((blockIdx.x * 131 + p) % n_table_pieces) * kTileTokens;
      const uint32_t dst = base + st * kStageBytes;
      if (warp_tma) {
        // lane: rows 4*lane .. 4*lane+3, two gather4 ops (dims 0-63 and 64-127)
        const int4 y = *reinterpret_cast<const int4*>(prow + 4 * lane);
        if (lane == 0) mbar_arrive_expect_tx(full + 8 * st, kStageBytes);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_gather4(dst + c * 16384 + lane * 512, &tm, c * 64, y.x, y.y, y.z, y.w, full + 8 * st);
        last = p;
        continue;
      }
      const int ch = lane & 15;
#pragma unroll 8
      for (int i = 0; i < 64; ++i) {
        const int t = 2 * i + (lane >> 4);
        const uint8_t* src = cache + static_cast<int64_t>(prow[t]) * (kHeadDim * 2) + ch * 16;
        const uint32_t d = dst + (ch >> 3) * 16384 + t * 128 + (((ch & 7) ^ (t & 7)) << 4);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(full + 8 * st)
                   : "memory");
    }
    if (!warp_tma) {
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (*ab && last >= 0 && lane == 0) {
      // after an abort the consumer may not have waited for this stage: let the newest copy
      // land (bounded) before the block exits
      probe_drain(full + 8 * st, (last / kProbeStages) & 1);
    }
  } else if (warp == kProbeStages) {
    for (int p = 0; p < pieces_per_cta; ++p) {
      const int st = p % kProbeStages;
      if (!__all_sync(0xffffffffu, probe_wait(full + 8 * st, (p / kProbeStages) & 1, ab, status)))
        break;
      if (lane == 0) mbar_arrive(empty + 8 * st);
      __syncwarp();
    }
    if (lane == 0) *reinterpret_cast<volatile int*>(&gather_done) = 1;
  } else if constexpr (MMA_MODE != 0) {
    // tensor-pipe load: batches of 16 MMAs, one commit each, at most two batches in flight
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&tmem_slot);
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, mma_n, false, false);
      volatile int* done = &gather_done;
      const unsigned long long t0 = probe_ns();
      int b = 0;
      while (b < mma_batches) {
        if (pieces_per_cta > 0 && b > 0 && *done) break;
#pragma unroll
        for (int k = 0; k < kProbeMmaBatch; ++k) {
          const uint64_t bd = sw128_desc(mma_b + (k & 3) * 32, 16, 1024);
          if constexpr (MMA_MODE == 1) {
            const uint64_t ad = sw128_desc(mma_a + (k & 3) * 32, 16, 1024);
            tc_mma(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
          } else {
            tc_mma_ts(tmem, tmem + 64 + 8 * (k & 3), bd, idesc, k > 0 ? 1u : 0u);
          }
        }
        tc_commit(mbar + 8 * (b & 1));
        ++b;
        // batch b-2 (the other barrier's previous use) must be done before this one is reused
        if (b >= 2 && !probe_wait(mbar + 8 * (b & 1), ((b - 2) >> 1) & 1, ab, status)) break;
      }
      if (b > 0) probe_drain(mbar + 8 * ((b - 1) & 1), ((b - 1) >> 1) & 1);
      const unsigned long long t1 = probe_ns();
      atomicAdd(&mma_stats[0], static_cast<unsigned long long>(b));
      atomicAdd(&mma_stats[1], t1 - t0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
  __syncthreads();
}

// Shared launch path of both entry points.  Returns the kernel's elapsed milliseconds, and for
// the MMA modes the number of MMAs issued over all SMs and their summed per-SM nanoseconds.
template <int MODE>
qsa_status run_probe(const void* cache, int64_t n_rows, const int32_t* rows, int64_t n_table_pieces,
                     int32_t pieces_per_cta, int32_t engine, int32_t mma_n, int32_t mma_batches,
                     cudaStream_t stream, float* ms_out, unsigned long long* stats_out) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QSA_ERR_CUDA;
  CUtensorMap tm;
  if (make_cache_map(&tm, cache, n_rows, kHeadDim) != cudaSuccess) return QSA_ERR_CUDA;
  const int smem = kProbeStages * kStageBytes + (MODE ? kProbeMmaA + kProbeMmaB : 0) +
                   16 * kProbeStages + 16 + 1024;
  if (cudaFuncSetAttribute(gather_probe_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return QSA_ERR_CUDA;
  // measurement helper, not the hot path: a status word, two counters and two events per call
  void* scratch = nullptr;
  if (cudaMallocAsync(&scratch, 32, stream) != cudaSuccess) return QSA_ERR_CUDA;
  int* status = static_cast<int*>(scratch);
  unsigned long long* stats = reinterpret_cast<unsigned long long*>(static_cast<char*>(scratch) + 16);
  cudaMemsetAsync(scratch, 0, 32, stream);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  cudaEventRecord(a, stream);
  const int threads = 32 * (kProbeWarps + (MODE ? 1 : 0));
  gather_probe_kernel<MODE><<<sms, threads, smem, stream>>>(
      tm, static_cast<const uint8_t*>(cache), rows, n_table_pieces, pieces_per_cta, engine, mma_n,
      mma_batches, status, stats);
  cudaEventRecord(b, stream);
  int h_status = 0;
  unsigned long long h_stats[2] = {0, 0};
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h_status, status, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h_stats, stats, sizeof(h_stats), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return QSA_ERR_CUDA;
  if (h_status != 0) return QSA_ERR_TIMEOUT;
  *ms_out = ms;
  if (stats_out) {
    stats_out[0] = h_stats[0];
    stats_out[1] = h_stats[1];
  }
  return QSA_OK;
}

}  // namespace
}  // namespace qsa

extern "C" qsa_status qsa_probe_gather_ceiling(const void* cache, int64_t n_rows,
                                               const int32_t* rows, int64_t n_table_pieces,
                                               int32_t pieces_per_cta, int32_t engine,
                                               float* ms_out, void* stream_v) {
  if (!cache || !rows || !ms_out || n_rows <= 0 || n_table_pieces <= 0 || pieces_per_cta <= 0 ||
      engine < 0 || engine > 2 || (reinterpret_cast<uintptr_t>(cache) & 15u) != 0)
    return QSA_ERR_INVALID_ARG;
  return qsa::run_probe<0>(cache, n_rows, rows, n_table_pieces, pieces_per_cta, engine, 16, 0,
                           static_cast<cudaStream_t>(stream_v), ms_out, nullptr);
}

extern "C" qsa_status qsa_probe_gather_mma(const void* cache, int64_t n_rows, const int32_t* rows,
                                           int64_t n_table_pieces, int32_t pieces_per_cta,
                                           int32_t engine, int32_t mma_mode, int32_t mma_n,
                                           int32_t mma_batches, float* ms_out, float* mma_ns_out,
                                           void* stream_v) {
  if (!cache || !rows || !ms_out || !mma_ns_out || n_rows <= 0 || n_table_pieces <= 0 ||
      pieces_per_cta < 0 || engine < 0 || engine > 2 || (mma_mode != 1 && mma_mode != 2) ||
      mma_n < 16 || mma_n > qsa::kProbeMmaMaxN || (mma_n & 15) != 0 || mma_batches < 1 ||
      mma_batches > (1 << 24) || (reinterpret_cast<uintptr_t>(cache) & 15u) != 0)
    return QSA_ERR_INVALID_ARG;
  unsigned long long stats[2] = {0, 0};
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const qsa_status st =
      mma_mode == 1
          ? qsa::run_probe<1>(cache, n_rows, rows, n_table_pieces, pieces_per_cta, engine, mma_n,
                              mma_batches, stream, ms_out, stats)
          : qsa::run_probe<2>(cache, n_rows, rows, n_table_pieces, pieces_per_cta, engine, mma_n,
                              mma_batches, stream, ms_out, stats);
  if (st != QSA_OK) return st;
  *mma_ns_out = stats[0] ? static_cast<float>(static_cast<double>(stats[1]) /
                                              (static_cast<double>(stats[0]) * qsa::kProbeMmaBatch))
                         : 0.f;
  return QSA_OK;
}
