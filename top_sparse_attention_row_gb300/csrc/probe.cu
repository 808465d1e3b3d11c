// Gather-ceiling probe: how fast can one GB300 SM pull random half-rows (256 B) of a KV cache
// from L2 into shared memory, with nothing else running?  It uses the same engines and shapes as
// the d=256 attention kernel's gather warps -- TMA tile::gather4 (4 rows x 128 B per op) or
// cp.async 16-byte copies, 32 KiB pieces of 128 rows x 256 B, 128-byte swizzled destinations, a
// 6-stage ring filled by two warps per stage, one per 64-dim block -- but the consumer only
// releases each stage, so the result bounds what the gather side of the kernel can approach.
#include "internal.h"
#include "ptx.cuh"

namespace qsa {
namespace {

constexpr int kProbeStages = 6;
constexpr int kProbeGatherWarps = kProbeStages * kBlocksPerStage;
constexpr int kProbeWarps = kProbeGatherWarps + 1;     // gather warps + one releasing consumer

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

// Bounded wait that ignores the abort flag: lets work already issued finish before teardown.
__device__ void probe_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = probe_ns();
  while (!mbar_try_wait(bar, parity) && probe_ns() - t0 < 1000000000ull) {
  }
}

__global__ void __launch_bounds__(32 * kProbeWarps, 1)
    gather_probe_kernel(const __grid_constant__ CUtensorMap tm, const uint8_t* __restrict__ cache,
                        const int32_t* __restrict__ rows, int64_t n_table_pieces,
                        int32_t pieces_per_cta, int use_tma, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t full = base + kProbeStages * kStageBytes;
  const uint32_t empty = full + 8 * kProbeStages;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kProbeStages; ++s) {
      // engine 2 (mixed): even stages TMA, odd stages cp.async
      const bool stage_tma = use_tma == 1 || (use_tma == 2 && (s & 1) == 0);
      mbar_init(full + 8 * s, stage_tma ? kBlocksPerStage : 32 * kBlocksPerStage);
      mbar_init(empty + 8 * s, 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* ab = &abort_flag;
  if (warp < kProbeGatherWarps) {
    const int st = warp / kBlocksPerStage, blk = warp % kBlocksPerStage;
    const bool warp_tma = use_tma == 1 || (use_tma == 2 && (st & 1) == 0);
    int last = -1;   // newest piece this warp issued
    for (int p = st; p < pieces_per_cta; p += kProbeStages) {
      const uint32_t par = ((p / kProbeStages) & 1) ^ 1;
      if (!__all_sync(0xffffffffu, probe_wait(empty + 8 * st, par, ab, status))) break;
      const int32_t* prow = rows + ((blockIdx.x * 131 + p) % n_table_pieces) * kTileTokens;
      const uint32_t dst = base + st * kStageBytes + blk * 16384;
      if (warp_tma) {
        // lane: rows 4*lane .. 4*lane+3 of this warp's 64-dim block
        const int4 y = *reinterpret_cast<const int4*>(prow + 4 * lane);
        if (lane == 0) mbar_arrive_expect_tx(full + 8 * st, kStageBytes / kBlocksPerStage);
        __syncwarp();
        tma_gather4(dst + lane * 512, &tm, blk * 64, y.x, y.y, y.z, y.w, full + 8 * st);
        last = p;
        continue;
      }
      const int ch = lane & 7;
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const int t = 4 * i + (lane >> 3);
        const uint8_t* src = cache + static_cast<int64_t>(prow[t]) * (kHeadDim * 2) + blk * 128 + ch * 16;
        const uint32_t d = dst + t * 128 + ((ch ^ (t & 7)) << 4);
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
  } else if (warp == kProbeGatherWarps) {
    for (int p = 0; p < pieces_per_cta; ++p) {
      const int st = p % kProbeStages;
      if (!__all_sync(0xffffffffu, probe_wait(full + 8 * st, (p / kProbeStages) & 1, ab, status)))
        break;
      if (lane == 0) mbar_arrive(empty + 8 * st);
      __syncwarp();
    }
  }
  __syncthreads();
}

// Launch path: returns the kernel's elapsed milliseconds.
qsa_status run_probe(const void* cache, int64_t n_rows, const int32_t* rows, int64_t n_table_pieces,
                     int32_t pieces_per_cta, int32_t engine, cudaStream_t stream, float* ms_out) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QSA_ERR_CUDA;
  CUtensorMap tm;
  if (make_cache_map(&tm, cache, n_rows, kHeadDim) != cudaSuccess) return QSA_ERR_CUDA;
  const int smem = kProbeStages * kStageBytes + 16 * kProbeStages + 1024;
  if (cudaFuncSetAttribute(gather_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return QSA_ERR_CUDA;
  // measurement helper, not the hot path: a status word and two events per call
  void* scratch = nullptr;
  if (cudaMallocAsync(&scratch, 16, stream) != cudaSuccess) return QSA_ERR_CUDA;
  int* status = static_cast<int*>(scratch);
  cudaMemsetAsync(scratch, 0, 16, stream);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  cudaEventRecord(a, stream);
  gather_probe_kernel<<<sms, 32 * kProbeWarps, smem, stream>>>(
      tm, static_cast<const uint8_t*>(cache), rows, n_table_pieces, pieces_per_cta, engine, status);
  cudaEventRecord(b, stream);
  int h_status = 0;
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h_status, status, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return QSA_ERR_CUDA;
  if (h_status != 0) return QSA_ERR_TIMEOUT;
  *ms_out = ms;
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
  return qsa::run_probe(cache, n_rows, rows, n_table_pieces, pieces_per_cta, engine,
                        static_cast<cudaStream_t>(stream_v), ms_out);
}
