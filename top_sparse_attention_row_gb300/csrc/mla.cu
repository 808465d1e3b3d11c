// sparse_mla_kernel<NP, UNION>: top-k sparse attention prefill in the MLA shape -- one latent
// KV row per slot (d_qk = 512 latent + 64 rope dims, V = the 512 latent dims of the same row),
// every query head attending over its row's gathered slots.  The shape is the second workload
// of "DSA prefill ... triton_sparse_mla" (Speed Tests: kv_lora_rank 512 + qk_rope_head_dim 64 =
// 576, d_v 512, topk 2048, 8 heads at TP8), with the same per-token and G-token union modes.
//
// Design (sm_103a):
//  * Swap-AB tcgen05 as in the d=256 kernel: slots are the MMA M (128 per tile), query columns
//    (heads, or G x heads in union mode) are N, padded to 16 or 32.
//    S^T = K_tile . Q^T takes 36 MMAs (K = 576 in steps of 16); O^T += V_tile^T . P^T takes
//    4 output chunks of 128 dims x 8 steps = 32 MMAs.
//  * V is part of the K tile, so each slot is gathered once (1152 bytes) and the tile stays in
//    shared memory from QK^T to P.V.  Latent dims arrive as four 32 KiB "pair" pieces (128
//    slots x 128 dims, two 128-byte-swizzled atoms) in a FIFO ring of 4-5 stages; the rope dims
//    as one 16 KiB piece in a one-stage ring.
//  * Issue order of the single MMA thread, per tile j: the first latent chunk (when the ring has
//    a spare stage) and the rope chunk of S(j+1) go first, overlapping the softmax of tile j;
//    then P.V(j), each 128-dim output chunk releasing its latent piece as soon as its MMAs
//    complete, so the gather of tile j+1 runs under P.V(j); then the rest of S(j+1).
//  * Gather: TMA tile::gather4 (4 rows x 128 bytes per op).  Ten gather warps share every
//    latent piece (each issues about a tenth of its 64 ops), so a stage freed by P.V refills in
//    a tenth of the time one warp would take; two more share the rope pieces.  Padding rows use
//    a row past the tensor map, which TMA zero-fills.
//  * 20 warps (five warpgroups) with warpgroup register reallocation, as in the d=256 kernel:
//    softmax (0-3), MMA and index (4-5), gather (6, 7, 9-11, 13-19; 8 and 12 idle so that the
//    MMA warp's sub-partition holds one gather warp).
//  * Online softmax, epilogue, union masks, bounded waits and failure containment follow the
//    d=256 kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <atomic>

#include "compact.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace qsa {
namespace {

constexpr unsigned long long kMlaWaitNs = 2000000000ull;    // 2 s per wait
constexpr unsigned long long kMlaDrainNs = 200000000ull;    // 0.2 s per drain wait
constexpr float kMlaRescale = 8.0f;                         // log2 units
constexpr float kMlaLn2 = 0.6931471805599453f;
constexpr int kMlaPairOwners = kMlaLatentWarps;             // gather warps sharing latent pieces

// Wait sites of this kernel in the status word (0x100 | site), after the d=256 kernel's.
enum MlaSite : int32_t {
  kMItemEmpty = 0x21, kMQEmpty, kMItemFull, kMLatEmpty, kMLatFull, kMRopeEmpty, kMRopeFull,
  kMSFree, kMSFull, kMPFull, kMPvDone, kMDrain, kMQFull
};

__device__ __forceinline__ unsigned long long mla_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mla_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* status, int32_t site,
                                           unsigned long long limit) {
  const unsigned long long t0 = mla_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mla_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicCAS(status, 0, 0x100 | site);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag: after an abort, lets copies and MMAs already issued
// complete before shared or tensor memory is given up.
__device__ __forceinline__ bool mla_drain(uint32_t bar, uint32_t parity, int32_t* status,
                                       unsigned long long limit) {
  const unsigned long long t0 = mla_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (mla_ns() - t0 > limit) {
      atomicCAS(status, 0, 0x100 | kMDrain);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool mla_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* status, int32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return mla_wait_slow(bar, parity, abort_flag, status, site, kMlaWaitNs);
}

__device__ __forceinline__ uint4 mla_ldg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void mla_sts_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

struct MlaItem {   // written by the index warp, read by every role
  int32_t n_valid, group, chunk, cols, row0, rows_in_group, pad0, pad1;
};

}  // namespace

// SC: query columns the softmax computes (SC < NP when an item's real columns fit in SC; the MMA
// still runs N = NP, and P's columns past SC stay zero).
template <int NP, bool UNION, int SC>
__global__ void __launch_bounds__(kMlaThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_u32);

  const int slot_cap = UNION ? 0 : p.slot_cap;
  const MlaSmemLayout L = mla_smem_layout(NP, p.pair_stages, slot_cap);
  const int RP = p.pair_stages;
  const int E = RP - kMlaPairs;        // latent chunks of S(j+1) issued before P.V(j): 0 or 1

  const uint32_t b_lfull = base + L.bars;          // latent stage full [RP]
  const uint32_t b_lempty = b_lfull + 8 * RP;      // latent stage empty [RP]
  const uint32_t b_rfull = b_lempty + 8 * RP;      // rope stage full
  const uint32_t b_rempty = b_rfull + 8;           // rope stage empty
  const uint32_t b_sfull = b_rempty + 8;           // [2]
  const uint32_t b_sfree = b_sfull + 16;
  const uint32_t b_pfull = b_sfree + 16;
  const uint32_t b_pvdone = b_pfull + 16;
  const uint32_t b_itemfull = b_pvdone + 16;
  const uint32_t b_itemempty = b_itemfull + 16;
  const uint32_t b_qempty = b_itemempty + 16;
  const uint32_t b_qfull = b_qempty + 8;
  const uint32_t b_fin = b_qfull + 8;

  MlaItem* const info = reinterpret_cast<MlaItem*>(gbase + L.misc);
  float* const red = reinterpret_cast<float*>(gbase + L.misc + 2 * sizeof(MlaItem));  // [2][4][NP]
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.misc + 2 * sizeof(MlaItem) +
                                                          2 * 4 * NP * sizeof(float));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* const vote = reinterpret_cast<int*>(tmem_slot + 2);   // [3]
  int32_t* const status = p.status;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RP; ++s) {
      mbar_init(b_lfull + 8 * s, kMlaPairOwners);   // each latent warp arms its share
      mbar_init(b_lempty + 8 * s, 1);
    }
    mbar_init(b_rfull, kMlaRopeWarps);   // each rope warp arms its share
    mbar_init(b_rempty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_sfull + 8 * b, 1);
      mbar_init(b_sfree + 8 * b, 128);
      mbar_init(b_pfull + 8 * b, 128);
      mbar_init(b_pvdone + 8 * b, 1);
      mbar_init(b_itemfull + 8 * b, 1);
      mbar_init(b_itemempty + 8 * b, 1 + 128 + kMlaProducerWarps);
    }
    mbar_init(b_qempty, 1);
    mbar_init(b_qfull, 1);
    mbar_init(b_fin, 1);
    *abort_flag = 0;
    vote[0] = 0;
    vote[1] = 0;
    vote[2] = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  if (warp == kGatherWarp0 && lane == 0) prefetch_tmap(&tmKV);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tm_s0 = tmem_base;              // S^T buffers: columns [0, NP), [NP, 2NP)
  const uint32_t tm_o = tmem_base + 2 * NP;      // O^T chunks c: [(2+c)NP, (3+c)NP)

  const int64_t n_items = p.n_items;
  const int64_t stride = gridDim.x;
  // Every role ends here and returns (no code shared by warpgroups with different register
  // counts after the reallocation).
  auto finish_role = [&]() {
    tc_fence_before();
    __syncthreads();
  };

  if (warp == kIndexWarp) {
    regs_inc<kRoleRegs>();
    // ------------------------------------------------------------ index / Q loader
    // Items as in the d=256 kernel: static round robin, or (union mode) longest-first from a
    // global counter; a record with n_valid = -1 ends every role.
    auto next_item = [&](int64_t cur) -> int64_t {
      if (p.item_counter == nullptr) return cur + stride;
      int32_t k = 0;
      if (lane == 0) k = atomicAdd(p.item_counter, 1);
      k = __shfl_sync(0xffffffffu, k, 0);
      return k < n_items ? n_items - 1 - k : n_items;
    };
    uint32_t it = 0;
    for (int64_t item = p.item_counter == nullptr ? static_cast<int64_t>(blockIdx.x) : next_item(0);;
         item = next_item(item), ++it) {
      // failure-detection test hook: withhold the first item so every other wait runs out
      if (p.stall_first_item) break;
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mla_wait(b_itemempty + 8 * b, ph ^ 1, abort_flag, status, kMItemEmpty)))
        break;
      if (item >= n_items) {
        if (lane == 0) {
          info[b].n_valid = -1;
          mbar_arrive(b_itemfull + 8 * b);
        }
        break;
      }
      const int32_t chunk = static_cast<int32_t>(item / p.n_groups);
      const int32_t group = static_cast<int32_t>(item - static_cast<int64_t>(chunk) * p.n_groups);
      int32_t cols, row0, rows_in_group;
      if (UNION) {
        row0 = group * p.union_g;
        rows_in_group = static_cast<int32_t>(p.n_rows - row0 < p.union_g ? p.n_rows - row0 : p.union_g);
        cols = rows_in_group * p.n_heads;
      } else {
        row0 = group;
        rows_in_group = 1;
        cols = min(p.chunk_cols, p.n_heads - chunk * p.chunk_cols);
      }
      int32_t nv;
      if (!UNION) {
        int32_t Lr = p.topk;
        if (p.topk_len) Lr = min(max(p.topk_len[row0], 0), p.topk);
        int32_t* const sl = reinterpret_cast<int32_t*>(gbase + L.slots) + b * slot_cap;
        const uint32_t sl_u32 = base + L.slots + b * slot_cap * 4;
        nv = compact_row_slots(p.indices + static_cast<int64_t>(row0) * p.topk, Lr, sl, sl_u32,
                               p.n_kv_slots, 1, 0, p.pad_row, p.pa, row0, lane);
      } else {
        nv = p.union_len[group];
      }
      if (lane == 0) {
        MlaItem& I = info[b];
        I.n_valid = nv;
        I.group = group;
        I.chunk = chunk;
        I.cols = cols;
        I.row0 = row0;
        I.rows_in_group = rows_in_group;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(b_itemfull + 8 * b);
      // Q tile: rows = query columns (NP, zero past cols), 9 atoms of 64 dims, SW128 K-major.
      if (!__all_sync(0xffffffffu, mla_wait(b_qempty, (it & 1) ^ 1, abort_flag, status, kMQEmpty))) break;
      const uint32_t qb = base + L.qbuf;
#pragma unroll 4
      for (int c = 0; c < NP; ++c) {
        const uint16_t* src = nullptr;
        if (c < cols) {
          int64_t row, head;
          if (UNION) {
            row = row0 + c / p.n_heads;
            head = c % p.n_heads;
          } else {
            row = row0;
            head = static_cast<int64_t>(chunk) * p.chunk_cols + c;
          }
          src = p.q + (row * p.n_heads + head) * kMlaDqk;
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int ch = lane + 32 * k;                   // 16-byte chunk of the 1152-byte row
          if (ch < kMlaDqk / 8) {
            const uint4 v = src ? mla_ldg_v4(src + ch * 8) : make_uint4(0u, 0u, 0u, 0u);
            mla_sts_v4(qb + (ch >> 3) * (NP * 128) + (c >> 3) * 1024 + (c & 7) * 128 +
                           (((ch & 7) ^ (c & 7)) << 4), v);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qfull);
    }
    finish_role();
    return;
  } else if (warp >= kGatherWarp0 || is_gather_warp(warp)) {
    // ------------------------------------------------------------ gather producers
    // Warps 6 and 7 gather at warpgroup 1's register count and warps 8 and 12 stay idle, so the
    // MMA warp's sub-partition keeps one gather warp (the same layout as the d=256 kernel).
    if (warp >= kGatherWarp0) regs_dec<kGatherRegs>(); else regs_inc<kRoleRegs>();
    if (!is_gather_warp(warp)) {
      finish_role();
      return;
    }
    // Gather warps 0-9 share every latent piece: gather4 op o = 32a + lane (o < 64; atom a,
    // slots 4*lane .. 4*lane+3) is issued by warp o % 10, and each warp arms the stage's barrier
    // with its own share of the bytes.  A warp's gather instructions issue one after another
    // (~40 ns each on GB300), and here a freed stage is on the critical path -- the next tile's
    // QK^T waits for it -- so many warps filling it together beat one owner per stage (five
    // warps: mla_8k 4.30 -> 3.61 ms).  Warps 10 and 11 share every rope piece the same way.
    const int pw = gather_index(warp);
    const int rw = pw - kMlaPairOwners;   // rope warp index (>= 0 for the rope warps)
    const uint32_t share_bytes =
        pw < kMlaPairOwners
            ? static_cast<uint32_t>((64 - pw + kMlaPairOwners - 1) / kMlaPairOwners) * 512u
            : static_cast<uint32_t>(32 / kMlaRopeWarps) * 512u;
    uint32_t lseq = 0, rseq = 0, it = 0;
    uint32_t l_issued = 0, r_issued = 0;
    bool aborted = false;
    RingPos lpos;   // ring position of the next latent piece (no division by the stage count)
    for (;; ++it) {
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mla_wait(b_itemfull + 8 * b, ph, abort_flag, status, kMItemFull))) {
        aborted = true;
        break;
      }
      const MlaItem I = info[b];
      if (I.n_valid < 0) break;                // no more items
      const int nv = I.n_valid;
      const int nt = (nv + kTileTokens - 1) / kTileTokens;
      const int32_t* sl = reinterpret_cast<const int32_t*>(gbase + L.slots) + b * slot_cap;
      const int32_t* ul =
          UNION ? p.union_idx + static_cast<int64_t>(I.group) * p.union_g * p.topk : nullptr;
      // tensor-map rows of the lane's four slots of tile `tile`
      auto rows_of = [&](int tile, int& y0, int& y1, int& y2, int& y3) {
        const int t = tile * kTileTokens + 4 * lane;
        int4 v;
        if (UNION) {
          v.x = t + 0 < nv ? ul[t + 0] : p.pad_row;
          v.y = t + 1 < nv ? ul[t + 1] : p.pad_row;
          v.z = t + 2 < nv ? ul[t + 2] : p.pad_row;
          v.w = t + 3 < nv ? ul[t + 3] : p.pad_row;
        } else {
          v = *reinterpret_cast<const int4*>(sl + t);
        }
        y0 = t + 0 < nv ? v.x : p.pad_row;
        y1 = t + 1 < nv ? v.y : p.pad_row;
        y2 = t + 2 < nv ? v.z : p.pad_row;
        y3 = t + 3 < nv ? v.w : p.pad_row;
      };
      // A tile's rows are read once, one tile ahead of their use, so the (global, in union mode)
      // load latency overlaps the previous tile's pieces.
      int n0 = 0, n1 = 0, n2 = 0, n3 = 0;
      if (nt > 0) rows_of(0, n0, n1, n2, n3);
      if (pw < kMlaPairOwners) {
        int y0 = 0, y1 = 0, y2 = 0, y3 = 0;
        for (int q = 0; q < kMlaPairs * nt; ++q) {
          const uint32_t s = lseq + q;
          const uint32_t st = lpos.st, lpar = lpos.par;
          ring_next(lpos, RP);
          const int tile = q / kMlaPairs, c = q % kMlaPairs;
          if (c == 0) {
            y0 = n0; y1 = n1; y2 = n2; y3 = n3;
            if (tile + 1 < nt) rows_of(tile + 1, n0, n1, n2, n3);
          }
          if (!__all_sync(0xffffffffu, mla_wait(b_lempty + 8 * st, lpar ^ 1, abort_flag, status,
                                                kMLatEmpty))) {
            aborted = true;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(b_lfull + 8 * st, share_bytes);
          __syncwarp();
          const uint32_t stage = base + L.pairs + st * kStageBytes;
#pragma unroll
          for (int a = 0; a < 2; ++a)
            if ((32 * a + lane) % kMlaPairOwners == pw)
              tma_gather4(stage + a * 16384 + lane * 512, &tmKV, 128 * c + 64 * a, y0, y1, y2, y3,
                          b_lfull + 8 * st);
          l_issued = s + 1;
        }
      } else {
        for (int j = 0; j < nt; ++j) {
          const uint32_t s = rseq + j;
          const int y0 = n0, y1 = n1, y2 = n2, y3 = n3;
          if (j + 1 < nt) rows_of(j + 1, n0, n1, n2, n3);
          if (!__all_sync(0xffffffffu, mla_wait(b_rempty, (s & 1) ^ 1, abort_flag, status, kMRopeEmpty))) {
            aborted = true;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(b_rfull, share_bytes);
          __syncwarp();
          if (lane % kMlaRopeWarps == rw)
            tma_gather4(base + L.rope + lane * 512, &tmKV, kMlaDv, y0, y1, y2, y3, b_rfull);
          r_issued = s + 1;
        }
      }
      if (aborted) break;
      lseq += kMlaPairs * nt;
      rseq += nt;
      __syncwarp();
      if (lane == 0) mbar_arrive(b_itemempty + 8 * b);
    }
    if (aborted && lane == 0) {
      // Drain: let the newest copy of every stage this warp shared in land (bounded).
      if (pw < kMlaPairOwners) {
        for (uint32_t s = l_issued > static_cast<uint32_t>(RP) ? l_issued - RP : 0; s < l_issued; ++s)
          mla_drain(b_lfull + 8 * (s % RP), (s / RP) & 1, status, kMlaDrainNs);
      } else if (r_issued > 0) {
        mla_drain(b_rfull, (r_issued - 1) & 1, status, kMlaDrainNs);
      }
    }
    finish_role();
    return;
  } else if (warp == kMmaWarp) {
    regs_inc<kRoleRegs>();
    // ------------------------------------------------------------ MMA issuer (one thread)
    constexpr uint32_t kIdescQK = idesc_bf16_f32(128, NP, false, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(128, NP, true, false);
    uint32_t rseq = 0, js = 0, it = 0;
    bool aborted = false;
    const uint32_t qaddr = base + L.qbuf;
    const uint32_t rope_addr = base + L.rope;
    // Latent pieces are read twice, each time in ring order: by QK^T (qk_pos) and, a tile
    // later, by P.V (pv_pos); running positions replace divisions by the stage count on the
    // issue path.
    RingPos qk_pos, pv_pos;
    auto lstage = [&](uint32_t st) { return base + L.pairs + st * kStageBytes; };
    // Operand descriptors as a per-buffer low word plus a constant offset: one add per operand
    // on the issue path (sw128_desc_lo / sw128_desc_hi).
    constexpr uint32_t kHi = sw128_desc_hi(1024);
    const uint32_t q_lo = sw128_desc_lo(qaddr, 16);
    const uint32_t rope_lo = sw128_desc_lo(rope_addr, 16);
    // S^T(sbuf) += latent chunk c (dims 128c .. 128c+127) of the tile held in `st_addr`
    auto qk_chunk = [&](uint32_t sb, int c, uint32_t st_addr, bool first) {
      const uint32_t a_lo = sw128_desc_lo(st_addr, 16);
#pragma unroll
      for (int kq = 0; kq < 8; ++kq) {
        const int g = 8 * c + kq;
        const uint32_t a_off = (kq >> 2) * 16384 + (kq & 3) * 32;
        const uint32_t b_off = (g >> 2) * (NP * 128) + (g & 3) * 32;
        tc_mma_w(tm_s0 + sb * NP, a_lo + (a_off >> 4), kHi, q_lo + (b_off >> 4), kHi, kIdescQK,
                 (first && kq == 0) ? 0u : 1u);
      }
    };
    // S^T(sbuf) += rope dims 512 .. 575
    auto qk_rope = [&](uint32_t sb, bool first) {
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const int g = 32 + kq;
        const uint32_t b_off = (g >> 2) * (NP * 128) + (g & 3) * 32;
        tc_mma_w(tm_s0 + sb * NP, rope_lo + ((kq * 32) >> 4), kHi, q_lo + (b_off >> 4), kHi,
                 kIdescQK, (first && kq == 0) ? 0u : 1u);
      }
    };
    // O^T chunk c += V^T(chunk c of the tile in st_addr) . P^T(pbuf)
    auto pv_chunk = [&](int c, uint32_t st_addr, uint32_t pbase, bool first) {
      const uint32_t a_lo = sw128_desc_lo(st_addr, 16384);
      const uint32_t p_lo = sw128_desc_lo(pbase, 16);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t b_off = (kk >> 2) * (NP * 128) + (kk & 3) * 32;
        tc_mma_w(tm_o + c * NP, a_lo + ((kk * 2048) >> 4), kHi, p_lo + (b_off >> 4), kHi, kIdescPV,
                 (first && kk == 0) ? 0u : 1u);
      }
    };
    for (;; ++it) {
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mla_wait(b_itemfull + 8 * b, ph, abort_flag, status, kMItemFull))) {
        aborted = true;
        break;
      }
      const int nv = info[b].n_valid;
      if (nv < 0) break;                        // no more items
      const int nt = (nv + kTileTokens - 1) / kTileTokens;
      __syncwarp();
      if (lane == 0) mbar_arrive(b_itemempty + 8 * b);
      if (!__all_sync(0xffffffffu, mla_wait(b_qfull, it & 1, abort_flag, status, kMQFull))) {
        aborted = true;
        break;
      }
      if (nt == 0) {
        if (lane == 0) tc_commit(b_qempty);
        __syncwarp();
        continue;
      }
      // ---- S(0): all latent chunks and the rope chunk
      {
        const uint32_t sb = js & 1, sph = (js >> 1) & 1;
        bool ok = mla_wait(b_sfree + 8 * sb, sph ^ 1, abort_flag, status, kMSFree);
        for (int c = 0; c < kMlaPairs && ok; ++c) {
          const RingPos at = qk_pos;
          ring_next(qk_pos, RP);
          ok = mla_wait(b_lfull + 8 * at.st, at.par, abort_flag, status, kMLatFull);
          if (ok) {
            tc_fence_after();
            if (lane == 0) qk_chunk(sb, c, lstage(at.st), c == 0);
          }
        }
        ok = ok && mla_wait(b_rfull, rseq & 1, abort_flag, status, kMRopeFull);
        if (!__all_sync(0xffffffffu, ok)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          qk_rope(sb, false);
          tc_commit(b_rempty);
          tc_commit(b_sfull + 8 * sb);
          if (nt == 1) tc_commit(b_qempty);
        }
        __syncwarp();
      }
      for (int j = 0; j < nt; ++j) {
        const int jj = j + 1;
        const uint32_t jsn = js + jj, sbn = jsn & 1, sphn = (jsn >> 1) & 1;
        bool ok = true;
        // ---- early part of S(j+1): E latent chunks and the rope chunk
        if (jj < nt) {
          ok = mla_wait(b_sfree + 8 * sbn, sphn ^ 1, abort_flag, status, kMSFree);
          for (int c = 0; c < E && ok; ++c) {
            const RingPos at = qk_pos;
            ring_next(qk_pos, RP);
            ok = mla_wait(b_lfull + 8 * at.st, at.par, abort_flag, status, kMLatFull);
            if (ok) {
              tc_fence_after();
              if (lane == 0) qk_chunk(sbn, c, lstage(at.st), c == 0);
            }
          }
          ok = ok && mla_wait(b_rfull, (rseq + jj) & 1, abort_flag, status, kMRopeFull);
          if (ok) {
            tc_fence_after();
            if (lane == 0) {
              qk_rope(sbn, E == 0);
              tc_commit(b_rempty);
            }
          }
        }
        // ---- P.V(j), releasing each latent piece after its output chunk
        const uint32_t jsp = js + j, pb = jsp & 1, pph = (jsp >> 1) & 1;
        ok = ok && mla_wait(b_pfull + 8 * pb, pph, abort_flag, status, kMPFull);
        if (!__all_sync(0xffffffffu, ok)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const RingPos pv_at = pv_pos;   // every lane keeps the position; lane 0 issues
        for (int c = 0; c < kMlaPairs; ++c) ring_next(pv_pos, RP);
        if (lane == 0) {
          const uint32_t pbase = base + L.pbuf + pb * L.p_bytes;
          RingPos at = pv_at;
          for (int c = 0; c < kMlaPairs; ++c) {
            pv_chunk(c, lstage(at.st), pbase, j == 0);
            tc_commit(b_lempty + 8 * at.st);
            ring_next(at, RP);
          }
          tc_commit(b_pvdone + 8 * pb);
        }
        __syncwarp();
        // ---- rest of S(j+1)
        if (jj < nt) {
          for (int c = E; c < kMlaPairs && ok; ++c) {
            const RingPos at = qk_pos;
            ring_next(qk_pos, RP);
            ok = mla_wait(b_lfull + 8 * at.st, at.par, abort_flag, status, kMLatFull);
            if (ok) {
              tc_fence_after();
              if (lane == 0) qk_chunk(sbn, c, lstage(at.st), false);
            }
          }
          if (!__all_sync(0xffffffffu, ok)) {
            aborted = true;
            break;
          }
          if (lane == 0) {
            tc_commit(b_sfull + 8 * sbn);
            if (jj == nt - 1) tc_commit(b_qempty);
          }
          __syncwarp();
        }
      }
      if (aborted) break;
      rseq += nt;
      js += nt;
    }
    // Every MMA this thread issued has completed once `fin` flips.
    if (lane == 0) {
      tc_commit(b_fin);
      mla_drain(b_fin, 0, status, aborted ? kMlaDrainNs : kMlaWaitNs);
    }
    __syncwarp();
    finish_role();
    tc_fence_after();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    return;
  } else if (warp < kSoftmaxWarps) {
    regs_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + epilogue (warps 0-3)
    const int t = threadIdx.x;                       // tensor-memory lane = slot within tile
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t js = 0, it = 0, rb = 0;
    bool bad = false;
    const float NEG_INF = -INFINITY;
    if constexpr (SC < NP) {
      // P columns SC .. NP-1 are never written: zero both P buffers once (the MMA reads them)
      for (int i = t; i < 2 * L.p_bytes / 16; i += 128)
        mla_sts_v4(base + L.pbuf + 16 * i, make_uint4(0u, 0u, 0u, 0u));
      fence_proxy_async_smem();
    }
    for (;; ++it) {
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      bad |= !mla_wait(b_itemfull + 8 * b, ph, abort_flag, status, kMItemFull);
      // Uniform decision before the item record is read (see the d=256 kernel).
      if (named_bar_any(3, 128, bad || *abort_flag)) break;
      const MlaItem I = info[b];
      if (I.n_valid < 0) break;                // no more items (same record for all 128)
      mbar_arrive(b_itemempty + 8 * b);
      const int nv = I.n_valid;
      const int nt = (nv + kTileTokens - 1) / kTileTokens;
      const int cols = I.cols;
      uint64_t colmask[8];
      const uint64_t allcols = (cols >= 64) ? ~0ull : ((1ull << cols) - 1ull);
      if (UNION) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int lo = u * p.n_heads, hi = min((u + 1) * p.n_heads, cols);
          uint64_t m = 0;
          if (lo < hi) {
            const uint64_t upto = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
            const uint64_t below = lo >= 64 ? ~0ull : ((1ull << lo) - 1ull);
            m = upto & ~below;
          }
          colmask[u] = m;
        }
      }
      const uint8_t* ub =
          UNION ? p.union_bits + static_cast<int64_t>(I.group) * p.union_g * p.topk : nullptr;
      // columns past the real ones start at a finite max of 0 (see the fully valid tiles below)
      float m_used[NP], l_part[NP];
#pragma unroll
      for (int c = 0; c < NP; ++c) {
        m_used[c] = c < cols ? NEG_INF : 0.f;
        l_part[c] = 0.f;
      }
      uint32_t bits_next = 0;
      if (UNION && nt > 0) bits_next = t < nv ? ub[t] : 0u;
      bool quit = false;
      for (int j = 0; j < nt; ++j) {
        const uint32_t jsj = js + j, sb = jsj & 1, sph = (jsj >> 1) & 1;
        const int token = j * kTileTokens + t;
        const bool valid = token < nv;
        uint64_t vmask = valid ? allcols : 0ull;
        if (UNION) {
          const uint32_t bits = bits_next;
          if (j + 1 < nt) bits_next = (token + kTileTokens) < nv ? ub[token + kTileTokens] : 0u;
          uint64_t m = 0;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if ((bits >> u) & 1u) m |= colmask[u];
          vmask &= m;
        }
        bad |= !mla_wait(b_sfull + 8 * sb, sph, abort_flag, status, kMSFull);
        tc_fence_after();
        float x[NP];
#pragma unroll
        for (int q = 0; q < NP / 16; ++q) tmem_ld16(tm_s0 + lane_off + sb * NP + 16 * q, x + 16 * q);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(b_sfree + 8 * sb);
        // As in the d=256 kernel: per-token warps whose slots are all valid skip the per-column
        // masking and the -inf guard (padding columns see S = 0, a max of 0 and P = 1, feeding
        // only unread O^T columns); columns past SC are not computed.
        const bool full = !UNION && __all_sync(0xffffffffu, vmask == allcols);
        bool need = false;
        if (full) {
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            if (c >= SC) {
              x[c] = NEG_INF;
              continue;
            }
            x[c] *= p.scale_log2;
            need |= x[c] > m_used[c] + kMlaRescale;
          }
        } else {
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            if (c >= SC) {
              x[c] = NEG_INF;
              continue;
            }
            x[c] = ((vmask >> c) & 1ull) ? x[c] * p.scale_log2 : NEG_INF;
            need |= x[c] > m_used[c] + kMlaRescale;
          }
        }
        const int myvote = (need ? 1 : 0) | ((bad || *abort_flag) ? 2 : 0);
        if (myvote) atomicOr(&vote[jsj % 3], myvote);
        named_bar_sync(2, 128);
        const int f = vote[jsj % 3];
        if (t == 0) vote[(jsj + 2) % 3] = 0;
        if (f & 2) {
          quit = true;
          break;
        }
        if (f & 1) {
          float* rbuf = red + rb * 4 * NP;
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            float v = x[c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) rbuf[warp * NP + c] = v;
          }
          named_bar_sync(1, 128);
          float alpha[NP];
          bool any_scale = false;
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            const float tmax = fmaxf(fmaxf(rbuf[c], rbuf[NP + c]), fmaxf(rbuf[2 * NP + c], rbuf[3 * NP + c]));
            const float m_new = fmaxf(m_used[c], tmax);
            alpha[c] = (m_new == NEG_INF) ? 1.f : fast_exp2(m_used[c] - m_new);
            any_scale |= alpha[c] != 1.f;
            m_used[c] = m_new;
            l_part[c] *= alpha[c];
          }
          rb ^= 1;
          if (j > 0 && any_scale) {
            // O^T columns shrink by alpha once the previous tile's P.V has landed.
            const uint32_t jprev = jsj - 1;
            bad |= !mla_wait(b_pvdone + 8 * (jprev & 1), (jprev >> 1) & 1, abort_flag, status, kMPvDone);
            tc_fence_after();
#pragma unroll
            for (int oc = 0; oc < kMlaPairs; ++oc) {
#pragma unroll
              for (int q = 0; q < NP / 16; ++q) {
                float o[16];
                const uint32_t ta = tm_o + lane_off + oc * NP + 16 * q;
                tmem_ld16(ta, o);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] *= alpha[16 * q + i];
                tmem_st16(ta, o);
              }
            }
            tc_wait_st();
          }
        }
        // P buffer sb is free once the P.V of tile jsj-2 has completed.
        bad |= !mla_wait(b_pvdone + 8 * sb, sph ^ 1, abort_flag, status, kMPvDone);
        uint8_t* pbuf = gbase + L.pbuf + sb * L.p_bytes;
        uint8_t* prow = pbuf + (t >> 6) * (NP * 128) + ((t & 7) << 1);
        const int tchunk = (t & 63) >> 3;
        auto store_p = [&](int c, float pv) {
          l_part[c] += pv;
          const __nv_bfloat16 pb16 = __float2bfloat16_rn(pv);
          *reinterpret_cast<__nv_bfloat16*>(prow + (c >> 3) * 1024 + (c & 7) * 128 +
                                            ((tchunk ^ (c & 7)) << 4)) = pb16;
        };
        if (full) {
#pragma unroll
          for (int c = 0; c < SC; ++c) store_p(c, fast_exp2(x[c] - m_used[c]));
        } else {
#pragma unroll
          for (int c = 0; c < SC; ++c) store_p(c, x[c] == NEG_INF ? 0.f : fast_exp2(x[c] - m_used[c]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(b_pfull + 8 * sb);
      }
      if (quit) break;
      // ---- epilogue: row sums, O / l, LSE
      float* rbuf = red + rb * 4 * NP;
#pragma unroll
      for (int c = 0; c < NP; ++c) {
        float v = l_part[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) rbuf[warp * NP + c] = v;
      }
      named_bar_sync(1, 128);
      // Thread t < cols finishes column t once (row sum, 1 / l, LSE, output offset) into the
      // other reduction buffer, whose last readers passed the barrier above.
      float* const inv_s = red + (rb ^ 1) * 4 * NP;
      int64_t* const off_s = reinterpret_cast<int64_t*>(inv_s + NP);
      const int64_t H = p.n_heads;
      if (t < cols) {
        const float l = (rbuf[t] + rbuf[NP + t]) + (rbuf[2 * NP + t] + rbuf[3 * NP + t]);
        float my_m = NEG_INF;
#pragma unroll
        for (int c = 0; c < NP; ++c)
          if (c == t) my_m = m_used[c];
        int64_t row, head;
        if (UNION) {
          row = I.row0 + t / p.n_heads;
          head = t % p.n_heads;
        } else {
          row = I.row0;
          head = static_cast<int64_t>(I.chunk) * p.chunk_cols + t;
        }
        inv_s[t] = l > 0.f ? 1.f / l : 0.f;
        off_s[t] = (row * H + head) * kMlaDv;
        if (p.lse != nullptr) p.lse[row * H + head] = l > 0.f ? (my_m + log2f(l)) * kMlaLn2 : NEG_INF;
      }
      named_bar_sync(1, 128);
      rb ^= 1;
      if (nt > 0) {
        const uint32_t jl = js + nt - 1;
        bad |= !mla_wait(b_pvdone + 8 * (jl & 1), (jl >> 1) & 1, abort_flag, status, kMPvDone);
        tc_fence_after();
      }
      __nv_bfloat16* const outp = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
      for (int oc = 0; oc < kMlaPairs; ++oc) {
        const int d = oc * 128 + t;
#pragma unroll
        for (int q = 0; q < NP / 16; ++q) {
          if (16 * q >= cols) break;
          float o[16];
          if (nt > 0) {
            tmem_ld16(tm_o + lane_off + oc * NP + 16 * q, o);
            tc_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 16 * q + i;
            if (c < cols) outp[off_s[c] + d] = __float2bfloat16_rn(o[i] * inv_s[c]);
          }
        }
      }
      tc_fence_before();
      js += nt;
    }
    finish_role();
    return;
  }
  // every warp of the CTA has returned from its role above
}

namespace {

template <int NP, bool UNION, int SC = NP>
cudaError_t launch_mla_np(const CUtensorMap& tm, const MlaParams& p, const MlaGeometry& g,
                          cudaStream_t stream) {
  auto kern = sparse_mla_kernel<NP, UNION, SC>;
  static std::atomic<int> opted_in[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || opted_in[dev].load() < g.smem_bytes) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) opted_in[dev].store(g.smem_bytes);
  }
  kern<<<g.grid, kMlaThreads, g.smem_bytes, stream>>>(tm, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mla(const MlaParams& p, const MlaGeometry& g, const void* kv_cache,
                       int64_t tmap_rows, cudaStream_t stream) {
  if (g.n_items == 0) return cudaSuccess;
  CUtensorMap tm;
  const cudaError_t e = make_cache_map(&tm, kv_cache, tmap_rows, kMlaDqk);
  if (e != cudaSuccess) return e;
  const bool u = p.union_g > 1;
  switch (g.np) {
    case 16: return u ? launch_mla_np<16, true>(tm, p, g, stream)
                      : (g.cols <= 8 ? launch_mla_np<16, false, 8>(tm, p, g, stream)
                                     : launch_mla_np<16, false>(tm, p, g, stream));
    case 32: return u ? launch_mla_np<32, true>(tm, p, g, stream) : launch_mla_np<32, false>(tm, p, g, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qsa
