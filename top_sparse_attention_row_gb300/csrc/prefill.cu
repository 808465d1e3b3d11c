// Top-k sparse attention prefill kernel for sm_103a (tcgen05 + TMA gather4).
//
// What it computes ("[QSA] Tune sm120 sparse prefill geometry", Motivation; "DSA prefill ...
// triton_sparse_mla", Motivation and Modifications): for every query row, the query heads
// that share one KV head attend over the K/V rows gathered at the row's selected slots
// (negative = padding, topk_len leading slots), scaled dot product, online softmax, and the
// kernel writes O (bf16) and the natural-log LSE (fp32) with no split-K partials.  In union
// mode a work item is G adjacent rows sharing the union of their slots; an ownership bit per
// (slot, row) masks every row's logits to its own support.
//
// Design (GB300-first, not the pages' Triton tiling):
//  * One persistent CTA per SM walks work items (row group x KV head x head chunk), KV-head
//    major so all CTAs stream one KV head's cache at a time (L2 locality).
//  * The MMA is "swap-AB": the gathered slots are the MMA M dimension (128 per tile) and the
//    query columns of the item (heads, or G x heads in union mode) are N, padded to 16 --
//    instead of padding the head dimension up to the MMA M.
//      S^T[128 x N]  = K_tile[128 x 256] . Q^T            (A: K-major SW128, B: K-major SW128)
//      O^T[256 x N] += V_tile^T[256 x 128] . P^T[128 x N]  (A: MN-major SW128, B: MN-major SW32 /
//                                                           SW64 for N = 16 / 32, else K-major SW128)
//    Accumulators live in tensor memory: L + 1 S buffers (L = MMA lookahead: 1 per-token, 2
//    union) and the two 128-row halves of O^T.
//  * K/V rows are gathered into a ring of 32 KiB stages (128 slots x 128 dims, 128-byte
//    swizzled rows) in exactly the order the MMA consumes them -- with L = 1: K(0), K(1), V(0),
//    K(2), V(1), ..., V(nt-1), two half-row pieces each -- so the ring drains FIFO; one commit
//    releases a piece pair's two stages, and the MMA thread and the gather warps track ring
//    positions by counting, never by dividing by the (runtime) stage count.  Two gather warps
//    fill each stage, one per 64-dim block: per-SM gather bandwidth grows with the number of
//    warps issuing copies concurrently, and a V tile -- which reuses the stages of the same
//    tile's K, freed when its QK^T completes -- lands in half the time.  Two gather engines:
//    TMA tile::gather4 (default; 4 slots x 128 B per instruction, out-of-bounds rows
//    zero-filled) and cp.async 16-byte copies (lanes arrive on the stage barrier as their copies
//    land and the MMA thread fences them into the async proxy).
//  * FP8 caches (template FP8): a piece's e4m3 rows land in the upper half of the stage and
//    the two gather warps each rewrite 64 of its rows in place as fp16; the MMAs run fp16 operands,
//    the K page scale multiplies the logit and the V page scale (normalised per item) the
//    probability fed to P.V.
//  * Online softmax in registers, one thread per slot (tensor-memory lane), over the SC columns
//    that can hold real heads (template SC <= NP: 8 or 12 for per-token N = 16 tiles).  The
//    running max is only raised when a tile's logits exceed it by more than 2^8 (log2 domain),
//    so the O^T rescale through tensor memory is rare; the result is exact either way because O
//    and the row sum use the same stale max.
//  * Warp roles (20 warps, five warpgroups): 0-3 softmax + epilogue; 4 MMA issue + tensor-memory
//    owner; 5 index/Q loader (per-token: compacts the row's valid slots into shared memory);
//    6, 7, 9-11, 13-19 gather, two per stage; 8 and 12 idle, so that the MMA warp's SM
//    sub-partition (warp index mod 4) has one gather warp instead of three.  Per-token N = 16
//    instances swap warps 5 and 16 (index on 16, at 64 registers), leaving that sub-partition
//    with none.  Warpgroup register reallocation (setmaxnreg) moves registers from the gather
//    warpgroups to the softmax and MMA/index warpgroups.  The MMA issue path builds operand
//    descriptors as per-buffer 32-bit words plus constant offsets.
//  * Per-token calls with fewer items than SMs split each row's tiles over a thread-block
//    cluster and merge (max, row sum, O) through distributed shared memory (split > 1).
//  * Every mbarrier wait is bounded (~2 s); a timeout records a code in a device status word,
//    all roles leave their loops, in-flight copies and MMAs are drained, tensor memory is
//    freed and the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "compact.cuh"
#include "ptx.cuh"

namespace qsa {

__device__ int32_t g_device_status = 0;

namespace {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s per wait
constexpr unsigned long long kDrainLimitNs = 200000000ull;   // 0.2 s per drain wait
constexpr float kRescaleThreshold = 8.0f;                    // log2 units (factor 256)
constexpr float kLn2 = 0.6931471805599453f;

enum WaitSite : int32_t {
  kSiteItemEmpty = 1, kSiteQEmpty, kSiteItemFull, kSiteStageEmpty, kSiteStageFull,
  kSiteSFree, kSiteSFull, kSitePFull, kSitePvDone, kSiteDrain, kSiteQFull, kSiteLanded,
  kSiteMerge
};

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int32_t site, unsigned long long limit) {
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicCAS(&g_device_status, 0, 0x100 | site);
      return false;
    }
  }
}

// Bounded wait that ignores the abort flag: after an abort, lets copies and MMAs already issued
// complete before shared or tensor memory is given up.  (The wait helpers are inlined: a called
// function would have to fit the register budgets of every warpgroup after the reallocation.)
__device__ __forceinline__ bool drain_bar(uint32_t bar, uint32_t parity, unsigned long long limit) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit) {
      atomicCAS(&g_device_status, 0, 0x100 | kSiteDrain);
      return false;
    }
  }
  return true;
}

// Bounded wait on a local mbarrier that other CTAs of the cluster arrive on (acquire at cluster
// scope).  False on timeout or abort.
__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int32_t site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicCAS(&g_device_status, 0, 0x100 | site);
      return false;
    }
  }
}

// Bounded wait for phase `parity` of mbarrier `bar`.  False on timeout or abort.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, abort_flag, site, kWaitLimitNs);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  __nv_bfloat162 b;
  memcpy(&b, &v, 4);
  const float2 f = __bfloat1622float2(b);
  const __half2 h = __floats2half2_rn(f.x, f.y);
  uint32_t r;
  memcpy(&r, &h, 4);
  return r;
}
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  return make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                    bf16x2_to_f16x2(v.w));
}
// Shared-memory descriptor high words for the narrower swizzles (layout type 4 = SWIZZLE_64B,
// 6 = SWIZZLE_32B; the low word as for 128 bytes).  An MN-major operand in these layouts has rows
// of 64 (32) bytes, one per K index, in 8-row atoms of 512 (256) bytes, its 16-byte chunks XORed
// with address bits 7-8 (bit 7).
__host__ __device__ constexpr uint32_t sw64_desc_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (4u << 29);
}
__host__ __device__ constexpr uint32_t sw32_desc_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (6u << 29);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  uint32_t r;
  memcpy(&r, &v, 4);
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  uint32_t r;
  memcpy(&r, &v, 4);
  return r;
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// MMA issue order of an item with lookahead L (lookahead_for): at step j the thread issues
// S^T(j) = K(j).Q^T (j < nt) and then O^T += V(j-L)^T.P^T(j-L) (j >= L), so the softmax of
// tile j has the issue time of L further QK^T groups and L-1 P.V groups before P.V(j) needs it.
// Pieces (two per entry: dims 0-127, 128-255) enter the ring in exactly that order:
//   K(0) .. K(L-1), then K(j), V(j-L) for L <= j < nt, then the remaining V.

template <int L>
__device__ __forceinline__ void piece_of(int q, int nt, int& tile, int& is_v, int& half) {
  const int e = q >> 1;
  half = q & 1;
  if (nt <= L) {
    is_v = e >= nt;
    tile = is_v ? e - nt : e;
  } else if (e < L) {
    is_v = 0;
    tile = e;
  } else if (e < 2 * nt - L) {
    const int d = e - L, j = L + (d >> 1);
    is_v = d & 1;
    tile = is_v ? j - L : j;
  } else {
    is_v = 1;
    tile = e - nt;
  }
}

__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// Arrive (without a pending-count increment) on `bar` once all earlier cp.async of this thread
// have completed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

struct ItemInfo {   // written by the index warp, read by every role
  int32_t n_valid, group, kvh, chunk, cols, row0, rows_in_group;
  float v_scale_max;   // FP8 caches: largest |V page scale| over the item's slots
  int32_t slot0;       // split items: first slot-list entry of this CTA's tile range
};
static_assert(2 * sizeof(ItemInfo) <= 2 * 12 * 4, "item records fit their shared-memory slot");

// One butterfly step of a warp reduce-scatter: lanes with bit `o` set keep the upper half of
// their N values, the others the lower half, and each adds (or maxes in) its partner's copy of
// the half it keeps.
template <int N, bool MAX>
__device__ __forceinline__ void reduce_scatter_step(float* v, bool upper, int o) {
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float send = upper ? v[i] : v[i + N / 2];
    const float keep = upper ? v[i + N / 2] : v[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, o);
    v[i] = MAX ? fmaxf(keep, r) : keep + r;
  }
}

// Warp-wide sum (or max) of each of NP = 16 or 32 per-lane columns in NP - 1 shuffles instead of
// 5 NP: afterwards v[0] of lane l holds column warp_column<NP>(l) reduced over all 32 lanes
// (for NP = 16 lanes l and l ^ 1 hold the same column).  v is overwritten.
template <int NP>
__device__ __forceinline__ int warp_column(int lane) { return NP == 32 ? lane : lane >> 1; }
template <int NP, bool MAX>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NP], int lane) {
  static_assert(NP == 16 || NP == 32, "reduce-scatter covers 16 or 32 columns");
  reduce_scatter_step<NP, MAX>(v, (lane & 16) != 0, 16);
  reduce_scatter_step<NP / 2, MAX>(v, (lane & 8) != 0, 8);
  reduce_scatter_step<NP / 4, MAX>(v, (lane & 4) != 0, 4);
  reduce_scatter_step<NP / 8, MAX>(v, (lane & 2) != 0, 2);
  if constexpr (NP == 32) {
    reduce_scatter_step<2, MAX>(v, (lane & 1) != 0, 1);
  } else {
    const float r = __shfl_xor_sync(0xffffffffu, v[0], 1);
    v[0] = MAX ? fmaxf(v[0], r) : v[0] + r;
  }
  return v[0];
}

// x / d for x >= 0, by a shift when d is a power of two (shift >= 0).
__device__ __forceinline__ int64_t div_by(int64_t x, int32_t d, int32_t shift) {
  return shift >= 0 ? (x >> shift) : x / d;
}

// FP8 caches: index of the page scale of slot `slot`, KV head `kvh`.
__device__ __forceinline__ int64_t scale_index(const PrefillParams& p, int64_t slot, int32_t kvh) {
  return div_by(slot, p.page_size, p.page_shift) * p.n_kvheads + kvh;
}

__device__ __forceinline__ void decode_item(const PrefillParams& p, int64_t item, int32_t& group,
                                            int32_t& kvh, int32_t& chunk) {
  const int64_t per_kv = static_cast<int64_t>(p.head_chunks) * p.n_groups;
  kvh = static_cast<int32_t>(item / per_kv);
  const int64_t rem = item - static_cast<int64_t>(kvh) * per_kv;
  chunk = static_cast<int32_t>(rem / p.n_groups);
  group = static_cast<int32_t>(rem - static_cast<int64_t>(chunk) * p.n_groups);
}

}  // namespace

// SC: query columns the softmax computes (SC < NP when an item's real columns fit in SC; the MMA
// still runs N = NP, and P's columns past SC stay zero).
template <int NP, bool UNION, bool FP8, int SC>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_prefill_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_u32);

  constexpr int kLookahead = lookahead_for(UNION);
  constexpr int kBPS = kBlocksPerStage;   // gather warps per stage, one per 64-dim block
  constexpr int kSBufs = kLookahead + 1;
  const int slot_cap = UNION ? 0 : p.slot_cap;
  // Split items (per-token bf16 tiles of at most 32 columns): the CTAs of a cluster share an
  // item.  FP8 instances are left without the split: its merge code in the softmax warpgroup cost
  // the FP8 per-token kernel 6 % on full-size calls (measured), through register allocation.
  constexpr bool kCanSplit = !UNION && !FP8 && NP <= kSplitMaxNPad;
  const int split = kCanSplit ? p.split : 1;
  // P^T is stored MN-major (a slot's columns contiguous, one 16-byte store per eight columns)
  // where N fits one 32- or 64-byte swizzle row; wider tiles keep the K-major 128-byte layout.
  constexpr bool kPMnMajor = NP == 16 || NP == 32;
  const SmemLayout L = smem_layout(NP, p.stages, slot_cap, FP8, split);
  const int R = p.stages;

  // barrier addresses
  const uint32_t b_full = base + L.bars;
  const uint32_t b_empty = b_full + 8 * R;
  const uint32_t b_sfull = b_empty + 8 * R;     // [kSBufs]
  const uint32_t b_sfree = b_sfull + 8 * kMaxSBufs;
  const uint32_t b_pfull = b_sfree + 8 * kMaxSBufs;
  const uint32_t b_pvdone = b_pfull + 16;
  const uint32_t b_itemfull = b_pvdone + 16;
  const uint32_t b_itemempty = b_itemfull + 16;
  const uint32_t b_qempty = b_itemempty + 16;     // Q buffer free (MMA commit, once per item)
  const uint32_t b_qfull = b_qempty + 8;          // Q buffer written (index warp, once per item)
  const uint32_t b_fin = b_qempty + 16;           // MMA issuer drained
  const uint32_t b_recv = b_fin + 8;              // split: every CTA's partials have arrived
  const uint32_t b_sendok = b_fin + 16;           // split: every CTA has read this one's partials
  const uint32_t b_land = b_fin + 24;             // FP8: a block's e4m3 bytes landed [R][2]

  ItemInfo* const info = reinterpret_cast<ItemInfo*>(gbase + L.misc);
  float* const red = reinterpret_cast<float*>(gbase + L.misc + 2 * sizeof(ItemInfo));  // [2][4][NP]
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.misc + 2 * sizeof(ItemInfo) +
                                                          2 * 4 * NP * sizeof(float));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* const vote = reinterpret_cast<int*>(tmem_slot + 2);   // [3]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < R; ++s) {
      // TMA: one expect_tx per gather warp; FP8: each warp arrives after rewriting its block;
      // cp.async: every lane of both warps
      mbar_init(b_full + 8 * s, (FP8 || p.gather_tma) ? kBPS : 32 * kBPS);
      mbar_init(b_empty + 8 * s, 1);   // stage pairs share empty[pair]: [0, R/2) are used
      if (FP8)
        for (int c = 0; c < kBPS; ++c) mbar_init(b_land + 8 * (kBPS * s + c), 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(b_sfull + 8 * b, 1);
      mbar_init(b_sfree + 8 * b, 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_pfull + 8 * b, 128);
      mbar_init(b_pvdone + 8 * b, 1);
      mbar_init(b_itemfull + 8 * b, 1);
      mbar_init(b_itemempty + 8 * b, 1 + 128 + kProducerWarps);
    }
    mbar_init(b_qempty, 1);
    mbar_init(b_qfull, 1);
    mbar_init(b_fin, 1);
    mbar_init(b_recv, 128 * split);     // 128 softmax threads of every CTA of the cluster
    mbar_init(b_sendok, 128 * split);
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
  if (warp == kGatherWarp0 && lane == 0 && p.gather_tma) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  // split items: every CTA's barriers are initialised before any CTA of the cluster can arrive
  // on them remotely
  if (split > 1) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tm_s0 = tmem_base;                 // S^T buffers: columns [b NP, (b+1) NP)
  const uint32_t tm_o = tmem_base + kSBufs * NP;    // O^T halves: the next 2 NP columns

  const int64_t n_items = p.n_items;
  // Per-token items go round robin over the grid's clusters (a cluster is one CTA unless items
  // are split); every CTA of a cluster takes the same items.
  const uint32_t crank = split > 1 ? cluster_ctarank() : 0u;
  const int64_t first_item = static_cast<int64_t>(blockIdx.x) / split;
  const int64_t stride = static_cast<int64_t>(gridDim.x) / split;
  // Every role ends here and returns, so no code is shared by warpgroups that run with
  // different register counts after the reallocation below.
  auto finish_role = [&]() {
    tc_fence_before();
    __syncthreads();
    // no CTA of a split cluster leaves while another may still access its shared memory
    if (split > 1) cluster_sync_all();
  };

  // Per-token tiles of N = 16 (the group-6 and group-12 shapes) move the index warp to warp 16
  // and let warp 5 gather: the MMA warp's sub-partition then holds no gather warp.  Its 64
  // registers hold Q rows for 8 columns ahead instead of 16; wider instances spill there and keep
  // the index warp on warp 5 (measured on GB300: group6_32k 1.539 -> 1.506 ms, FP8 1.874 ->
  // 1.592 ms; union G = 4 0.501 -> 0.595 ms with the move).
  constexpr bool kIdxSub0 = !UNION && NP == 16;
  constexpr int kIdxWarp = kIdxSub0 ? 16 : kIndexWarp;
  if (warp == kIdxWarp) {
    // ------------------------------------------------------------ index / Q loader
    if constexpr (kIdxSub0) regs_dec<kGatherRegs>(); else regs_inc<kRoleRegs>();
    // Items: a static round robin over the grid, or (union mode) taken from a global counter in
    // reverse order -- the later row groups of a prefill have the longest union lists, so the
    // long items go first and the short ones even out the CTAs' finishing times.  After the
    // last item the warp publishes an item record with n_valid = -1, which ends every role.
    auto next_item = [&](int64_t cur) -> int64_t {
      if (p.item_counter == nullptr) return cur + stride;
      int32_t k = 0;
      if (lane == 0) k = atomicAdd(p.item_counter, 1);
      k = __shfl_sync(0xffffffffu, k, 0);
      return k < n_items ? n_items - 1 - k : n_items;
    };
    uint32_t it = 0;
    for (int64_t item = p.item_counter == nullptr ? first_item : next_item(0);;
         item = next_item(item), ++it) {
      // failure-detection test hook: withhold the first item so every other wait runs out
      if (p.stall_first_item) break;
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      bool ok = wait_bar(b_itemempty + 8 * b, ph ^ 1, abort_flag, kSiteItemEmpty);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (item >= n_items) {
        if (lane == 0) {
          info[b].n_valid = -1;
          mbar_arrive(b_itemfull + 8 * b);
        }
        break;
      }
      int32_t group, kvh, chunk;
      decode_item(p, item, group, kvh, chunk);
      int32_t cols, row0, rows_in_group;
      if (UNION) {
        row0 = group * p.union_g;
        rows_in_group = static_cast<int32_t>(p.n_rows - row0 < p.union_g ? p.n_rows - row0 : p.union_g);
        cols = rows_in_group * p.group;
      } else {
        row0 = group;
        rows_in_group = 1;
        cols = min(p.chunk_cols, p.group - chunk * p.chunk_cols);
      }
      // Q tile rows = query columns c (NP, zero beyond cols), 4 regions of 64 dims, SW128.
      // One shared buffer: the first kQPre rows are fetched into registers now and stored once
      // the previous item's last QK^T has read the buffer.
      auto q_src = [&](int c) -> const uint16_t* {
        int64_t row, head;
        if (UNION) {
          row = row0 + c / p.group;
          head = static_cast<int64_t>(kvh) * p.group + c % p.group;
        } else {
          row = row0;
          head = static_cast<int64_t>(kvh) * p.group + chunk * p.chunk_cols + c;
        }
        return p.q + (row * p.n_qheads + head) * kHeadDim + lane * 8;
      };
      constexpr int kQPre = kIdxSub0 ? 8 : (NP < 16 ? NP : 16);
      uint4 qv[kQPre];
#pragma unroll
      for (int c = 0; c < kQPre; ++c) qv[c] = c < cols ? ldg_nc_v4(q_src(c)) : make_uint4(0u, 0u, 0u, 0u);
      int32_t nv, nv_all, slot0 = 0;
      if (!UNION) {
        // Compact the row's valid slots (in order) into the slot list, as tensor-map rows.
        int32_t Lr = p.topk;
        if (p.topk_len) Lr = min(max(p.topk_len[row0], 0), p.topk);
        int32_t* const sl = reinterpret_cast<int32_t*>(gbase + L.slots) + b * slot_cap;
        const uint32_t sl_u32 = base + L.slots + b * slot_cap * 4;
        const int32_t n = compact_row_slots(p.indices + static_cast<int64_t>(row0) * p.topk, Lr, sl,
                                            sl_u32, p.n_kv_slots, p.n_kvheads, kvh, p.pad_row, p.pa,
                                            row0, lane);
        nv = n;
        nv_all = n;
        if (kCanSplit && split > 1) {
          // this CTA's contiguous range of the row's 128-slot tiles
          const int32_t nt_all = (n + kTileTokens - 1) / kTileTokens;
          const int32_t ta = static_cast<int32_t>(crank) * nt_all / split;
          const int32_t tb = (static_cast<int32_t>(crank) + 1) * nt_all / split;
          slot0 = ta * kTileTokens;
          nv = max(0, min(n, tb * kTileTokens) - slot0);
        }
      } else {
        nv = p.union_len[group];
        nv_all = nv;
      }
      // FP8 caches: the largest |V page scale| of the item's slots, for the softmax's per-item
      // normalisation; eight loads per lane in flight, one item ahead of the softmax.
      float vmax = 0.f;
      if (FP8) {
        const int32_t* sl_b = reinterpret_cast<const int32_t*>(gbase + L.slots) + b * slot_cap;
        const int32_t* ul_b =
            UNION ? p.union_idx + static_cast<int64_t>(group) * p.union_g * p.topk : nullptr;
        for (int t0 = 0; t0 < nv_all; t0 += 256) {
          float sc[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int t = t0 + 32 * u + lane;
            sc[u] = 0.f;
            if (t < nv_all) {
              const int64_t slot = UNION ? static_cast<int64_t>(ul_b[t])
                                         : div_by(sl_b[t], p.n_kvheads, p.kv_shift);
              sc[u] = fabsf(__ldg(p.v_scale + scale_index(p, slot, kvh)));
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) vmax = fmaxf(vmax, sc[u]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
      }
      if (lane == 0) {
        ItemInfo& I = info[b];
        I.n_valid = nv;
        I.group = group;
        I.kvh = kvh;
        I.chunk = chunk;
        I.cols = cols;
        I.row0 = row0;
        I.rows_in_group = rows_in_group;
        I.v_scale_max = vmax;
        I.slot0 = slot0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(b_itemfull + 8 * b);
      // Q: wait until the previous item's QK^T MMAs are done with the buffer.
      if (!__all_sync(0xffffffffu, wait_bar(b_qempty, (it & 1) ^ 1, abort_flag, kSiteQEmpty))) break;
      const uint32_t qb = base + L.qbuf;
      const int rg = lane >> 3, jc = lane & 7;
      auto q_store = [&](int c, uint4 v) {
        if (FP8) v = bf16x8_to_f16x8(v);   // FP8 caches run the f16 MMA: Q in f16
        sts_v4(qb + rg * (NP * 128) + (c >> 3) * 1024 + (c & 7) * 128 + ((jc ^ (c & 7)) << 4), v);
      };
#pragma unroll
      for (int c = 0; c < kQPre; ++c) q_store(c, qv[c]);
#pragma unroll
      for (int c = kQPre; c < NP; ++c) q_store(c, c < cols ? ldg_nc_v4(q_src(c)) : make_uint4(0u, 0u, 0u, 0u));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qfull);
    }
    finish_role();
    return;
  } else if (warp >= kGatherWarp0 || warp == 6 || warp == 7 || (kIdxSub0 && warp == kIndexWarp)) {
    // ------------------------------------------------------------ gather producers
    // Warpgroups 2-4 give registers back to the CTA's pool for the softmax warpgroup (warpgroup
    // register reallocation); warps 6 and 7 gather at warpgroup 1's count, and warps 8 and 12
    // stay idle so that the MMA warp's sub-partition keeps a single gather warp.
    if (warp >= kGatherWarp0) regs_dec<kGatherRegs>(); else regs_inc<kRoleRegs>();
    if (warp == 8 || warp == 12) {   // idle
      finish_role();
      return;
    }
    // Stage st is filled by warps 2 st and 2 st + 1, each gathering one 64-dim block of every
    // piece that lands on it (32 TMA gather4, one per lane, or 32 cp.async of four slots x 16
    // bytes per lane), in order.  Every piece's two halves are issued at once by two warps, and
    // no warp ever waits on a stage it does not fill.  (With one owner warp per stage a piece
    // took ~2.3 us to issue, and a V tile's pieces -- which reuse the stages of the same tile's
    // K, freed only when its QK^T completes -- were the wait of every P.V.)  FP8 pieces are
    // gathered and rewritten whole by the stage's first warp.
    const int pw = (kIdxSub0 && warp == kIndexWarp) ? kIdxWarp - kGatherWarp0 : gather_index(warp);
    const uint32_t st = static_cast<uint32_t>(pw / kBPS);   // this warp's stage
    const int blk = pw % kBPS;                              // and first 64-dim block
    const bool tma = p.gather_tma != 0;
    const bool active = static_cast<int>(st) < R;
    uint32_t seq = 0, it = 0, uses = 0;   // uses: fills of stage st so far
    int32_t last_issued = -1;             // the newest fill this warp issued copies for
    bool aborted = false;
    for (;; ++it) {
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, wait_bar(b_itemfull + 8 * b, ph, abort_flag, kSiteItemFull))) {
        aborted = true;
        break;
      }
      const ItemInfo I = info[b];
      if (I.n_valid < 0) break;                // no more items
      const int nv = I.n_valid;
      const int nt = (nv + kTileTokens - 1) / kTileTokens;
      const int32_t* sl = reinterpret_cast<const int32_t*>(gbase + L.slots) + b * slot_cap +
                          (kCanSplit ? I.slot0 : 0);
      const int32_t* ul =
          UNION ? p.union_idx + static_cast<int64_t>(I.group) * p.union_g * p.topk : nullptr;
      const int n_pieces = 4 * nt;
      // This warp's pieces are those on stage st: q = q_first + k R.
      const int sq = static_cast<int>(seq % static_cast<uint32_t>(R));
      const int q_first = active ? (static_cast<int>(st) - sq + R) % R : n_pieces;
      // tensor-map row of union slot t; a slot whose row would pass the map (or int32) becomes
      // padding, as in the per-token compaction
      auto union_row = [&](int t) -> int32_t {
        if (t >= nv) return p.pad_row;
        const int64_t y = static_cast<int64_t>(ul[t]) * p.n_kvheads + I.kvh;
        return y < static_cast<int64_t>(p.pad_row) ? static_cast<int32_t>(y) : p.pad_row;
      };
      // union slots of a piece's tile (global memory): lane holds tokens 4*lane .. 4*lane+3
      auto union_rows = [&](int q) {
        int tile, is_v, half;
        piece_of<kLookahead>(q, nt, tile, is_v, half);
        const int t = tile * kTileTokens + 4 * lane;
        return make_int4(union_row(t), union_row(t + 1), union_row(t + 2), union_row(t + 3));
      };
      // The union slots of the warp's next piece are loaded one piece ahead, so their latency
      // overlaps the wait for the current piece's stage and its issue.
      int4 uy_next = make_int4(0, 0, 0, 0);
      if (UNION && q_first < n_pieces) uy_next = union_rows(q_first);
      for (int q = q_first; q < n_pieces; q += R) {
        const int4 uy = uy_next;
        if (UNION && q + R < n_pieces) uy_next = union_rows(q + R);
        const uint32_t use = uses++;
        int tile, is_v, half;
        piece_of<kLookahead>(q, nt, tile, is_v, half);
        const int t0 = tile * kTileTokens;
        const uint32_t empty_bar = b_empty + 8 * (st >> 1);   // the stage pair's barrier
        if (!__all_sync(0xffffffffu, wait_bar(empty_bar, (use & 1) ^ 1, abort_flag, kSiteStageEmpty))) {
          aborted = true;
          break;
        }
        const uint32_t stage = base + L.ring + st * kStageBytes;
        int y0, y1, y2, y3;   // tensor-map rows of slots 4 lane .. 4 lane + 3 of the tile
        if (UNION) {
          y0 = uy.x; y1 = uy.y; y2 = uy.z; y3 = uy.w;
        } else {
          const int t = t0 + 4 * lane;
          const int4 v = *reinterpret_cast<const int4*>(sl + t);
          y0 = t + 0 < nv ? v.x : p.pad_row;
          y1 = t + 1 < nv ? v.y : p.pad_row;
          y2 = t + 2 < nv ? v.z : p.pad_row;
          y3 = t + 3 < nv ? v.w : p.pad_row;
        }
        const CUtensorMap* tm = is_v ? &tmV : &tmK;
        if (FP8) {
          // The piece's e4m3 rows (128 B: its 128 dims) land in the stage's upper 16 KiB, and
          // each of the stage's two warps gathers and rewrites 64 of the 128 slot rows: 16
          // gather4 (half the requests of a bf16 piece's block), then the rows in place as fp16.
          // A row's upper fp16 block overwrites only its own e4m3 bytes, so the rows, and the
          // two warps, are independent: dims 0-63 (lower block, no overlap) are written from the
          // first four input chunks before the last four are read.
          const uint32_t land = b_land + 8 * (kBPS * st + blk);
          const int g = 16 * blk + (lane & 15);          // this lane's 4-slot group of the tile
          int f0, f1, f2, f3;
          if (UNION) {
            f0 = __shfl_sync(0xffffffffu, y0, g);
            f1 = __shfl_sync(0xffffffffu, y1, g);
            f2 = __shfl_sync(0xffffffffu, y2, g);
            f3 = __shfl_sync(0xffffffffu, y3, g);
          } else {
            const int t = t0 + 4 * g;
            const int4 v = *reinterpret_cast<const int4*>(sl + t);
            f0 = t + 0 < nv ? v.x : p.pad_row;
            f1 = t + 1 < nv ? v.y : p.pad_row;
            f2 = t + 2 < nv ? v.z : p.pad_row;
            f3 = t + 3 < nv ? v.w : p.pad_row;
          }
          if (lane == 0) mbar_arrive_expect_tx(land, 64 * 128);
          __syncwarp();
          if (lane < 16) tma_gather4(stage + 16384 + g * 512, tm, half * 128, f0, f1, f2, f3, land);
          last_issued = static_cast<int32_t>(use);
          if (!__all_sync(0xffffffffu, wait_bar(land, use & 1, abort_flag, kSiteLanded))) {
            aborted = true;
            break;
          }
#pragma unroll 1
          for (int k = 0; k < 2; ++k) {
            const int t = 64 * blk + lane + 32 * k;
            const uint32_t sw = static_cast<uint32_t>(t & 7);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              uint4 in[4];
#pragma unroll
              for (int c = 0; c < 4; ++c)
                in[c] = lds_v4(stage + 16384 + t * 128 + (((4 * hb + c) ^ sw) << 4));
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                // dims 16(4 hb + c) .. +15 -> atom hb, 16-byte chunks 2c, 2c + 1
                const uint4 lo = make_uint4(e4m3x2_to_f16x2(in[c].x & 0xffffu), e4m3x2_to_f16x2(in[c].x >> 16),
                                            e4m3x2_to_f16x2(in[c].y & 0xffffu), e4m3x2_to_f16x2(in[c].y >> 16));
                const uint4 hi = make_uint4(e4m3x2_to_f16x2(in[c].z & 0xffffu), e4m3x2_to_f16x2(in[c].z >> 16),
                                            e4m3x2_to_f16x2(in[c].w & 0xffffu), e4m3x2_to_f16x2(in[c].w >> 16));
                const uint32_t row = stage + hb * 16384 + t * 128;
                sts_v4(row + (((2 * c) ^ sw) << 4), lo);
                sts_v4(row + (((2 * c + 1) ^ sw) << 4), hi);
              }
            }
          }
          fence_proxy_async_smem();   // generic writes -> tensor-core (async proxy) reads
          __syncwarp();
          if (lane == 0) mbar_arrive(b_full + 8 * st);
          continue;
        }
        if (tma) {
          // per lane and block: slots 4 lane .. 4 lane + 3, dims half * 128 + 64 c .. +63
          if (lane == 0) mbar_arrive_expect_tx(b_full + 8 * st, kStageBytes / kBPS);
          __syncwarp();
#pragma unroll
          for (int c = blk; c < kBlocksPerStage; c += kBPS)
            tma_gather4(stage + c * 16384 + lane * 512, tm, half * 128 + c * 64, y0, y1, y2, y3,
                        b_full + 8 * st);
        } else {
          // 16-byte copies: eight lanes per slot row of 128 bytes, four slots per instruction
          const int ch = lane & 7;
#pragma unroll 1
          for (int c = blk; c < kBlocksPerStage; c += kBPS) {
            const uint8_t* cache = (is_v ? p.v_bytes : p.k_bytes) + half * 256 + c * 128;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
              const int t = 4 * i + (lane >> 3);          // slot within the tile
              const int src_lane = t >> 2, el = t & 3;
              const int a0 = __shfl_sync(0xffffffffu, y0, src_lane), a1 = __shfl_sync(0xffffffffu, y1, src_lane);
              const int a2 = __shfl_sync(0xffffffffu, y2, src_lane), a3 = __shfl_sync(0xffffffffu, y3, src_lane);
              const int32_t y = el == 0 ? a0 : el == 1 ? a1 : el == 2 ? a2 : a3;
              const bool pad = y == p.pad_row;
              const uint8_t* src = cache + (pad ? 0 : static_cast<int64_t>(y) * (kHeadDim * 2)) + ch * 16;
              const uint32_t dst = stage + c * 16384 + t * 128 + ((ch ^ (t & 7)) << 4);
              cp_async_16_zfill(dst, src, pad ? 0u : 16u);
            }
          }
          // Each lane's arrival fires once all its earlier copies have landed; the MMA thread
          // orders them before its tensor-core reads with a proxy fence after the wait.
          cp_async_arrive_noinc(b_full + 8 * st);
        }
        last_issued = static_cast<int32_t>(use);
      }
      if (aborted) break;
      seq += 4 * nt;
      __syncwarp();
      if (lane == 0) mbar_arrive(b_itemempty + 8 * b);
    }
    if (!tma && !FP8) {
      cp_async_wait_0();
    } else if (aborted && lane == 0 && last_issued >= 0) {
      // Drain: wait (bounded) for this warp's newest copy into its stage to land.
      const uint32_t landed = FP8 ? b_land + 8 * (kBPS * st + blk) : b_full + 8 * st;
      drain_bar(landed, static_cast<uint32_t>(last_issued) & 1, kDrainLimitNs);
    }
    finish_role();
    return;
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    regs_inc<kRoleRegs>();
    constexpr uint32_t kIdescQK = FP8 ? idesc_f16_f32(128, NP, false, false)
                                      : idesc_bf16_f32(128, NP, false, false);
    constexpr uint32_t kIdescPV = FP8 ? idesc_f16_f32(128, NP, true, kPMnMajor)
                                      : idesc_bf16_f32(128, NP, true, kPMnMajor);
    uint32_t js = 0, it = 0;
    bool aborted = false;
    const bool cp_engine = !FP8 && p.gather_tma == 0;
    // The MMA consumes tile entries (a stage pair each) in exactly the ring's FIFO order, so a
    // running pointer (pair index, parity) replaces per-piece divisions by the stage count,
    // which sat on the issue path (measured: ~4 % of group6_32k, ~18 % with the gather removed).
    const uint32_t n_pairs = static_cast<uint32_t>(R) / 2;
    // Operand descriptors as a per-buffer low word plus a constant offset (one add per operand).
    constexpr uint32_t kHi = sw128_desc_hi(1024);
    const uint32_t q_lo = sw128_desc_lo(base + L.qbuf, 16);
    const uint32_t ring_k_lo = sw128_desc_lo(base + L.ring, 16);          // K-major stage reads
    const uint32_t ring_v_lo = sw128_desc_lo(base + L.ring, 16384);       // MN-major stage reads
    // P^T MN-major (N = 16: 32-byte rows, N = 32: 64-byte rows; one row per slot): 8-slot
    // groups kPSbo apart.  The leading offset is given the same value, so the operand stays
    // inside its 16 slots under either reading of the two fields.
    constexpr uint32_t kPSbo = 8 * NP * 2;
    constexpr uint32_t kPHi = !kPMnMajor ? kHi : NP == 16 ? sw32_desc_hi(kPSbo) : sw64_desc_hi(kPSbo);
    const uint32_t pbuf_lo = sw128_desc_lo(base + L.pbuf, kPMnMajor ? kPSbo : 16);
    uint32_t c_pair = 0, c_par = 0;
    auto advance = [&]() {
      if (++c_pair == n_pairs) {
        c_pair = 0;
        c_par ^= 1;
      }
    };
    for (;; ++it) {
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, wait_bar(b_itemfull + 8 * b, ph, abort_flag, kSiteItemFull))) {
        aborted = true;
        break;
      }
      const int nv = info[b].n_valid;
      if (nv < 0) break;                        // no more items
      const int nt = (nv + kTileTokens - 1) / kTileTokens;
      __syncwarp();
      if (lane == 0) mbar_arrive(b_itemempty + 8 * b);
      if (!__all_sync(0xffffffffu, wait_bar(b_qfull, it & 1, abort_flag, kSiteQFull))) {
        aborted = true;
        break;
      }
      for (int j = 0; j < nt + kLookahead; ++j) {
        if (j < nt) {
          // S^T(j) = K(j) . Q^T
          const uint32_t st_lo = 2 * c_pair, st_hi = st_lo + 1, e_pair = c_pair;
          const uint32_t jsj = js + j, sb = jsj % kSBufs, sph = (jsj / kSBufs) & 1;
          bool ok = wait_bar(b_full + 8 * st_lo, c_par, abort_flag, kSiteStageFull);
          ok = ok && wait_bar(b_full + 8 * st_hi, c_par, abort_flag, kSiteStageFull);
          ok = ok && wait_bar(b_sfree + 8 * sb, sph ^ 1, abort_flag, kSiteSFree);
          advance();
          if (!__all_sync(0xffffffffu, ok)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          // cp.async stage writes -> tensor-core (async proxy) reads; TMA writes are already in
          // the async proxy, and the FP8 rewrite fences on the writer side
          if (cp_engine) fence_proxy_async_smem();
          if (lane == 0) {
            const uint32_t k_lo = ring_k_lo + st_lo * (kStageBytes >> 4);   // stages st_lo, st_hi
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const int kq = kk & 7;
              const uint32_t a_off = (kk < 8 ? 0u : static_cast<uint32_t>(kStageBytes)) +
                                     (kq >> 2) * 16384 + (kq & 3) * 32;
              const uint32_t b_off = (kk >> 2) * (NP * 128) + (kk & 3) * 32;
              tc_mma_w(tm_s0 + sb * NP, k_lo + (a_off >> 4), kHi, q_lo + (b_off >> 4), kHi, kIdescQK,
                       kk > 0 ? 1u : 0u);
            }
            tc_commit(b_empty + 8 * e_pair);   // one commit frees the stage pair
            tc_commit(b_sfull + 8 * sb);
            if (j == nt - 1) tc_commit(b_qempty);
          }
          __syncwarp();
        }
        if (j >= kLookahead && j - kLookahead < nt) {
          // O^T += V(j-L)^T . P^T(j-L)
          const int jp = j - kLookahead;
          const uint32_t jsp = js + jp, pb = jsp & 1, pph = (jsp >> 1) & 1;
          const uint32_t st_vlo = 2 * c_pair, st_vhi = st_vlo + 1, e_pair = c_pair;
          bool ok = wait_bar(b_pfull + 8 * pb, pph, abort_flag, kSitePFull);
          ok = ok && wait_bar(b_full + 8 * st_vlo, c_par, abort_flag, kSiteStageFull);
          ok = ok && wait_bar(b_full + 8 * st_vhi, c_par, abort_flag, kSiteStageFull);
          advance();
          if (!__all_sync(0xffffffffu, ok)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          // cp.async stage writes -> tensor-core (async proxy) reads; TMA writes are already in
          // the async proxy, and the FP8 rewrite fences on the writer side
          if (cp_engine) fence_proxy_async_smem();
          if (lane == 0) {
            const uint32_t v_lo = ring_v_lo + st_vlo * (kStageBytes >> 4);   // stages st_vlo, st_vhi
            const uint32_t p_lo = pbuf_lo + pb * (static_cast<uint32_t>(L.p_bytes) >> 4);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a_off = hh * kStageBytes + kk * 2048;
                const uint32_t b_off = kPMnMajor ? kk * (16 * NP * 2)
                                                 : (kk >> 2) * (NP * 128) + (kk & 3) * 32;
                tc_mma_w(tm_o + hh * NP, v_lo + (a_off >> 4), kHi, p_lo + (b_off >> 4), kPHi, kIdescPV,
                         (jp == 0 && kk == 0) ? 0u : 1u);
              }
            }
            tc_commit(b_empty + 8 * e_pair);
            tc_commit(b_pvdone + 8 * pb);
          }
          __syncwarp();
        }
      }
      if (aborted) break;
      if (nt == 0 && lane == 0) tc_commit(b_qempty);
      __syncwarp();
      js += nt;
    }
    // Every MMA this thread issued has completed once `fin` flips.
    if (lane == 0) {
      tc_commit(b_fin);
      drain_bar(b_fin, 0, aborted ? kDrainLimitNs : kWaitLimitNs);
    }
    __syncwarp();
    finish_role();
    tc_fence_after();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    return;
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax + epilogue (warps 0-3)
    regs_inc<kSoftmaxRegs>();   // the registers warpgroups 2-4 returned
    const int t = threadIdx.x;                       // tensor-memory lane = slot within tile
    if constexpr (SC < NP) {
      // P columns SC .. NP-1 are never written: zero both P buffers once (the MMA reads them)
      for (int i = t; i < 2 * L.p_bytes / 16; i += 128) sts_v4(base + L.pbuf + 16 * i, make_uint4(0u, 0u, 0u, 0u));
      fence_proxy_async_smem();
    }
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t js = 0, it = 0, rb = 0;
    bool bad = false;
    const float NEG_INF = -INFINITY;
    for (;; ++it) {
      const uint32_t b = it & 1, ph = (it >> 1) & 1;
      bad |= !wait_bar(b_itemfull + 8 * b, ph, abort_flag, kSiteItemFull);
      // Uniform decision before the item record is read: if any softmax thread's wait gave up
      // (or another role aborted), all 128 leave together.
      if (named_bar_any(3, 128, bad || *abort_flag)) break;
      const ItemInfo I = info[b];
      if (I.n_valid < 0) break;                // no more items (same record for all 128)
      // FP8 reads the item's slot list for the scales until its last tile, so it hands the
      // item slot back at the end of the item instead.
      if (!FP8) mbar_arrive(b_itemempty + 8 * b);
      const int nv = I.n_valid;
      const int nt = (nv + kTileTokens - 1) / kTileTokens;
      const int cols = I.cols;
      const int32_t* slots_b = reinterpret_cast<const int32_t*>(gbase + L.slots) + b * slot_cap +
                               (kCanSplit ? I.slot0 : 0);
      const int32_t* ul_b =
          UNION ? p.union_idx + static_cast<int64_t>(I.group) * p.union_g * p.topk : nullptr;
      // Column masks: bit c of colmask[u] set when query column c belongs to row u of the group.
      uint64_t colmask[8];
      uint64_t allcols = (cols >= 64) ? ~0ull : ((1ull << cols) - 1ull);
      if (UNION) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int lo = u * p.group, hi = min((u + 1) * p.group, cols);
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
      // Columns past the item's real ones start (and stay) at a finite max of 0, so that a tile
      // whose slots are all valid can exponentiate every column without a -inf guard.
      float m_used[NP], l_part[NP];
#pragma unroll
      for (int c = 0; c < NP; ++c) {
        m_used[c] = c < cols ? NEG_INF : 0.f;
        l_part[c] = 0.f;
      }
      // FP8 caches: P is stored in fp16 as p * v_scale with p <= 2^8 (the lazy rescale
      // threshold), so a large V page scale could overflow fp16.  The item's V scales are
      // normalised by 2^-v_exp, v_exp the binary exponent of their largest magnitude (every
      // stored P then stays below 2^8), and the epilogue multiplies O back by 2^v_exp -- both
      // exact power-of-two scalings.
      int v_exp = 0;
      float v_norm = 1.f;
      if (FP8) {
        frexpf(I.v_scale_max, &v_exp);   // (computed by the index warp) < 2^v_exp
        v_exp = max(-126, min(v_exp, 126));
        v_norm = ldexpf(1.f, -v_exp);
      }
      uint32_t bits_next = 0;
      if (UNION && nt > 0) bits_next = t < nv ? ub[t] : 0u;
      bool quit = false;
      for (int j = 0; j < nt; ++j) {
        const uint32_t jsj = js + j, sb = jsj & 1, sph = (jsj >> 1) & 1;     // P buffer
        const uint32_t ss = jsj % kSBufs, ssph = (jsj / kSBufs) & 1;       // S^T buffer
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
        // FP8 caches: the slot's page scales -- K's multiplies the logit, V's the probability
        // fed to P.V (the row sum keeps the unscaled probability).
        float logit_scale = p.scale_log2, v_scale = 1.f;
        if (FP8 && valid) {
          const int64_t slot = UNION ? static_cast<int64_t>(ul_b[token])
                                     : div_by(slots_b[token], p.n_kvheads, p.kv_shift);
          const int64_t si = scale_index(p, slot, I.kvh);
          logit_scale *= __ldg(p.k_scale + si);
          v_scale = __ldg(p.v_scale + si) * v_norm;
        }
        bad |= !wait_bar(b_sfull + 8 * ss, ssph, abort_flag, kSiteSFull);
        tc_fence_after();
        float x[NP];
#pragma unroll
        for (int q = 0; q < NP / 16; ++q) tmem_ld16(tm_s0 + lane_off + ss * NP + 16 * q, x + 16 * q);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(b_sfree + 8 * ss);
        // A warp whose 32 slots are valid for every real column (all but a row's last tile and
        // the union tiles with unowned slots) skips the per-column masking, and its P loop the
        // -inf guard: its padding columns see S = 0 (Q's padding rows are zero), a finite max of 0
        // and P = 1, and feed only O^T columns the epilogue never reads.
        // (bf16 per-token instances only: in the union and FP8 instances the second copy of the
        // loops cost registers and measured slower.)
        constexpr bool kFastTiles = !UNION && !FP8;
        const bool full = kFastTiles && __all_sync(0xffffffffu, vmask == allcols);
        bool need = false;
        if (full) {
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            if (c >= SC) {   // no real column past SC: P stays zero there
              x[c] = NEG_INF;
              continue;
            }
            x[c] *= logit_scale;
            need |= x[c] > m_used[c] + kRescaleThreshold;
          }
        } else {
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            if (c >= SC) {
              x[c] = NEG_INF;
              continue;
            }
            x[c] = ((vmask >> c) & 1ull) ? x[c] * logit_scale : NEG_INF;
            need |= x[c] > m_used[c] + kRescaleThreshold;
          }
        }
        // One barrier per tile decides, uniformly for the 128 threads, whether the max moves
        // and whether some role gave up.
        const int myvote = (need ? 1 : 0) | ((bad || *abort_flag) ? 2 : 0);
        // vote[] is used round robin over the CTA's tile sequence: the word for tile jsj+2
        // is cleared here, after every thread has read it at tile jsj-1 and before any
        // thread can pass the next barrier and write it.
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
          if constexpr (NP == 16 || NP == 32) {
            float v[NP];
#pragma unroll
            for (int c = 0; c < NP; ++c) v[c] = x[c];
            const float m = warp_reduce_scatter<NP, true>(v, lane);
            if (NP == 32 || (lane & 1) == 0) rbuf[warp * NP + warp_column<NP>(lane)] = m;
          } else {
#pragma unroll
            for (int c = 0; c < NP; ++c) {
              float v = x[c];
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
              if (lane == 0) rbuf[warp * NP + c] = v;
            }
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
            bad |= !wait_bar(b_pvdone + 8 * (jprev & 1), (jprev >> 1) & 1, abort_flag, kSitePvDone);
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
              for (int q = 0; q < NP / 16; ++q) {
                float o[16];
                const uint32_t ta = tm_o + lane_off + hh * NP + 16 * q;
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
        bad |= !wait_bar(b_pvdone + 8 * sb, sph ^ 1, abort_flag, kSitePvDone);
        if (full) {   // every x and every max is finite here (see above)
#pragma unroll
          for (int c = 0; c < SC; ++c) x[c] = fast_exp2(x[c] - m_used[c]);
        } else {
#pragma unroll
          for (int c = 0; c < SC; ++c) x[c] = x[c] == NEG_INF ? 0.f : fast_exp2(x[c] - m_used[c]);
        }
#pragma unroll
        for (int c = 0; c < SC; ++c) l_part[c] += x[c];
        if constexpr (kPMnMajor) {
          // This thread's slot is one row of P^T: its columns in 16-byte chunks (eight columns
          // each; past SC zero), chunk i at position i ^ (address bits 7-8, or bit 7 for N = 16).
          const uint32_t prow = base + L.pbuf + sb * L.p_bytes + t * (NP * 2);
          const uint32_t sw = NP == 16 ? ((t >> 2) & 1) : ((t >> 1) & 3);
#pragma unroll
          for (int i = 0; i < (SC + 7) / 8; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int c = 8 * i + 2 * h;
              const float a = c < SC ? x[c] : 0.f, b = c + 1 < SC ? x[c + 1] : 0.f;
              w[h] = FP8 ? pack_f16x2(a * v_scale, b * v_scale) : pack_bf16x2(a, b);
            }
            sts_v4(prow + ((i ^ sw) << 4), make_uint4(w[0], w[1], w[2], w[3]));
          }
        } else {
          uint8_t* pbuf = gbase + L.pbuf + sb * L.p_bytes;
          uint8_t* prow = pbuf + (t >> 6) * (NP * 128) + ((t & 7) << 1);
          const int tchunk = (t & 63) >> 3;
#pragma unroll
          for (int c = 0; c < SC; ++c) {
            uint8_t* const dst = prow + (c >> 3) * 1024 + (c & 7) * 128 + ((tchunk ^ (c & 7)) << 4);
            if (FP8)
              *reinterpret_cast<__half*>(dst) = __float2half_rn(x[c] * v_scale);
            else
              *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(x[c]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(b_pfull + 8 * sb);
      }
      if (quit) break;
      // ---- epilogue: row sums, O / l, LSE
      float* rbuf = red + rb * 4 * NP;
      if constexpr (NP == 16 || NP == 32) {
        const float l = warp_reduce_scatter<NP, false>(l_part, lane);   // l_part is done with
        if (NP == 32 || (lane & 1) == 0) rbuf[warp * NP + warp_column<NP>(lane)] = l;
      } else {
#pragma unroll
        for (int c = 0; c < NP; ++c) {
          float v = l_part[c];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) rbuf[warp * NP + c] = v;
        }
      }
      named_bar_sync(1, 128);
      __nv_bfloat16* const outp = reinterpret_cast<__nv_bfloat16*>(p.out);
      const int64_t Hq = p.n_qheads;
      if (kCanSplit && split > 1) {
        // ---- split item: this CTA holds (m, l, O) over its own tile range.  The partials are
        // merged by dims: CTA s of the cluster finishes dims [s D, (s + 1) D), D = 256 / split, of
        // every column, from what every CTA (itself included) sends it through distributed shared
        // memory.  merge_o[src][dim - s D][column] and merge_ml[src][column] = (m, l) are this
        // CTA's receive buffers; b_sendok says every CTA has read the previous item's.
        const int D = kHeadDim / split;
        constexpr int RF = merge_row_floats(NP);
        bad |= !wait_cluster(b_sendok, (it & 1) ^ 1, abort_flag, kSiteMerge);
        if (t < cols) {
          const float l = (rbuf[t] + rbuf[NP + t]) + (rbuf[2 * NP + t] + rbuf[3 * NP + t]);
          float my_m = NEG_INF;
#pragma unroll
          for (int c = 0; c < NP; ++c)
            if (c == t) my_m = m_used[c];
          const uint32_t ml = base + L.merge_ml + (crank * NP + t) * 8;
          for (int s = 0; s < split; ++s) st_cluster_v2(cluster_map(ml, s), my_m, l);
        }
        named_bar_sync(1, 128);   // rbuf is read before the next item's reductions reuse it
        rb ^= 1;
        if (nt > 0) {
          const uint32_t jl = js + nt - 1;
          bad |= !wait_bar(b_pvdone + 8 * (jl & 1), (jl >> 1) & 1, abort_flag, kSitePvDone);
          tc_fence_after();
        }
        // this thread's dims are t (O^T half 0) and t + 128 (half 1)
#pragma unroll
        for (int q = 0; q < NP / 16; ++q) {
          if (16 * q >= cols) break;
          float o[2][16];
          if (nt > 0) {
            tmem_ld16(tm_o + lane_off + 16 * q, o[0]);
            tmem_ld16(tm_o + lane_off + NP + 16 * q, o[1]);
            tc_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[0][i] = o[1][i] = 0.f;
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int d = t + 128 * hh;
            const int s = d / D, dl = d - s * D;
            const uint32_t dst = cluster_map(
                base + L.merge_o + ((static_cast<int>(crank) * D + dl) * RF + 16 * q) * 4, s);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              st_cluster_v4(dst + 16 * k4, o[hh][4 * k4], o[hh][4 * k4 + 1], o[hh][4 * k4 + 2],
                            o[hh][4 * k4 + 3]);
          }
        }
        for (int s = 0; s < split; ++s) mbar_arrive_cluster(cluster_map(b_recv, s));
        bad |= !wait_cluster(b_recv, it & 1, abort_flag, kSiteMerge);
        const float* const mo = reinterpret_cast<const float*>(gbase + L.merge_o);
        const float2* const mml = reinterpret_cast<const float2*>(gbase + L.merge_ml);
        const int tpd = 128 / D;                 // threads per dim: split / 2
        const int dl = t % D, cg = t / D;
        for (int c = cg; c < cols; c += tpd) {
          float M = NEG_INF;
          for (int s = 0; s < split; ++s) M = fmaxf(M, mml[s * NP + c].x);
          float lsum = 0.f, acc = 0.f;
          if (M != NEG_INF) {
            for (int s = 0; s < split; ++s) {
              const float2 ml = mml[s * NP + c];
              const float w = ml.x == NEG_INF ? 0.f : fast_exp2(ml.x - M);
              lsum += w * ml.y;
              acc += w * mo[(s * D + dl) * RF + c];
            }
          }
          const float inv = lsum > 0.f ? (FP8 ? ldexpf(1.f / lsum, v_exp) : 1.f / lsum) : 0.f;
          const int64_t head = static_cast<int64_t>(I.kvh) * p.group + I.chunk * p.chunk_cols + c;
          const int64_t row = I.row0;
          outp[(row * Hq + head) * kHeadDim + static_cast<int>(crank) * D + dl] =
              __float2bfloat16_rn(acc * inv);
          if (crank == 0 && dl == 0 && p.lse != nullptr)
            p.lse[row * Hq + head] = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : NEG_INF;
        }
        // this thread is done with every CTA's partials in its receive buffers
        for (int s = 0; s < split; ++s) mbar_arrive_cluster(cluster_map(b_sendok, s));
      } else {
        // Thread t < cols finishes column t once: its row sum, 1 / l, LSE and output offset go to
        // the other reduction buffer (free: its last readers passed the barrier above), so the
        // store loop below reads them instead of every thread redoing NP divisions.
        float* const inv_s = red + (rb ^ 1) * 4 * NP;
        int64_t* const off_s = reinterpret_cast<int64_t*>(inv_s + NP);
        if (t < cols) {
          const float l = (rbuf[t] + rbuf[NP + t]) + (rbuf[2 * NP + t] + rbuf[3 * NP + t]);
          float my_m = NEG_INF;
#pragma unroll
          for (int c = 0; c < NP; ++c)
            if (c == t) my_m = m_used[c];
          int64_t row, head;
          if (UNION) {
            row = I.row0 + t / p.group;
            head = static_cast<int64_t>(I.kvh) * p.group + t % p.group;
          } else {
            row = I.row0;
            head = static_cast<int64_t>(I.kvh) * p.group + I.chunk * p.chunk_cols + t;
          }
          inv_s[t] = l > 0.f ? (FP8 ? ldexpf(1.f / l, v_exp) : 1.f / l) : 0.f;
          off_s[t] = (row * Hq + head) * kHeadDim;
          if (p.lse != nullptr) p.lse[row * Hq + head] = l > 0.f ? (my_m + log2f(l)) * kLn2 : NEG_INF;
        }
        named_bar_sync(1, 128);
        rb ^= 1;
        if (nt > 0) {
          const uint32_t jl = js + nt - 1;
          bad |= !wait_bar(b_pvdone + 8 * (jl & 1), (jl >> 1) & 1, abort_flag, kSitePvDone);
          tc_fence_after();
        }
        // 16 columns at a time, both 128-dim halves loaded before one wait
#pragma unroll
        for (int q = 0; q < NP / 16; ++q) {
          if (16 * q >= cols) break;
          float o[2][16];
          if (nt > 0) {
            tmem_ld16(tm_o + lane_off + 16 * q, o[0]);
            tmem_ld16(tm_o + lane_off + NP + 16 * q, o[1]);
            tc_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o[0][i] = o[1][i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 16 * q + i;
            if (c < cols) {
              const float il = inv_s[c];
              __nv_bfloat16* const dst = outp + off_s[c] + t;
              dst[0] = __float2bfloat16_rn(o[0][i] * il);
              dst[128] = __float2bfloat16_rn(o[1][i] * il);
            }
          }
        }
      }
      tc_fence_before();
      js += nt;
      if (FP8) mbar_arrive(b_itemempty + 8 * b);
    }
    finish_role();
    return;
  }
  // every warp of the CTA has returned from its role above
}

// ---------------------------------------------------------------------------- host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

// 2-D map over a KV cache viewed as [rows, row_elems] bf16 (rows = slots x kv_heads), box 64 x 1,
// 128-byte swizzle.
cudaError_t make_cache_map(CUtensorMap* m, const void* cache, int64_t rows, int row_elems) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_elems), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems) * 2};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// 2-D map over an e4m3 KV cache viewed as [rows, 256] bytes, box 128 x 1 (one 128-dim half row),
// 128-byte swizzle.
cudaError_t make_cache_map_e4m3(CUtensorMap* m, const void* cache, int64_t rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim)};
  const cuuint32_t box[2] = {128, 1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NP, bool UNION, bool FP8, int SC = NP>
cudaError_t launch_np(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                      const Geometry& g, cudaStream_t stream) {
  auto kern = sparse_prefill_kernel<NP, UNION, FP8, SC>;
  // The shared-memory opt-in is set once per device and size, so calls made while a stream
  // is being captured into a CUDA graph only enqueue the launch.
  static std::atomic<int> opted_in[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || opted_in[dev].load() < g.smem_bytes) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) opted_in[dev].store(g.smem_bytes);
  }
  if (g.split <= 1) {
    kern<<<g.grid, kThreads, g.smem_bytes, stream>>>(tk, tv, p);
    return cudaGetLastError();
  }
  // Split items: clusters of g.split CTAs (one per SM).  Fewer clusters may fit at once than the
  // SM count suggests (a cluster's CTAs share one GPC), so the grid is capped at the clusters that
  // can be resident together, looked up once per device and shape.
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(g.split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(g.smem_bytes);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static std::atomic<int> max_clusters[64][kMaxSplit + 1];
  int fit = dev >= 0 && dev < 64 ? max_clusters[dev][g.split].load() : 0;
  if (fit <= 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(g.grid));
    e = cudaOccupancyMaxActiveClusters(&fit, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (fit <= 0) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) max_clusters[dev][g.split].store(fit);
  }
  const int clusters = std::min(g.grid / g.split, fit);
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * g.split));
  e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const Geometry& g, const void* k_cache,
                           const void* v_cache, int64_t tmap_rows, cudaStream_t stream) {
  if (g.n_items == 0) return cudaSuccess;
  CUtensorMap tk, tv;
  const bool fp8 = p.k_scale != nullptr;
  cudaError_t e = fp8 ? make_cache_map_e4m3(&tk, k_cache, tmap_rows)
                      : make_cache_map(&tk, k_cache, tmap_rows, kHeadDim);
  if (e != cudaSuccess) return e;
  e = fp8 ? make_cache_map_e4m3(&tv, v_cache, tmap_rows)
          : make_cache_map(&tv, v_cache, tmap_rows, kHeadDim);
  if (e != cudaSuccess) return e;
  const bool u = p.union_g > 1;
  if (fp8) {
    switch (g.np) {
      case 16: return u ? launch_np<16, true, true>(tk, tv, p, g, stream)
                        : (g.cols <= 8 ? launch_np<16, false, true, 8>(tk, tv, p, g, stream)
                                       : launch_np<16, false, true>(tk, tv, p, g, stream));
      case 32: return u ? launch_np<32, true, true>(tk, tv, p, g, stream) : launch_np<32, false, true>(tk, tv, p, g, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (g.np) {
    case 16: return u ? launch_np<16, true, false>(tk, tv, p, g, stream)
                      : (g.cols <= 8    ? launch_np<16, false, false, 8>(tk, tv, p, g, stream)
                         : g.cols <= 12 ? launch_np<16, false, false, 12>(tk, tv, p, g, stream)
                                        : launch_np<16, false, false>(tk, tv, p, g, stream));
    case 32: return u ? launch_np<32, true, false>(tk, tv, p, g, stream) : launch_np<32, false, false>(tk, tv, p, g, stream);
    case 48: return u ? launch_np<48, true, false>(tk, tv, p, g, stream) : launch_np<48, false, false>(tk, tv, p, g, stream);
    case 64: return u ? launch_np<64, true, false>(tk, tv, p, g, stream) : launch_np<64, false, false>(tk, tv, p, g, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t device_status_address(int32_t** addr) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
  *addr = static_cast<int32_t*>(p);
  return e;
}

cudaError_t read_and_clear_device_status(cudaStream_t stream, int32_t* status) {
  int32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_device_status, sizeof(int32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(int32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace qsa
