// Declarations shared by the host API (api.cpp) and the CUDA translation units.
#pragma once

#include <cstddef>
#include <climits>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "qsa.h"   // include/ is on the compiler include path

namespace qsa {

constexpr int kHeadDim = 256;
constexpr int kTileTokens = 128;             // gathered slots per MMA tile (MMA M)
constexpr int kStageBytes = kTileTokens * 128 * 2;  // 128 slots x 128 dims bf16 = 32 KiB
constexpr int kMaxNPad = 64;                 // largest MMA N per tile
constexpr int kFp8MaxNPad = 32;              // largest MMA N per tile with FP8 caches
constexpr int kSoftmaxWarps = 4;             // warps 0-3: softmax + epilogue (TMEM lanes 0-127)
constexpr int kMmaWarp = 4;                  // MMA issue + tensor-memory owner
constexpr int kIndexWarp = 5;                // slot compaction, Q tile, item info
constexpr int kProducerWarp0 = 6;            // first gather warp
// d=256 kernel: each 32 KiB stage is filled by two gather warps, one per 64-dim block (a warp
// issues TMA gathers one after another at ~13 GB/s, so two warps land a stage in half the time).
// 20 warps = five warpgroups: softmax (0-3); MMA and index warps and two gather warps (4-7); ten
// gather warps and two idle ones (8-19), whose spare registers go to the softmax warpgroup
// (setmaxnreg).
constexpr int kBlocksPerStage = 2;
constexpr int kMaxStages = 6;
constexpr int kGatherWarp0 = 8;
constexpr int kProducerWarps = kBlocksPerStage * kMaxStages;
constexpr int kThreads = 640;
constexpr int kLaunchRegs = 96;              // 65536 / 640, rounded down to a multiple of 8
constexpr int kSoftmaxRegs = 176;            // after setmaxnreg.inc (warpgroup 0)
constexpr int kRoleRegs = 112;               // after setmaxnreg.inc (warpgroup 1: MMA, index)
constexpr int kGatherRegs = 64;              // after setmaxnreg.dec (warpgroups 2-4)
static_assert(kGatherWarp0 + kProducerWarps == kThreads / 32 && kGatherWarp0 % 4 == 0,
              "gather warps fill whole warpgroups at the end of the CTA");
static_assert(128 * kSoftmaxRegs + 128 * kRoleRegs + 384 * kGatherRegs <= kThreads * kLaunchRegs,
              "register split within the launch's registers");
// A warp's SM sub-partition (scheduler) is its index mod 4.  The MMA warp (4) issues measurably
// slower while gather warps share its sub-partition (their TMA request streams compete with its
// MMA issue), so in the d=256 kernel two of sub-partition 0's gather slots (warps 8 and 12) stay
// idle and warps 6 and 7 of warpgroup 1 gather in their place; sub-partition 0 keeps one gather
// warp (16).  Measured on GB300: group6_32k 1.639 -> 1.532 ms, union_8k G = 4 0.515 -> 0.502.
__host__ __device__ constexpr bool is_gather_warp(int warp) {
  return warp == 6 || warp == 7 || (warp >= kGatherWarp0 && warp != 8 && warp != 12);
}
// index of gather warp `warp` in 0 .. kProducerWarps - 1: stage index / kBlocksPerStage, block
// index % kBlocksPerStage (warps 6 and 7 take the idle slots' indices)
__host__ __device__ constexpr int gather_index(int warp) {
  return warp == 6 ? 8 - kGatherWarp0 : warp == 7 ? 12 - kGatherWarp0 : warp - kGatherWarp0;
}
// MLA kernel: the same 20-warp layout and register split; gather warps 8-17 share every latent
// piece and warps 18-19 every rope piece.
constexpr int kMlaLatentWarps = 10;
constexpr int kMlaRopeWarps = 2;
constexpr int kMlaProducerWarps = kMlaLatentWarps + kMlaRopeWarps;
constexpr int kMlaThreads = kThreads;
static_assert(kGatherWarp0 + kMlaProducerWarps == kMlaThreads / 32, "MLA gather warpgroups");
constexpr int kMinStages = 4;                // ring must hold V(j) and K(j+1) together
// MMA issue lookahead of the d=256 kernel: QK^T(j+L) is issued before P.V(j), with L + 1 S^T
// buffers.  Measured on GB300: per-token tiles (N = 16) run fastest at L = 1 (L = 2 or 3 cost
// 1 %); union tiles (N = 32, twice the softmax work per tile) gain 3 % at L = 2.
__host__ __device__ constexpr int lookahead_for(bool union_mode) { return union_mode ? 2 : 1; }
// The two stages of a piece pair (dims 0-127 and 128-255 of one K or V tile) are always
// consumed by the same MMA group, so one tcgen05.commit releases both through a shared empty
// barrier (each commit costs ~45 ns of issue; measured 0.5 % faster per-token).  The stage
// count is therefore even.
constexpr int kMaxSBufs = 3;
constexpr int kSmemLimit = 232448;           // 227 KiB opt-in dynamic shared memory
constexpr int kUnionMaxSmem = 200 * 1024;    // union-build kernel shared-memory cap

// In-kernel paged addressing: rows carry logical per-request positions, translated to physical
// cache slots through a page table.  page_table == nullptr = the indices are physical slots.
struct PagedAddr {
  const int32_t* page_table;    // [n_requests, pages_per_req] physical page ids (< 0 = none)
  const int32_t* cu_seqlens_q;  // [n_requests + 1] first row of each request, then n_rows
  const int32_t* kv_lens;       // [n_requests] logical KV length (nullable = pages_per_req pages)
  int32_t n_requests;
  int32_t pages_per_req;        // row stride of page_table
  int32_t page_size;
  int32_t page_shift;           // log2(page_size) when a power of two, else -1
  int64_t n_pages;              // physical pages in the cache (0 = unchecked)
};

// Everything the attention kernel needs besides the two tensor maps.
struct PrefillParams {
  const uint16_t* q;            // bf16 bits [n_rows, n_qheads, 256]
  const int32_t* indices;       // per-token mode
  const int32_t* topk_len;      // nullable
  uint16_t* out;
  float* lse;                   // nullable
  const int32_t* union_idx;     // union mode: [n_groups, union_g * topk]
  const uint8_t* union_bits;
  const int32_t* union_len;
  int64_t n_rows;
  int64_t n_items;
  int64_t n_kv_slots;           // 0 = unchecked
  int32_t n_qheads, n_kvheads, group;   // group = n_qheads / n_kvheads
  int32_t topk;
  int32_t union_g;              // 1 = per-token
  int32_t n_groups;             // row groups
  int32_t head_chunks, chunk_cols;
  int32_t stages;
  int32_t slot_cap;             // per-token slot-list capacity (multiple of 128)
  int32_t pad_row;              // tensor-map row used for padding gathers (out of bounds)
  int32_t tmem_cols;
  int32_t gather_tma;           // 1 = TMA tile::gather4, 0 = cp.async 16-byte row copies
  const uint8_t* k_bytes;       // caches as bytes, for the cp.async gather
  const uint8_t* v_bytes;
  float scale_log2;             // scale * log2(e)
  PagedAddr pa;                 // per-token mode: page_table != nullptr = logical indices
  // FP8 e4m3 caches: the value of a cache byte x at slot s, KV head h is
  // e4m3(x) * scale[(s / page_size) * n_kvheads + h]
  const float* k_scale;
  const float* v_scale;
  int32_t page_size;
  int32_t page_shift;           // log2(page_size) when a power of two, else -1
  int32_t kv_shift;             // log2(n_kvheads) when a power of two, else -1
  int32_t stall_first_item;     // failure-detection test: the index warp withholds its items
  // Per-token calls with fewer work items than SMs: the `split` CTAs of a thread-block cluster
  // share one item, each taking a contiguous range of its 128-slot tiles, and merge their
  // (max, row sum, O) partials through distributed shared memory.  1 = no split.
  int32_t split;
  // Union mode: items are handed out through this counter (zeroed by the union build) in
  // reverse order, longest groups first; nullptr = static round robin over the grid.
  int32_t* item_counter;
};

struct Geometry {
  int np;             // MMA N (padded query columns)
  int cols;           // real columns per item (max)
  int head_chunks;
  int chunk_cols;
  int union_g;        // effective
  int stages;
  int grid;
  int smem_bytes;
  int tmem_cols;
  int slot_cap;
  int64_t n_items;
  int n_groups;
  int split;          // CTAs sharing one item (a cluster); 1 = none
};

// Split items: at most eight CTAs per cluster (the portable cluster size), per-token tiles of
// at most 32 query columns.
constexpr int kMaxSplit = 8;
constexpr int kSplitMaxNPad = 32;
// Row stride (floats) of a split item's received O partials: NP columns + 4 of padding, so the
// merge's loads of one column by consecutive dims spread over the banks.
__host__ __device__ constexpr int merge_row_floats(int np) { return np + 4; }

// Shared-memory layout of the attention kernel (offsets from a 1024-aligned base).
struct SmemLayout {
  int ring, qbuf, pbuf, slots, bars, misc, merge_o, merge_ml, total;
  int q_bytes, p_bytes;
};
__host__ __device__ inline SmemLayout smem_layout(int np, int stages, int slot_cap, bool fp8,
                                                  int split = 1) {
  SmemLayout L;
  L.q_bytes = np * 512;
  L.p_bytes = np * 256;
  L.ring = 0;
  L.qbuf = stages * kStageBytes;
  L.pbuf = L.qbuf + L.q_bytes;          // one Q tile buffer
  L.slots = L.pbuf + 2 * L.p_bytes;
  L.bars = L.slots + 2 * slot_cap * 4;
  // full[st], empty[st], s_full[kMaxSBufs], s_free[kMaxSBufs], p_full[2], pv_done[2],
  // item_full[2], item_empty[2], q_empty, q_full, final, merge_recv, merge_sendok,
  // landed[st][block] (FP8 caches only)
  L.misc = L.bars + ((fp8 ? 2 + kBlocksPerStage : 2) * stages + 2 * kMaxSBufs + 13) * 8;
  // info[2][12] int32, red[2][4][np] float, tmem base, abort flag, vote[3]
  int misc_bytes = 2 * 12 * 4 + 2 * 4 * np * 4 + 32;
  L.merge_o = (L.misc + misc_bytes + 15) & ~15;
  // split items: O partials [split][256 / split dims][merge_row_floats(np)] and the (max, row
  // sum) pairs [split][np] of every CTA of the cluster
  const int merge_bytes = split > 1 ? 256 * merge_row_floats(np) * 4 : 0;
  L.merge_ml = L.merge_o + merge_bytes;
  const int ml_bytes = split > 1 ? split * np * 8 : 0;
  L.total = L.merge_ml + ml_bytes + 1024;   // + alignment slack for the 1024-aligned base
  return L;
}

// ---------------------------------------------------------------------------- MLA shape
// One latent KV row per slot: d_qk = 512 latent + 64 rope dims, V = the latent dims of the same
// row, one KV head shared by every query head.
constexpr int kMlaDqk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaPairs = kMlaDv / 128;            // 32 KiB latent pieces per tile (128 dims)
constexpr int kMlaRopeBytes = kTileTokens * 128;  // 128 slots x 64 rope dims bf16 = 16 KiB
constexpr int kMlaMaxNPad = 32;

struct MlaParams {
  const uint16_t* q;            // bf16 bits [n_rows, n_heads, 576]
  const int32_t* indices;       // per-token mode
  const int32_t* topk_len;      // nullable
  uint16_t* out;                // bf16 bits [n_rows, n_heads, 512]
  float* lse;                   // nullable
  const int32_t* union_idx;     // union mode: [n_groups, union_g * topk]
  const uint8_t* union_bits;
  const int32_t* union_len;
  int32_t* status;              // device status word (0x100 | wait site on a timeout)
  int64_t n_rows;
  int64_t n_items;
  int64_t n_kv_slots;           // 0 = unchecked
  int32_t n_heads;
  int32_t topk;
  int32_t union_g;
  int32_t n_groups;
  int32_t head_chunks, chunk_cols;
  int32_t pair_stages;          // latent ring depth (4 or 5)
  int32_t slot_cap;
  int32_t pad_row;
  int32_t tmem_cols;
  float scale_log2;
  PagedAddr pa;                 // page_table == nullptr = physical slots
  int32_t stall_first_item;     // failure-detection test: the index warp withholds its items
  // Per-token calls with fewer work items than SMs: the `split` CTAs of a thread-block cluster
  // share one item, each taking a contiguous range of its 128-slot tiles, and merge their
  // (max, row sum, O) partials through distributed shared memory.  1 = no split.
  int32_t split;
  int32_t* item_counter;        // union mode: longest-first item counter (as PrefillParams)
};

struct MlaSmemLayout {
  int pairs, rope, qbuf, pbuf, slots, bars, misc, total;
  int q_bytes, p_bytes;
};
__host__ __device__ inline MlaSmemLayout mla_smem_layout(int np, int pair_stages, int slot_cap) {
  MlaSmemLayout L;
  L.q_bytes = np * kMlaDqk * 2;
  L.p_bytes = np * 256;
  L.pairs = 0;
  L.rope = pair_stages * kStageBytes;
  L.qbuf = L.rope + kMlaRopeBytes;
  L.pbuf = L.qbuf + L.q_bytes;
  L.slots = L.pbuf + 2 * L.p_bytes;
  L.bars = L.slots + 2 * slot_cap * 4;
  // pair full/empty[stages], rope full/empty, s_full[2], s_free[2], p_full[2], pv_done[2],
  // item_full[2], item_empty[2], q_empty, q_full, final
  L.misc = L.bars + (2 * pair_stages + 2 + 15) * 8;
  const int misc_bytes = 2 * 8 * 4 + 2 * 4 * np * 4 + 32;
  L.total = L.misc + misc_bytes + 1024;
  return L;
}

struct MlaGeometry {
  int np, cols, head_chunks, chunk_cols, union_g, pair_stages, grid, smem_bytes, tmem_cols;
  int slot_cap, n_groups;
  int64_t n_items;
};

cudaError_t launch_mla(const MlaParams& p, const MlaGeometry& g, const void* kv_cache,
                       int64_t tmap_rows, cudaStream_t stream);
// ---------------------------------------------------------------------------- page split
constexpr int kMaxPageSections = 8;
struct PageSections {          // per-token byte widths of a page's sections, in page order
  int32_t n;
  int32_t bytes[kMaxPageSections];
  int64_t token_bytes;         // sum of bytes[]
};
cudaError_t launch_page_mark(const int32_t* indices, int64_t n_indices, int32_t src_page_size,
                             int64_t n_src_pages, uint8_t* mark, int num_sms, cudaStream_t stream);
cudaError_t launch_page_split(const void* src, void* dst, const uint8_t* mark, int64_t n_src_pages,
                              int32_t src_page_size, int32_t dst_page_size,
                              const PageSections& sec, cudaStream_t stream);

// Device address of the attention kernels' status word (prefill.cu), for kernels in other units.
cudaError_t device_status_address(int32_t** addr);

// Host launchers (prefill.cu / union.cu).  Return cudaSuccess or the launch error.
// TMA map over a KV cache viewed as [rows, row_elems] bf16 (row = slot x kv_heads + kv_head),
// box 64 x 1 with 128-byte swizzle: the gather4 source of the attention kernels and the probe.
cudaError_t make_cache_map(CUtensorMap* m, const void* cache, int64_t rows, int row_elems);
cudaError_t launch_prefill(const PrefillParams& p, const Geometry& g, const void* k_cache,
                           const void* v_cache, int64_t tmap_rows, cudaStream_t stream);
cudaError_t launch_union_build(const int32_t* indices, const int32_t* topk_len, int64_t n_rows,
                               int32_t topk, int32_t union_g, int64_t n_kv_slots,
                               int32_t* sorted_out, int32_t* union_idx, uint8_t* union_bits,
                               int32_t* union_len, bool pad_outputs, const PagedAddr* paged,
                               cudaStream_t stream, int32_t* item_counter = nullptr);
size_t union_build_smem_bytes(int32_t topk, int32_t union_g);   // hot-path (bitmap) kernel
size_t union_sort_smem_bytes(int32_t topk, int32_t union_g);    // sorted-rows (bitonic) kernel
cudaError_t read_and_clear_device_status(cudaStream_t stream, int32_t* status);

}  // namespace qsa
