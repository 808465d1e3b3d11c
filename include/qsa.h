/*
 * qsa.h -- C ABI of the top-k sparse attention prefill library (libqsa.so), GB300 / sm_103a.
 *
 * The operation ("[QSA] Tune sm120 sparse prefill geometry", Motivation; "DSA prefill ...
 * triton_sparse_mla", Motivation and Modifications): an indexer has chosen, for every query
 * row, up to `topk` KV token slots (int32, negative = padding).  For each row, the query
 * heads that share one KV head attend only over the K/V rows gathered at those slots --
 * scaled dot product, numerically stable softmax -- and the library writes O and the
 * per-head natural-log log-sum-exp of the scaled logits.  Optionally G adjacent rows share
 * one gathered union of their slots, with a per-slot ownership bitmask that keeps every
 * row's own softmax support (same page, Modifications: union mode).
 *
 * Conventions for every entry point:
 *  - Layouts are contiguous, row-major:
 *      q        [n_rows, n_qheads, head_dim]   bf16
 *      k_cache  [n_slots, n_kvheads, head_dim] bf16   (physical slots)
 *      v_cache  [n_slots, n_kvheads, head_dim] bf16
 *      indices  [n_rows, topk]                 int32  physical slots; < 0 = padding
 *      topk_len [n_rows]                       int32  leading slots considered (clamped to
 *                                                     [0, topk]); NULL = all topk
 *      out      [n_rows, n_qheads, head_dim]   bf16   (the [tokens, heads, d_v] contract)
 *      lse      [n_rows, n_qheads]             fp32   NULL = not written
 *    One index row serves every KV head; query head h reads KV head h / (n_qheads/n_kvheads).
 *  - Every pointer argument except the ones marked host-side is a DEVICE pointer of the
 *    current CUDA device.  The caller owns all memory; the library never frees or keeps a
 *    pointer past the call.  q, k_cache, v_cache and out must be 16-byte aligned.
 *  - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *    stream).  Calls return before the GPU finishes and make no host synchronisation.
 *  - No exception crosses the ABI.  Argument errors are detected on the host before any
 *    GPU work and return a status; nothing is enqueued then.
 *  - A row with no valid slot gets O = 0 and LSE = -inf.  A slot listed twice in one row is
 *    weighted twice (per-token path).
 *  - Results are deterministic: no atomics take part in any reduction.
 *  - Environment: QSA_LOG=1 prints one stderr line per attention call with the selected launch
 *    geometry; QSA_GATHER=cpasync selects cp.async copies instead of TMA gather4 for the bf16
 *    d=256 kernel (same results, bit for bit).
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qsa_status {
  QSA_OK = 0,
  QSA_ERR_INVALID_ARG = 1,   /* null required pointer, bad size, misaligned pointer */
  QSA_ERR_UNSUPPORTED = 2,   /* head_dim != 256, device is not sm_103, shape beyond limits */
  QSA_ERR_WORKSPACE = 3,     /* caller workspace smaller than qsa_union_workspace_bytes() */
  QSA_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  QSA_ERR_TIMEOUT = 5        /* a kernel wait ran past its limit (see qsa_get_device_status) */
} qsa_status;

/* Launch geometry chosen by the selector ("[QSA] Tune sm120 sparse prefill geometry",
 * Modifications: a measured launch table per group size, top-k and head dimension). */
typedef struct qsa_geometry {
  int32_t tile_tokens;      /* gathered slots per MMA tile (128) */
  int32_t stages;           /* shared-memory pipeline stages, each 128 slots x 128 dims bf16 */
  int32_t n_pad;            /* MMA N: query columns of a tile, padded to a multiple of 16 */
  int32_t cols;             /* real query columns of a tile (heads x rows of the group) */
  int32_t head_chunks;      /* tiles of query heads per KV head (1 unless the group > 64) */
  int32_t union_g;          /* effective union group size (1 = per-token) */
  int32_t grid;             /* CTAs launched (persistent, <= SM count) */
  int32_t threads;          /* threads per CTA */
  int32_t smem_bytes;       /* dynamic shared memory per CTA */
  int32_t tmem_cols;        /* tensor-memory columns allocated per CTA */
  int64_t n_items;          /* work items: row groups x KV heads x head chunks */
  int32_t split;            /* CTAs (one thread-block cluster) sharing each work item: 1, 2, 4 or 8.
                               Per-token bf16 calls (tiles of <= 32 columns) with fewer items
                               than SMs split each row's 128-slot tiles over a cluster and
                               merge the partial softmax statistics and outputs through
                               distributed shared memory ("[QSA] Tune sm120 sparse prefill
                               geometry", Query-count sweep: small row counts).  A row's result
                               is then summed in another order than with split 1 (within the
                               stated tolerance, deterministic per geometry). */
} qsa_geometry;

/* Per-path call counters (host side, process wide), in the spirit of the pages' invocation
 * counts ("DSA prefill ... triton_sparse_mla", Speed Tests: every run counts invocations of
 * the kernel, so that a path which quietly did nothing could not look like a speed-up). */
typedef struct qsa_counters {
  uint64_t calls_per_token;    /* calls served by the per-token path */
  uint64_t calls_union;        /* calls served by the union path */
  uint64_t union_fallbacks;    /* union requested but illegal for the shape -> per-token */
  uint64_t step_downs;         /* forced geometry stepped down to fit shared memory */
  uint64_t kernel_launches;    /* kernels enqueued by this library */
} qsa_counters;

/* Main entry: sparse prefill attention for all rows.
 *   union_g: 0 or 1 = per-token path; 2..8 = union of union_g consecutive rows with ownership
 *            bits.  A union shape the kernel cannot tile (union_g * group > 64) runs the
 *            per-token path instead and counts a fallback; the result is the same.  Union mode
 *            requires each row's valid slots to be distinct (a repeated slot is used once).
 *   Slots must be < n_slots of the caches (not checked: the signature carries no slot
 *   count; use qsa_sparse_prefill_ex with n_kv_slots to have them treated as padding).
 *   Union mode allocates its workspace on `stream` (cudaMallocFromPoolAsync / cudaFreeAsync) from
 *   a stream-ordered memory pool the library creates per device, whose release threshold is
 *   unbounded: freed workspaces stay in that pool for later calls (until the process exits), so
 *   steady-state calls make no driver allocation. */
qsa_status qsa_sparse_prefill(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* indices, const int32_t* topk_len,
                              void* out, float* lse,
                              int64_t n_rows, int32_t n_qheads, int32_t n_kvheads,
                              int32_t head_dim, int32_t topk, float scale,
                              int32_t union_g, void* stream);

/* Extended entry.
 *   n_kv_slots: 0 = unchecked; > 0 = slots >= n_kv_slots are padding (and gathers are
 *               bounds-checked against it).
 *   workspace / workspace_bytes: caller scratch for union mode (NULL = allocate on stream);
 *               must hold qsa_union_workspace_bytes(n_rows, topk, effective union_g) bytes and be
 *               256-byte aligned.  Unused by the per-token path.
 *   forced:     host pointer, NULL = selector; fields > 0 override stages, grid and split (an
 *               oversized stage count is stepped down to fit and counted; split is rounded down
 *               to a power of two <= 8 and applies to per-token bf16 tiles of <= 32 columns
 *               only). */
qsa_status qsa_sparse_prefill_ex(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* indices, const int32_t* topk_len,
                                 void* out, float* lse,
                                 int64_t n_rows, int32_t n_qheads, int32_t n_kvheads,
                                 int32_t head_dim, int32_t topk, float scale,
                                 int32_t union_g, int64_t n_kv_slots,
                                 void* workspace, size_t workspace_bytes,
                                 const qsa_geometry* forced, void* stream);

/* Paged entry: the indexer's slots are LOGICAL positions inside each row's request, and the
 * library translates them through the request's page table in the kernels (no translated index
 * tensor is written).  The pages route a batch's top-k indices through a PAGED or a RAGGED
 * transform chosen per batch kind, key the valid length on the cache sequence lengths, and serve
 * with paged KV caches of 64 or 128 slots per page ("DSA prefill ... triton_sparse_mla",
 * Modifications: Robustness, and the review follow-up on MIXED batches; "[QSA] Tune sm120 sparse
 * prefill geometry", serving command --page-size 128).
 *   k_cache, v_cache [n_pages * page_size, n_kvheads, head_dim] bf16: physical page p holds slots
 *               p*page_size .. p*page_size + page_size - 1 (the layout of qsa_sparse_prefill).
 *   indices     [n_rows, topk] int32 logical positions in the row's request, < 0 = padding.
 *   cu_seqlens_q [n_requests + 1] int32: rows of request i are cu_seqlens_q[i] .. [i+1] - 1;
 *               non-decreasing, [0] = 0, [n_requests] = n_rows (not checked: the device data is
 *               not read on the host).
 *   kv_lens     [n_requests] int32 logical KV length of each request, nullable; a position at or
 *               past it is padding.
 *   page_table  [n_requests, pages_per_req] int32 physical page of each logical page, < 0 = none.
 *   n_pages     physical pages in the caches; > 0 = pages >= n_pages are padding (gathers are
 *               bounds-checked), 0 = unchecked.
 * Position x of request i reads physical slot page_table[i][x / page_size] * page_size +
 * x % page_size.  It is padding when x < 0, x >= kv_lens[i], x / page_size >= pages_per_req, or
 * the page is < 0 or >= n_pages.  Everything else (topk_len, union_g, lse, errors, streams)
 * is as for qsa_sparse_prefill; with union_g > 1 the groups are union_g consecutive rows and
 * may span requests (the union is built over physical slots).
 * Errors: QSA_ERR_INVALID_ARG for a null cu_seqlens_q or page_table, n_requests < 1,
 * pages_per_req < 1, page_size < 1 or n_pages < 0; QSA_ERR_UNSUPPORTED when
 * n_pages * page_size * n_kvheads >= 2^31. */
qsa_status qsa_sparse_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* indices, const int32_t* topk_len,
                                    const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                    const int32_t* page_table, void* out, float* lse,
                                    int64_t n_rows, int32_t n_requests, int32_t pages_per_req,
                                    int32_t page_size, int64_t n_pages, int32_t n_qheads,
                                    int32_t n_kvheads, int32_t head_dim, int32_t topk, float scale,
                                    int32_t union_g, void* stream);

/* FP8 KV cache: K and V stored as e4m3 bytes with a fp32 scale per page and KV head, dequantised
 * in the gather ("DSA prefill ... triton_sparse_mla", Robustness and Accuracy Tests: the Triton
 * kernel refuses a packed FP8 pool and takes dequantised rows; flashinfer reads the FP8 cache
 * together with its scales).  The value of cache byte x at slot s, KV head h is
 *   e4m3(x) * k_scale[(s / page_size) * n_kvheads + h]      (v_scale likewise)
 * and the result is that of qsa_sparse_prefill on the dequantised caches.
 *   k_cache, v_cache [n_slots, n_kvheads, head_dim] e4m3 bytes (16-byte aligned)
 *   k_scale, v_scale [ceil(n_slots / page_size), n_kvheads] fp32 (device)
 * Other arguments as qsa_sparse_prefill, plus n_kv_slots as in qsa_sparse_prefill_ex.  The
 * tensor cores run fp16 operands here: q is rounded to fp16 (|q| must stay below 65504), the
 * e4m3 values convert to fp16 exactly, and each slot's V scale multiplies its probability.
 * Query columns per tile are capped at 32: larger head groups run in head chunks, and unions
 * wider than 32 columns run as per-token calls instead (counted). */
qsa_status qsa_sparse_prefill_fp8(const void* q, const void* k_cache, const void* v_cache,
                                  const float* k_scale, const float* v_scale, int32_t page_size,
                                  const int32_t* indices, const int32_t* topk_len, void* out,
                                  float* lse, int64_t n_rows, int32_t n_qheads, int32_t n_kvheads,
                                  int32_t head_dim, int32_t topk, float scale, int32_t union_g,
                                  int64_t n_kv_slots, void* stream);

/* FP8 caches over a paged pool: qsa_sparse_prefill_fp8's e4m3 caches and scales with
 * qsa_sparse_prefill_paged's logical indices, translated in the kernels ("DSA prefill ...
 * triton_sparse_mla", Robustness and Accuracy Tests: the served FP8 KV pool is paged).  The
 * scale of a physical slot s is k_scale[(s / fp8_page_size) * n_kvheads + h] (v_scale likewise),
 * fp8_page_size being the scale granularity and page_size the paging of the pool; everything
 * else as qsa_sparse_prefill_paged and qsa_sparse_prefill_fp8. */
qsa_status qsa_sparse_prefill_fp8_paged(const void* q, const void* k_cache, const void* v_cache,
                                        const float* k_scale, const float* v_scale,
                                        int32_t fp8_page_size, const int32_t* indices,
                                        const int32_t* topk_len, const int32_t* cu_seqlens_q,
                                        const int32_t* kv_lens, const int32_t* page_table,
                                        void* out, float* lse, int64_t n_rows, int32_t n_requests,
                                        int32_t pages_per_req, int32_t page_size, int64_t n_pages,
                                        int32_t n_qheads, int32_t n_kvheads, int32_t head_dim,
                                        int32_t topk, float scale, int32_t union_g, void* stream);

/* MLA-shaped sparse prefill ("DSA prefill ... triton_sparse_mla", Motivation and Speed Tests:
 * one latent KV row per token, kv_lora_rank 512 + qk_rope_head_dim 64 = 576 dims for QK^T, the
 * 512 latent dims as V, topk 2048, 8 heads at TP8, union G = 2 / 4).  Every query head attends
 * over its row's selected slots of the single latent KV head.
 *   q        [n_rows, n_heads, d_qk]  bf16
 *   kv_cache [n_slots, d_qk]          bf16; K = the whole row, V = its first d_v dims
 *   indices  [n_rows, topk] int32 physical slots (< 0 = padding); topk_len as above
 *   out      [n_rows, n_heads, d_v]   bf16;  lse [n_rows, n_heads] fp32 (nullable)
 *   d_qk must be 576 and d_v 512 (QSA_ERR_UNSUPPORTED otherwise).  union_g as in
 *   qsa_sparse_prefill; a union needs union_g * n_heads <= 32, otherwise the per-token path
 *   runs and counts a fallback.  n_kv_slots: 0 = unchecked, > 0 = slots >= n_kv_slots are
 *   padding.  q, kv_cache and out must be 16-byte aligned.  Union workspace is allocated on
 *   `stream` from the library's pool (as for qsa_sparse_prefill).  Errors, streams and
 *   determinism are as for qsa_sparse_prefill. */
qsa_status qsa_sparse_mla_prefill(const void* q, const void* kv_cache, const int32_t* indices,
                                  const int32_t* topk_len, void* out, float* lse, int64_t n_rows,
                                  int32_t n_heads, int32_t d_qk, int32_t d_v, int32_t topk,
                                  float scale, int32_t union_g, int64_t n_kv_slots, void* stream);

/* MLA shape over a paged latent cache: indices are logical positions of each row's request,
 * translated through page_table in the kernels exactly as in qsa_sparse_prefill_paged
 * (kv_cache [n_pages * page_size, d_qk]); everything else as qsa_sparse_mla_prefill. */
qsa_status qsa_sparse_mla_prefill_paged(const void* q, const void* kv_cache, const int32_t* indices,
                                        const int32_t* topk_len, const int32_t* cu_seqlens_q,
                                        const int32_t* kv_lens, const int32_t* page_table,
                                        void* out, float* lse, int64_t n_rows, int32_t n_requests,
                                        int32_t pages_per_req, int32_t page_size, int64_t n_pages,
                                        int32_t n_heads, int32_t d_qk, int32_t d_v, int32_t topk,
                                        float scale, int32_t union_g, void* stream);

/* Host-only geometry selection for qsa_sparse_mla_prefill (stages = latent ring depth). */
qsa_status qsa_select_mla_geometry(int32_t n_heads, int32_t union_g, int32_t topk, int32_t d_qk,
                                   int32_t d_v, int64_t n_rows, int32_t num_sms,
                                   qsa_geometry* out);

/* Touched-page mark and masked page split ("[SM120] Only split touched SWA pages in FlashMLA
 * page-split kernel", Modifications): re-lay a KV pool from src_page_size-token pages to
 * dst_page_size-token pages, copying only the pages that a step's sparse indices reference.
 * Page layout (both pools): a page of P tokens holds n_sections sections one after another,
 * section k being P x section_bytes[k] bytes, token-major.  Destination page p * ratio + i
 * (ratio = src_page_size / dst_page_size) holds tokens i * dst_page_size ..
 * (i + 1) * dst_page_size - 1 of source page p, section by section.
 *   qsa_page_mark: mark [n_src_pages] uint8 (device, caller-owned) is zeroed, then
 *     mark[t / src_page_size] = 1 for every index t >= 0 of indices [n_indices] (int32 token
 *     slots of the source pool; slots past the pool are ignored).  No atomics, no host read.
 *   qsa_page_split: copies every destination page whose source page is marked (mark NULL =
 *     every page).  Destination pages of unmarked source pages are left untouched.  The launch
 *     grid is one CTA per source page whatever the mark holds, so a captured CUDA graph replays
 *     it; an unmarked page costs one byte load.
 *   qsa_split_touched_pages: mark + masked split in one call.
 * Requirements: src_pool and dst_pool 16-byte aligned (host pointer section_bytes, each entry a
 * positive multiple of 16, 1 <= n_sections <= 8), src_page_size a multiple of dst_page_size,
 * n_src_pages * ratio < 2^31.  Errors: QSA_ERR_INVALID_ARG / QSA_ERR_UNSUPPORTED before any
 * GPU work. */
qsa_status qsa_page_mark(const int32_t* indices, int64_t n_indices, int32_t src_page_size,
                         int64_t n_src_pages, uint8_t* mark, void* stream);
qsa_status qsa_page_split(const void* src_pool, void* dst_pool, const uint8_t* mark,
                          int64_t n_src_pages, int32_t src_page_size, int32_t dst_page_size,
                          int32_t n_sections, const int32_t* section_bytes, void* stream);
qsa_status qsa_split_touched_pages(const int32_t* indices, int64_t n_indices, const void* src_pool,
                                   void* dst_pool, uint8_t* mark, int64_t n_src_pages,
                                   int32_t src_page_size, int32_t dst_page_size,
                                   int32_t n_sections, const int32_t* section_bytes,
                                   void* stream);

/* Allocation-free variant of qsa_sparse_prefill (same arguments, same results).  The pages
 * have no counterpart: it exists for callers that must not allocate device memory -- code
 * whose GPU memory is owned entirely by a framework's pool, latency-critical loops where an
 * allocator call (and the device synchronisation it may cause) is unacceptable, and plugin
 * hosts that give kernels no allocator.  Union-mode scratch lives in a fixed array of
 * QSA_NOALLOC_SCRATCH_BYTES in device global memory that the library owns; every GPU on which
 * the library is loaded holds that array until the process exits.
 *   - A call whose union workspace (qsa_union_workspace_bytes) exceeds QSA_NOALLOC_SCRATCH_BYTES is
 *     rejected with QSA_ERR_WORKSPACE before anything is enqueued.  The per-token path needs
 *     no scratch and has no such limit.
 *   - The first union call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first union call before any
 *     stream capture.  Per-token calls never touch the array.
 *   - Every call uses the same array, which keeps the previous call's contents; nothing in it
 *     needs to start at zero (each call writes every entry it later reads).  Calls whose work
 *     overlaps on the GPU (different streams, or different host threads) race on the array:
 *     order them on one stream or with events.
 *   - No cudaMalloc, cudaFree or other allocating routine is called. */
#define QSA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
qsa_status qsa_sparse_prefill_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* indices, const int32_t* topk_len,
                                      void* out, float* lse,
                                      int64_t n_rows, int32_t n_qheads, int32_t n_kvheads,
                                      int32_t head_dim, int32_t topk, float scale,
                                      int32_t union_g, void* stream);

/* Bytes of union-mode workspace for a call (0 when union_g <= 1): the groups' slot lists,
 * ownership bytes and list lengths, and the counter the attention kernel hands its items out
 * through (zeroed by the union build of the same call).  The workspace is what union mode
 * allocates per call ("DSA prefill ... triton_sparse_mla", Modifications: the union lists and
 * ownership bits are built per step before the attention kernel reads them).
 * qsa_workspace_bytes is the same function under its earlier name. */
size_t qsa_union_workspace_bytes(int64_t n_rows, int32_t topk, int32_t union_g);
size_t qsa_workspace_bytes(int64_t n_rows, int32_t topk, int32_t union_g);

/* Union build on its own ("DSA prefill ... triton_sparse_mla", Modifications and Accuracy
 * Tests: every row's selection is sorted by itself; a slot enters the group's list through
 * the first row holding it, its bits mark every row of the group that selected it, it is
 * listed once, and -1 padding is left out).
 *   sorted_out [n_rows, topk] (nullable): each row's valid slots ascending, then -1.
 *   union_idx  [n_groups, union_g*topk]: group list, canonical order (row 0's emitted slots
 *              ascending, then row 1's, ...), -1 padded.
 *   union_bits [n_groups, union_g*topk] uint8: bit u = row u of the group owns the slot; 0 pad.
 *   union_len  [n_groups]: emitted count.  n_groups = ceil(n_rows / union_g); the last group
 *              may hold fewer rows.  union_g in [1, 8]. */
qsa_status qsa_union_build(const int32_t* indices, const int32_t* topk_len,
                           int64_t n_rows, int32_t topk, int32_t union_g, int64_t n_kv_slots,
                           int32_t* sorted_out, int32_t* union_idx, uint8_t* union_bits,
                           int32_t* union_len, void* stream);

/* Host-only geometry selection (no GPU needed).  num_sms <= 0 queries the current device.
 * Returns QSA_ERR_UNSUPPORTED for shapes the kernel cannot run. */
qsa_status qsa_select_geometry(int32_t n_qheads, int32_t n_kvheads, int32_t union_g,
                               int32_t topk, int32_t head_dim, int64_t n_rows,
                               int32_t num_sms, qsa_geometry* out);

/* Measurement helper: the gather ceiling.  Gathers the first 256 bytes of the cache rows listed
 * in `rows` ([n_table_pieces, 128] int32 row numbers < n_rows of a [n_rows, 256] bf16 cache,
 * 16-byte aligned), 128 rows (32 KiB) per piece, `pieces_per_cta` pieces on every SM, into shared
 * memory with one of the attention kernel's gather engines (engine 0 = cp.async 16-byte copies,
 * 1 = TMA tile::gather4, 2 = both, on alternate stages) and its ring shape, and nothing else.  Writes the elapsed GPU time in
 * milliseconds to *ms_out (host pointer) and synchronises `stream`.  The pages motivate
 * it: the gather is the share of the sparse kernel that grows on newer parts ("DSA prefill ...
 * triton_sparse_mla", Speed Tests), so the kernel's gather rate is reported against this one. */
qsa_status qsa_probe_gather_ceiling(const void* cache, int64_t n_rows, const int32_t* rows,
                                    int64_t n_table_pieces, int32_t pieces_per_cta,
                                    int32_t engine, float* ms_out, void* stream);

/* Failure-detection test hook (no counterpart on the pages): the next attention call
 * (qsa_sparse_prefill*, qsa_sparse_mla_prefill) launches with its index warps withholding their
 * items, so every other role's bounded wait (2 s) runs out.  The kernel records
 * 0x100 | wait site in the device status word, abandons the call (its outputs are unspecified),
 * frees its tensor memory and returns; the context stays usable and qsa_get_device_status then
 * returns QSA_ERR_TIMEOUT.  One-shot, process wide. */
void qsa_debug_stall_next_call(void);

void qsa_get_counters(qsa_counters* out);   /* host pointer */
void qsa_reset_counters(void);
const char* qsa_status_string(qsa_status s);
const char* qsa_version(void);

/* Reads and clears the device status word that kernels set when a bounded wait gives up
 * (0 = no error).  Synchronises `stream`.  Returns QSA_ERR_TIMEOUT if the word was set. */
qsa_status qsa_get_device_status(void* stream, int32_t* status_out);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
