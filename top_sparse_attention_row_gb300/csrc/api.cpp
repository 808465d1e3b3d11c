// C-ABI entry points of libqsa: argument validation, the launch-geometry selector, union-mode
// workspace handling, counters and status reporting.  Every argument error is caught here,
// before any CUDA call, so a bad call enqueues nothing.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace {

using qsa::Geometry;

std::atomic<uint64_t> g_calls_per_token{0}, g_calls_union{0}, g_union_fallbacks{0},
    g_step_downs{0}, g_launches{0};
std::atomic<int> g_stall_next{0};   // armed by qsa_debug_stall_next_call

constexpr size_t kWsAlign = 256;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

// Per-call union workspaces come from a library-owned stream-ordered memory pool per device
// whose release threshold is unbounded: a freed workspace stays in the pool for the next call
// instead of going back to the driver at the next synchronisation, so steady-state calls make
// no driver allocation (the pool holds the largest workspace in use until the process exits).
// Falls back to the device's default pool if a pool cannot be created.
cudaError_t ws_alloc(void** ptr, size_t bytes, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaMallocAsync(ptr, bytes, stream);
  static std::once_flag once[64];
  static cudaMemPool_t pools[64];
  static bool have[64];
  std::call_once(once[dev], [dev] {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    if (cudaMemPoolCreate(&pools[dev], &props) == cudaSuccess) {
      uint64_t threshold = UINT64_MAX;
      have[dev] = cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold,
                                          &threshold) == cudaSuccess;
    }
  });
  return have[dev] ? cudaMallocFromPoolAsync(ptr, bytes, pools[dev], stream)
                   : cudaMallocAsync(ptr, bytes, stream);
}

struct WsLayout {
  size_t idx, bits, len, ctr, total;
};
WsLayout ws_layout(int64_t n_rows, int32_t topk, int32_t G) {
  WsLayout w{};
  if (G <= 1 || n_rows <= 0) return w;
  const int64_t n_groups = ceil_div(n_rows, G);
  const size_t cap = static_cast<size_t>(n_groups) * G * topk;
  w.idx = 0;
  w.bits = round_up(static_cast<int64_t>(cap * 4), kWsAlign);
  w.len = w.bits + round_up(static_cast<int64_t>(cap), kWsAlign);
  w.ctr = w.len + round_up(n_groups * 4, kWsAlign);   // the attention kernel's item counter
  w.total = w.ctr + kWsAlign;
  return w;
}

// Pure host selection.  `forced` may override stages / grid; a stage count that does not fit
// is reduced to the largest that does, rather than refused ("DSA prefill ...
// triton_sparse_mla", Robustness: shared-memory limits are met by a smaller tile).
qsa_status select(int32_t Hq, int32_t Hkv, int32_t union_g, int32_t topk, int32_t head_dim,
                  int64_t n_rows, int32_t num_sms, const qsa_geometry* forced, Geometry* g,
                  bool* fell_back, bool* stepped, bool fp8 = false) {
  // FP8 caches run tiles of at most 32 query columns (fewer kernel instances).
  const int max_np = fp8 ? qsa::kFp8MaxNPad : qsa::kMaxNPad;
  *fell_back = false;
  *stepped = false;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || topk <= 0 || n_rows < 0 || head_dim <= 0 ||
      union_g < 0 || union_g > 8 || num_sms <= 0)
    return QSA_ERR_INVALID_ARG;
  if (head_dim != qsa::kHeadDim) return QSA_ERR_UNSUPPORTED;
  if (n_rows > INT32_MAX) return QSA_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  int G = union_g <= 1 ? 1 : union_g;
  if (G > 1) {
    const int np_u = static_cast<int>(round_up(G * group, 16));
    const bool legal = G * group <= max_np &&
                       qsa::smem_layout(np_u, qsa::kMinStages, 0, fp8).total <= qsa::kSmemLimit &&
                       qsa::union_build_smem_bytes(topk, G) <= static_cast<size_t>(qsa::kUnionMaxSmem) &&
                       static_cast<int64_t>(G) * topk <= INT32_MAX / 2;
    if (!legal) {
      G = 1;
      *fell_back = true;
    }
  }
  int chunks, chunk_cols, np, slot_cap;
  if (G == 1) {
    chunks = static_cast<int>(ceil_div(group, max_np));
    chunk_cols = static_cast<int>(ceil_div(group, chunks));
    np = static_cast<int>(round_up(chunk_cols, 16));
    slot_cap = static_cast<int>(round_up(topk, qsa::kTileTokens));
  } else {
    chunks = 1;
    chunk_cols = G * group;
    np = static_cast<int>(round_up(chunk_cols, 16));
    slot_cap = 0;
  }
  const int64_t n_groups = ceil_div(n_rows, G);
  const int64_t n_items = n_groups * Hkv * chunks;
  // Split items: per-token bf16 calls with fewer items than SMs give each item a cluster of
  // `split` CTAs (each a contiguous range of the row's 128-slot tiles, at least one tile each), so
  // a short call still fills the GPU ("[QSA] Tune sm120 sparse prefill geometry", Query-count
  // sweep: the row count decides the launch shape).
  int split = 1;
  if (G == 1 && !fp8 && np <= qsa::kSplitMaxNPad) {
    const int64_t tiles = ceil_div(topk, qsa::kTileTokens);
    for (int c = qsa::kMaxSplit; c >= 2; c /= 2) {
      if (n_items > 0 && n_items * c <= num_sms && c <= tiles) {
        split = c;
        break;
      }
    }
    if (forced && forced->split > 0) {
      split = 1;
      while (split * 2 <= forced->split && split * 2 <= qsa::kMaxSplit) split *= 2;
    }
  }
  int stages = 0;
  // even stage counts: a piece pair's two stages share one empty barrier
  for (int s = qsa::kMaxStages; s >= qsa::kMinStages; s -= 2) {
    if (qsa::smem_layout(np, s, slot_cap, fp8, split).total <= qsa::kSmemLimit) {
      stages = s;
      break;
    }
  }
  if (stages == 0) return QSA_ERR_UNSUPPORTED;   // per-token slot list too large for topk
  if (forced && forced->stages > 0) {
    int want = forced->stages < qsa::kMinStages ? qsa::kMinStages : forced->stages & ~1;
    if (want > stages) {
      *stepped = true;
      want = stages;
    }
    stages = want;
  }
  // grid: whole clusters, at most one CTA per SM
  int64_t clusters = n_items < num_sms / split ? n_items : num_sms / split;
  if (clusters < 1) clusters = 1;
  if (forced && forced->grid > 0 && forced->grid / split < clusters)
    clusters = forced->grid / split > 0 ? forced->grid / split : 1;
  const int64_t grid = clusters * split;
  g->np = np;
  g->cols = chunk_cols;
  g->head_chunks = chunks;
  g->chunk_cols = chunk_cols;
  g->union_g = G;
  g->stages = stages;
  g->grid = static_cast<int>(grid);
  g->smem_bytes = qsa::smem_layout(np, stages, slot_cap, fp8, split).total;
  g->split = split;
  // S^T buffers (lookahead + 1) + two O^T halves
  g->tmem_cols = pow2_at_least((qsa::lookahead_for(G > 1) + 3) * np);
  g->slot_cap = slot_cap;
  g->n_items = n_items;
  g->n_groups = static_cast<int>(n_groups);
  return QSA_OK;
}

// MLA shape (d_qk 576, d_v 512, one latent KV row per slot): N = heads (or G x heads) padded
// to 16 or 32; the latent ring takes 5 stages when shared memory allows (one spare stage lets
// the next tile's first latent chunk overlap the softmax), else 4.
qsa_status select_mla(int32_t n_heads, int32_t union_g, int32_t topk, int32_t d_qk, int32_t d_v,
                      int64_t n_rows, int32_t num_sms, qsa::MlaGeometry* g, bool* fell_back) {
  *fell_back = false;
  if (n_heads <= 0 || topk <= 0 || n_rows < 0 || d_qk <= 0 || d_v <= 0 || union_g < 0 ||
      union_g > 8 || num_sms <= 0)
    return QSA_ERR_INVALID_ARG;
  if (d_qk != qsa::kMlaDqk || d_v != qsa::kMlaDv) return QSA_ERR_UNSUPPORTED;
  if (n_rows > INT32_MAX) return QSA_ERR_UNSUPPORTED;
  auto stages_for = [](int np, int slot_cap) {
    for (int rp = qsa::kMlaPairs + 1; rp >= qsa::kMlaPairs; --rp)
      if (qsa::mla_smem_layout(np, rp, slot_cap).total <= qsa::kSmemLimit) return rp;
    return 0;
  };
  int G = union_g <= 1 ? 1 : union_g;
  if (G > 1) {
    const int np_u = static_cast<int>(round_up(static_cast<int64_t>(G) * n_heads, 16));
    const bool legal = static_cast<int64_t>(G) * n_heads <= qsa::kMlaMaxNPad &&
                       stages_for(np_u, 0) > 0 &&
                       qsa::union_build_smem_bytes(topk, G) <= static_cast<size_t>(qsa::kUnionMaxSmem) &&
                       static_cast<int64_t>(G) * topk <= INT32_MAX / 2;
    if (!legal) {
      G = 1;
      *fell_back = true;
    }
  }
  int chunks, chunk_cols, slot_cap;
  if (G == 1) {
    chunks = static_cast<int>(ceil_div(n_heads, qsa::kMlaMaxNPad));
    chunk_cols = static_cast<int>(ceil_div(n_heads, chunks));
    slot_cap = static_cast<int>(round_up(topk, qsa::kTileTokens));
  } else {
    chunks = 1;
    chunk_cols = G * n_heads;
    slot_cap = 0;
  }
  const int np = static_cast<int>(round_up(chunk_cols, 16));
  const int rp = stages_for(np, slot_cap);
  if (rp == 0) return QSA_ERR_UNSUPPORTED;   // per-token slot list too large for topk
  const int64_t n_groups = ceil_div(n_rows, G);
  const int64_t n_items = n_groups * chunks;
  g->np = np;
  g->cols = chunk_cols;
  g->head_chunks = chunks;
  g->chunk_cols = chunk_cols;
  g->union_g = G;
  g->pair_stages = rp;
  g->grid = static_cast<int>(n_items < num_sms ? n_items : num_sms);
  g->smem_bytes = qsa::mla_smem_layout(np, rp, slot_cap).total;
  g->tmem_cols = pow2_at_least(6 * np);
  g->slot_cap = slot_cap;
  g->n_items = n_items;
  g->n_groups = static_cast<int>(n_groups);
  return QSA_OK;
}

void mla_to_public(const qsa::MlaGeometry& g, qsa_geometry* out) {
  out->tile_tokens = qsa::kTileTokens;
  out->stages = g.pair_stages;
  out->n_pad = g.np;
  out->cols = g.cols;
  out->head_chunks = g.head_chunks;
  out->union_g = g.union_g;
  out->grid = g.grid;
  out->threads = qsa::kMlaThreads;
  out->smem_bytes = g.smem_bytes;
  out->tmem_cols = g.tmem_cols;
  out->n_items = g.n_items;
  out->split = 1;
}

void to_public(const Geometry& g, qsa_geometry* out) {
  out->tile_tokens = qsa::kTileTokens;
  out->stages = g.stages;
  out->n_pad = g.np;
  out->cols = g.cols;
  out->head_chunks = g.head_chunks;
  out->union_g = g.union_g;
  out->grid = g.grid;
  out->threads = qsa::kThreads;
  out->smem_bytes = g.smem_bytes;
  out->tmem_cols = g.tmem_cols;
  out->n_items = g.n_items;
  out->split = g.split;
}

// Gather engine: TMA tile::gather4 by default; QSA_GATHER=cpasync selects cp.async 16-byte
// copies (both are exact; the switch exists to compare them).
bool gather_engine_is_tma() {
  static const bool tma = [] {
    const char* e = std::getenv("QSA_GATHER");
    return e == nullptr || std::strcmp(e, "cpasync") != 0;
  }();
  return tma;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// QSA_LOG=1: one stderr line per attention call with the geometry the selector chose.
bool log_geometry() {
  static const bool on = [] {
    const char* e = std::getenv("QSA_LOG");
    return e != nullptr && std::strcmp(e, "1") == 0;
  }();
  return on;
}

// Device checks: compute capability 10.3 and the SM count (cached per device).
qsa_status device_sms(int32_t* sms) {
  static std::atomic<int32_t> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QSA_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    const int32_t c = cache[dev].load();
    if (c > 0) {
      *sms = c;
      return QSA_OK;
    }
  }
  int major = 0, minor = 0, n = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return QSA_ERR_CUDA;
  if (major != 10 || minor != 3) return QSA_ERR_UNSUPPORTED;
  if (dev >= 0 && dev < 64) cache[dev].store(n);
  *sms = n;
  return QSA_OK;
}

// FP8 caches: e4m3 bytes with per-page, per-KV-head fp32 scales.
struct Fp8Cache {
  const float* k_scale;
  const float* v_scale;
  int32_t page_size;
};

qsa_status run(const void* q, const void* k_cache, const void* v_cache, const int32_t* indices,
               const int32_t* topk_len, void* out, float* lse, int64_t n_rows, int32_t n_qheads,
               int32_t n_kvheads, int32_t head_dim, int32_t topk, float scale, int32_t union_g,
               int64_t n_kv_slots, void* workspace, size_t workspace_bytes,
               const qsa_geometry* forced, const qsa::PagedAddr* paged, void* stream_v,
               const Fp8Cache* fp8 = nullptr) {
  if (!q || !k_cache || !v_cache || !indices || !out) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return QSA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || n_kv_slots < 0) return QSA_ERR_INVALID_ARG;
  if (n_kvheads > 0 && n_kv_slots > 0 && n_kv_slots * n_kvheads >= INT32_MAX)
    return QSA_ERR_UNSUPPORTED;
  Geometry g{};
  bool fell_back = false, stepped = false;
  // Validate the shape on the host first (num_sms = 1 stands in until the device is known).
  qsa_status st = select(n_qheads, n_kvheads, union_g, topk, head_dim, n_rows, 1, forced, &g,
                         &fell_back, &stepped, fp8 != nullptr);
  if (st != QSA_OK) return st;
  if (n_rows == 0) return QSA_OK;
  int32_t sms = 0;
  st = device_sms(&sms);
  if (st != QSA_OK) return st;
  st = select(n_qheads, n_kvheads, union_g, topk, head_dim, n_rows, sms, forced, &g, &fell_back,
              &stepped, fp8 != nullptr);
  if (st != QSA_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  if (log_geometry())
    std::fprintf(stderr,
                 "qsa: d=256 rows=%lld heads=%d/%d topk=%d union=%d%s -> N=%d cols=%d chunks=%d "
                 "stages=%d grid=%d split=%d smem=%d tmem=%d items=%lld%s%s\n",
                 static_cast<long long>(n_rows), n_qheads, n_kvheads, topk, g.union_g,
                 fp8 ? " fp8" : (paged ? " paged" : ""), g.np, g.cols, g.head_chunks, g.stages,
                 g.grid, g.split, g.smem_bytes, g.tmem_cols, static_cast<long long>(g.n_items),
                 fell_back ? " (union fallback)" : "", stepped ? " (stepped down)" : "");

  qsa::PrefillParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.indices = indices;
  p.topk_len = topk_len;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.n_rows = n_rows;
  p.n_items = g.n_items;
  p.n_kv_slots = n_kv_slots;
  p.n_qheads = n_qheads;
  p.n_kvheads = n_kvheads;
  p.group = n_qheads / n_kvheads;
  p.topk = topk;
  p.union_g = g.union_g;
  p.n_groups = g.n_groups;
  p.head_chunks = g.head_chunks;
  p.chunk_cols = g.chunk_cols;
  p.stages = g.stages;
  p.slot_cap = g.slot_cap;
  p.tmem_cols = g.tmem_cols;
  p.gather_tma = gather_engine_is_tma() ? 1 : 0;
  p.k_bytes = static_cast<const uint8_t*>(k_cache);
  p.v_bytes = static_cast<const uint8_t*>(v_cache);
  p.scale_log2 = scale * 1.4426950408889634f;
  const int64_t tmap_rows = n_kv_slots > 0 ? n_kv_slots * n_kvheads : static_cast<int64_t>(INT32_MAX);
  p.pad_row = static_cast<int32_t>(tmap_rows);
  if (paged) p.pa = *paged;
  p.stall_first_item = g_stall_next.exchange(0);
  p.split = g.split;
  if (fp8) {
    p.k_scale = fp8->k_scale;
    p.v_scale = fp8->v_scale;
    p.page_size = fp8->page_size;
    p.page_shift = -1;
    p.kv_shift = -1;
    for (int s = 0; s < 31; ++s) {
      if ((int32_t{1} << s) == fp8->page_size) p.page_shift = s;
      if ((int32_t{1} << s) == n_kvheads) p.kv_shift = s;
    }
    p.gather_tma = 1;   // the FP8 gather is TMA only
  }

  void* ws = nullptr;
  bool own_ws = false;
  if (g.union_g > 1) {
    const WsLayout w = ws_layout(n_rows, topk, g.union_g);
    if (workspace) {
      if (workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0)
        return QSA_ERR_WORKSPACE;
      ws = workspace;
    } else {
      if (ws_alloc(&ws, w.total, stream) != cudaSuccess) return QSA_ERR_CUDA;
      own_ws = true;
    }
    uint8_t* b = static_cast<uint8_t*>(ws);
    p.union_idx = reinterpret_cast<int32_t*>(b + w.idx);
    p.union_bits = b + w.bits;
    p.union_len = reinterpret_cast<int32_t*>(b + w.len);
    p.item_counter = reinterpret_cast<int32_t*>(b + w.ctr);
    cudaError_t e = qsa::launch_union_build(indices, topk_len, n_rows, topk, g.union_g, n_kv_slots,
                                            nullptr, const_cast<int32_t*>(p.union_idx),
                                            const_cast<uint8_t*>(p.union_bits),
                                            const_cast<int32_t*>(p.union_len), false, paged,
                                            stream, p.item_counter);
    if (e != cudaSuccess) {
      if (own_ws) cudaFreeAsync(ws, stream);
      return QSA_ERR_CUDA;
    }
    g_launches.fetch_add(1);
  }
  cudaError_t e = qsa::launch_prefill(p, g, k_cache, v_cache, tmap_rows, stream);
  if (own_ws) cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) return QSA_ERR_CUDA;
  g_launches.fetch_add(1);
  if (g.union_g > 1) g_calls_union.fetch_add(1); else g_calls_per_token.fetch_add(1);
  if (fell_back) g_union_fallbacks.fetch_add(1);
  if (stepped) g_step_downs.fetch_add(1);
  return QSA_OK;
}

qsa_status run_mla(const void* q, const void* kv_cache, const int32_t* indices,
                   const int32_t* topk_len, void* out, float* lse, int64_t n_rows, int32_t n_heads,
                   int32_t d_qk, int32_t d_v, int32_t topk, float scale, int32_t union_g,
                   int64_t n_kv_slots, const qsa::PagedAddr* paged, void* stream_v) {
  if (!q || !kv_cache || !indices || !out) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return QSA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || n_kv_slots < 0) return QSA_ERR_INVALID_ARG;
  if (n_kv_slots >= INT32_MAX) return QSA_ERR_UNSUPPORTED;
  qsa::MlaGeometry g{};
  bool fell_back = false;
  qsa_status st = select_mla(n_heads, union_g, topk, d_qk, d_v, n_rows, 1, &g, &fell_back);
  if (st != QSA_OK) return st;
  if (n_rows == 0) return QSA_OK;
  int32_t sms = 0;
  st = device_sms(&sms);
  if (st != QSA_OK) return st;
  st = select_mla(n_heads, union_g, topk, d_qk, d_v, n_rows, sms, &g, &fell_back);
  if (st != QSA_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  if (log_geometry())
    std::fprintf(stderr,
                 "qsa: mla rows=%lld heads=%d topk=%d union=%d%s -> N=%d cols=%d chunks=%d "
                 "latent_stages=%d grid=%d smem=%d tmem=%d items=%lld%s\n",
                 static_cast<long long>(n_rows), n_heads, topk, g.union_g, paged ? " paged" : "",
                 g.np, g.cols, g.head_chunks, g.pair_stages, g.grid, g.smem_bytes, g.tmem_cols,
                 static_cast<long long>(g.n_items), fell_back ? " (union fallback)" : "");

  qsa::MlaParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.indices = indices;
  p.topk_len = topk_len;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  if (qsa::device_status_address(&p.status) != cudaSuccess) return QSA_ERR_CUDA;
  p.n_rows = n_rows;
  p.n_items = g.n_items;
  p.n_kv_slots = n_kv_slots;
  p.n_heads = n_heads;
  p.topk = topk;
  p.union_g = g.union_g;
  p.n_groups = g.n_groups;
  p.head_chunks = g.head_chunks;
  p.chunk_cols = g.chunk_cols;
  p.pair_stages = g.pair_stages;
  p.slot_cap = g.slot_cap;
  p.tmem_cols = g.tmem_cols;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int64_t tmap_rows = n_kv_slots > 0 ? n_kv_slots : static_cast<int64_t>(INT32_MAX);
  p.pad_row = static_cast<int32_t>(tmap_rows);
  if (paged) p.pa = *paged;
  p.stall_first_item = g_stall_next.exchange(0);

  void* ws = nullptr;
  if (g.union_g > 1) {
    const WsLayout w = ws_layout(n_rows, topk, g.union_g);
    if (ws_alloc(&ws, w.total, stream) != cudaSuccess) return QSA_ERR_CUDA;
    uint8_t* b = static_cast<uint8_t*>(ws);
    p.union_idx = reinterpret_cast<int32_t*>(b + w.idx);
    p.union_bits = b + w.bits;
    p.union_len = reinterpret_cast<int32_t*>(b + w.len);
    p.item_counter = reinterpret_cast<int32_t*>(b + w.ctr);
    cudaError_t e = qsa::launch_union_build(indices, topk_len, n_rows, topk, g.union_g, n_kv_slots,
                                            nullptr, const_cast<int32_t*>(p.union_idx),
                                            const_cast<uint8_t*>(p.union_bits),
                                            const_cast<int32_t*>(p.union_len), false, paged,
                                            stream, p.item_counter);
    if (e != cudaSuccess) {
      cudaFreeAsync(ws, stream);
      return QSA_ERR_CUDA;
    }
    g_launches.fetch_add(1);
  }
  cudaError_t e = qsa::launch_mla(p, g, kv_cache, tmap_rows, stream);
  if (ws) cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) return QSA_ERR_CUDA;
  g_launches.fetch_add(1);
  if (g.union_g > 1) g_calls_union.fetch_add(1); else g_calls_per_token.fetch_add(1);
  if (fell_back) g_union_fallbacks.fetch_add(1);
  return QSA_OK;
}

qsa_status page_split_args(const void* src_pool, void* dst_pool, int64_t n_src_pages,
                           int32_t src_page_size, int32_t dst_page_size, int32_t n_sections,
                           const int32_t* section_bytes, qsa::PageSections* sec) {
  if (!src_pool || !dst_pool || !section_bytes || n_src_pages < 0 || src_page_size < 1 ||
      dst_page_size < 1 || src_page_size % dst_page_size != 0 || n_sections < 1 ||
      n_sections > qsa::kMaxPageSections || !aligned16(src_pool) || !aligned16(dst_pool))
    return QSA_ERR_INVALID_ARG;
  sec->n = n_sections;
  sec->token_bytes = 0;
  for (int k = 0; k < n_sections; ++k) {
    if (section_bytes[k] <= 0 || section_bytes[k] % 16 != 0) return QSA_ERR_INVALID_ARG;
    sec->bytes[k] = section_bytes[k];
    sec->token_bytes += section_bytes[k];
  }
  if (n_src_pages * (src_page_size / dst_page_size) >= INT32_MAX) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

// Paged-call metadata -> PagedAddr and the physical slot count (0 = unchecked).
qsa_status paged_args(const int32_t* cu_seqlens_q, const int32_t* kv_lens, const int32_t* page_table,
                      int32_t n_requests, int32_t pages_per_req, int32_t page_size,
                      int64_t n_pages, int32_t n_kvheads, qsa::PagedAddr* pa, int64_t* n_kv_slots) {
  if (!cu_seqlens_q || !page_table) return QSA_ERR_INVALID_ARG;
  if (n_requests < 1 || pages_per_req < 1 || page_size < 1 || n_pages < 0)
    return QSA_ERR_INVALID_ARG;
  *n_kv_slots = 0;
  if (n_pages > 0) {
    *n_kv_slots = n_pages * page_size;
    if (n_kvheads > 0 && *n_kv_slots * n_kvheads >= INT32_MAX) return QSA_ERR_UNSUPPORTED;
  }
  pa->page_table = page_table;
  pa->cu_seqlens_q = cu_seqlens_q;
  pa->kv_lens = kv_lens;
  pa->n_requests = n_requests;
  pa->pages_per_req = pages_per_req;
  pa->page_size = page_size;
  pa->page_shift = -1;
  for (int s = 0; s < 31; ++s)
    if ((int32_t{1} << s) == page_size) pa->page_shift = s;
  pa->n_pages = n_pages;
  return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status qsa_sparse_mla_prefill(const void* q, const void* kv_cache, const int32_t* indices,
                                  const int32_t* topk_len, void* out, float* lse, int64_t n_rows,
                                  int32_t n_heads, int32_t d_qk, int32_t d_v, int32_t topk,
                                  float scale, int32_t union_g, int64_t n_kv_slots, void* stream) {
  return run_mla(q, kv_cache, indices, topk_len, out, lse, n_rows, n_heads, d_qk, d_v, topk, scale,
                 union_g, n_kv_slots, nullptr, stream);
}

qsa_status qsa_page_mark(const int32_t* indices, int64_t n_indices, int32_t src_page_size,
                         int64_t n_src_pages, uint8_t* mark, void* stream) {
  if (!mark || (!indices && n_indices > 0) || n_indices < 0 || src_page_size < 1 || n_src_pages < 0)
    return QSA_ERR_INVALID_ARG;
  if (n_src_pages == 0) return QSA_OK;
  int32_t sms = 0;
  qsa_status st = device_sms(&sms);
  if (st != QSA_OK) return st;
  if (qsa::launch_page_mark(indices, n_indices, src_page_size, n_src_pages, mark, sms,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QSA_ERR_CUDA;
  if (n_indices > 0) g_launches.fetch_add(1);
  return QSA_OK;
}


qsa_status qsa_page_split(const void* src_pool, void* dst_pool, const uint8_t* mark,
                          int64_t n_src_pages, int32_t src_page_size, int32_t dst_page_size,
                          int32_t n_sections, const int32_t* section_bytes, void* stream) {
  qsa::PageSections sec{};
  qsa_status st = page_split_args(src_pool, dst_pool, n_src_pages, src_page_size, dst_page_size,
                                  n_sections, section_bytes, &sec);
  if (st != QSA_OK || n_src_pages == 0) return st;
  int32_t sms = 0;
  st = device_sms(&sms);
  if (st != QSA_OK) return st;
  if (qsa::launch_page_split(src_pool, dst_pool, mark, n_src_pages, src_page_size, dst_page_size,
                             sec, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QSA_ERR_CUDA;
  g_launches.fetch_add(1);
  return QSA_OK;
}

qsa_status qsa_split_touched_pages(const int32_t* indices, int64_t n_indices, const void* src_pool,
                                   void* dst_pool, uint8_t* mark, int64_t n_src_pages,
                                   int32_t src_page_size, int32_t dst_page_size,
                                   int32_t n_sections, const int32_t* section_bytes,
                                   void* stream) {
  qsa::PageSections sec{};
  qsa_status st = page_split_args(src_pool, dst_pool, n_src_pages, src_page_size, dst_page_size,
                                  n_sections, section_bytes, &sec);
  if (st != QSA_OK) return st;
  if (!mark || (!indices && n_indices > 0) || n_indices < 0) return QSA_ERR_INVALID_ARG;
  st = qsa_page_mark(indices, n_indices, src_page_size, n_src_pages, mark, stream);
  if (st != QSA_OK || n_src_pages == 0) return st;
  if (qsa::launch_page_split(src_pool, dst_pool, mark, n_src_pages, src_page_size, dst_page_size,
                             sec, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QSA_ERR_CUDA;
  g_launches.fetch_add(1);
  return QSA_OK;
}

qsa_status qsa_select_mla_geometry(int32_t n_heads, int32_t union_g, int32_t topk, int32_t d_qk,
                                   int32_t d_v, int64_t n_rows, int32_t num_sms,
                                   qsa_geometry* out) {
  if (!out) return QSA_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    qsa_status st = device_sms(&num_sms);
    if (st != QSA_OK) return st;
  }
  qsa::MlaGeometry g{};
  bool fb = false;
  qsa_status st = select_mla(n_heads, union_g, topk, d_qk, d_v, n_rows, num_sms, &g, &fb);
  if (st != QSA_OK) return st;
  mla_to_public(g, out);
  return QSA_OK;
}


qsa_status qsa_sparse_prefill(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* indices, const int32_t* topk_len, void* out, float* lse,
                              int64_t n_rows, int32_t n_qheads, int32_t n_kvheads, int32_t head_dim,
                              int32_t topk, float scale, int32_t union_g, void* stream) {
  return run(q, k_cache, v_cache, indices, topk_len, out, lse, n_rows, n_qheads, n_kvheads,
             head_dim, topk, scale, union_g, 0, nullptr, 0, nullptr, nullptr, stream);
}

qsa_status qsa_sparse_prefill_fp8(const void* q, const void* k_cache, const void* v_cache,
                                  const float* k_scale, const float* v_scale, int32_t page_size,
                                  const int32_t* indices, const int32_t* topk_len, void* out,
                                  float* lse, int64_t n_rows, int32_t n_qheads, int32_t n_kvheads,
                                  int32_t head_dim, int32_t topk, float scale, int32_t union_g,
                                  int64_t n_kv_slots, void* stream) {
  if (!k_scale || !v_scale || page_size < 1) return QSA_ERR_INVALID_ARG;
  const Fp8Cache f{k_scale, v_scale, page_size};
  return run(q, k_cache, v_cache, indices, topk_len, out, lse, n_rows, n_qheads, n_kvheads,
             head_dim, topk, scale, union_g, n_kv_slots, nullptr, 0, nullptr, nullptr, stream, &f);
}

qsa_status qsa_sparse_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* indices, const int32_t* topk_len,
                                    const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                    const int32_t* page_table, void* out, float* lse,
                                    int64_t n_rows, int32_t n_requests, int32_t pages_per_req,
                                    int32_t page_size, int64_t n_pages, int32_t n_qheads,
                                    int32_t n_kvheads, int32_t head_dim, int32_t topk, float scale,
                                    int32_t union_g, void* stream) {
  qsa::PagedAddr pa{};
  int64_t n_kv_slots = 0;
  const qsa_status st = paged_args(cu_seqlens_q, kv_lens, page_table, n_requests, pages_per_req,
                                   page_size, n_pages, n_kvheads, &pa, &n_kv_slots);
  if (st != QSA_OK) return st;
  return run(q, k_cache, v_cache, indices, topk_len, out, lse, n_rows, n_qheads, n_kvheads,
             head_dim, topk, scale, union_g, n_kv_slots, nullptr, 0, nullptr, &pa, stream);
}

qsa_status qsa_sparse_prefill_fp8_paged(const void* q, const void* k_cache, const void* v_cache,
                                        const float* k_scale, const float* v_scale,
                                        int32_t fp8_page_size, const int32_t* indices,
                                        const int32_t* topk_len, const int32_t* cu_seqlens_q,
                                        const int32_t* kv_lens, const int32_t* page_table,
                                        void* out, float* lse, int64_t n_rows, int32_t n_requests,
                                        int32_t pages_per_req, int32_t page_size, int64_t n_pages,
                                        int32_t n_qheads, int32_t n_kvheads, int32_t head_dim,
                                        int32_t topk, float scale, int32_t union_g, void* stream) {
  if (!k_scale || !v_scale || fp8_page_size < 1) return QSA_ERR_INVALID_ARG;
  qsa::PagedAddr pa{};
  int64_t n_kv_slots = 0;
  const qsa_status st = paged_args(cu_seqlens_q, kv_lens, page_table, n_requests, pages_per_req,
                                   page_size, n_pages, n_kvheads, &pa, &n_kv_slots);
  if (st != QSA_OK) return st;
  const Fp8Cache f{k_scale, v_scale, fp8_page_size};
  return run(q, k_cache, v_cache, indices, topk_len, out, lse, n_rows, n_qheads, n_kvheads,
             head_dim, topk, scale, union_g, n_kv_slots, nullptr, 0, nullptr, &pa, stream, &f);
}

qsa_status qsa_sparse_mla_prefill_paged(const void* q, const void* kv_cache, const int32_t* indices,
                                        const int32_t* topk_len, const int32_t* cu_seqlens_q,
                                        const int32_t* kv_lens, const int32_t* page_table,
                                        void* out, float* lse, int64_t n_rows, int32_t n_requests,
                                        int32_t pages_per_req, int32_t page_size, int64_t n_pages,
                                        int32_t n_heads, int32_t d_qk, int32_t d_v, int32_t topk,
                                        float scale, int32_t union_g, void* stream) {
  qsa::PagedAddr pa{};
  int64_t n_kv_slots = 0;
  const qsa_status st = paged_args(cu_seqlens_q, kv_lens, page_table, n_requests, pages_per_req,
                                   page_size, n_pages, 1, &pa, &n_kv_slots);
  if (st != QSA_OK) return st;
  return run_mla(q, kv_cache, indices, topk_len, out, lse, n_rows, n_heads, d_qk, d_v, topk, scale,
                 union_g, n_kv_slots, &pa, stream);
}

qsa_status qsa_sparse_prefill_ex(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* indices, const int32_t* topk_len, void* out,
                                 float* lse, int64_t n_rows, int32_t n_qheads, int32_t n_kvheads,
                                 int32_t head_dim, int32_t topk, float scale, int32_t union_g,
                                 int64_t n_kv_slots, void* workspace, size_t workspace_bytes,
                                 const qsa_geometry* forced, void* stream) {
  return run(q, k_cache, v_cache, indices, topk_len, out, lse, n_rows, n_qheads, n_kvheads,
             head_dim, topk, scale, union_g, n_kv_slots, workspace, workspace_bytes, forced, nullptr,
             stream);
}

size_t qsa_union_workspace_bytes(int64_t n_rows, int32_t topk, int32_t union_g) {
  if (topk <= 0 || n_rows <= 0 || union_g <= 1 || union_g > 8) return 0;
  return ws_layout(n_rows, topk, union_g).total;
}

size_t qsa_workspace_bytes(int64_t n_rows, int32_t topk, int32_t union_g) {
  return qsa_union_workspace_bytes(n_rows, topk, union_g);
}

qsa_status qsa_union_build(const int32_t* indices, const int32_t* topk_len, int64_t n_rows,
                           int32_t topk, int32_t union_g, int64_t n_kv_slots, int32_t* sorted_out,
                           int32_t* union_idx, uint8_t* union_bits, int32_t* union_len,
                           void* stream) {
  if (!indices || !union_idx || !union_bits || !union_len) return QSA_ERR_INVALID_ARG;
  if (n_rows < 0 || topk <= 0 || union_g < 1 || union_g > 8 || n_kv_slots < 0)
    return QSA_ERR_INVALID_ARG;
  const size_t need = sorted_out ? qsa::union_sort_smem_bytes(topk, union_g)
                                 : qsa::union_build_smem_bytes(topk, union_g);
  if (n_rows > INT32_MAX || need > static_cast<size_t>(qsa::kUnionMaxSmem)) return QSA_ERR_UNSUPPORTED;
  if (n_rows == 0) return QSA_OK;
  int32_t sms = 0;
  qsa_status st = device_sms(&sms);
  if (st != QSA_OK) return st;
  cudaError_t e = qsa::launch_union_build(indices, topk_len, n_rows, topk, union_g, n_kv_slots,
                                          sorted_out, union_idx, union_bits, union_len, true,
                                          nullptr, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return QSA_ERR_CUDA;
  g_launches.fetch_add(1);
  return QSA_OK;
}

qsa_status qsa_select_geometry(int32_t n_qheads, int32_t n_kvheads, int32_t union_g, int32_t topk,
                               int32_t head_dim, int64_t n_rows, int32_t num_sms,
                               qsa_geometry* out) {
  if (!out) return QSA_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    qsa_status st = device_sms(&num_sms);
    if (st != QSA_OK) return st;
  }
  Geometry g{};
  bool fb = false, sd = false;
  qsa_status st = select(n_qheads, n_kvheads, union_g, topk, head_dim, n_rows, num_sms, nullptr, &g,
                         &fb, &sd);
  if (st != QSA_OK) return st;
  to_public(g, out);
  return QSA_OK;
}

void qsa_debug_stall_next_call(void) { g_stall_next.store(1); }

void qsa_get_counters(qsa_counters* out) {
  if (!out) return;
  out->calls_per_token = g_calls_per_token.load();
  out->calls_union = g_calls_union.load();
  out->union_fallbacks = g_union_fallbacks.load();
  out->step_downs = g_step_downs.load();
  out->kernel_launches = g_launches.load();
}

void qsa_reset_counters(void) {
  g_calls_per_token = 0;
  g_calls_union = 0;
  g_union_fallbacks = 0;
  g_step_downs = 0;
  g_launches = 0;
}

const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument";
    case QSA_ERR_UNSUPPORTED: return "unsupported shape or device";
    case QSA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case QSA_ERR_CUDA: return "CUDA error";
    case QSA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* qsa_version(void) { return "qsa 0.1.0 (sm_103a, tcgen05 + TMA gather4)"; }

qsa_status qsa_get_device_status(void* stream, int32_t* status_out) {
  if (!status_out) return QSA_ERR_INVALID_ARG;
  int32_t s = 0;
  if (qsa::read_and_clear_device_status(static_cast<cudaStream_t>(stream), &s) != cudaSuccess)
    return QSA_ERR_CUDA;
  *status_out = s;
  return s == 0 ? QSA_OK : QSA_ERR_TIMEOUT;
}

}  // extern "C"
