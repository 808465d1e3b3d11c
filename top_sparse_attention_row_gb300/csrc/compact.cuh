// Per-row slot compaction shared by the attention kernels' index warps: the row's considered
// slots (the first Lr entries; negative, out-of-range and, for paged calls, untranslatable ones
// dropped) are written in order to a shared-memory list as tensor-map rows slot * n_kvheads +
// kvh.  Warp-collective.
#pragma once

#include "internal.h"
#include "paged.cuh"
#include "ptx.cuh"

namespace qsa {

__device__ __forceinline__ int32_t compact_row_slots(const int32_t* __restrict__ src, int32_t Lr,
                                                     int32_t* sl, uint32_t sl_u32,
                                                     int64_t n_kv_slots, int32_t n_kvheads,
                                                     int32_t kvh, int32_t pad_row,
                                                     const PagedAddr& pa, int64_t row, int lane) {
  for (int j = lane; j < Lr; j += 32) cp_async_4(sl_u32 + 4 * j, src + j);
  cp_async_commit_wait_all();
  __syncwarp();
  int32_t n = 0;
  if (pa.page_table == nullptr) {
    for (int j0 = 0; j0 < Lr; j0 += 32) {
      const int j = j0 + lane;
      const int32_t x = j < Lr ? sl[j] : -1;
      bool valid = x >= 0 && (n_kv_slots == 0 || x < n_kv_slots);
      const int64_t y = static_cast<int64_t>(x) * n_kvheads + kvh;
      valid = valid && y < static_cast<int64_t>(pad_row);
      const uint32_t m = __ballot_sync(0xffffffffu, valid);
      if (valid) sl[n + __popc(m & ((1u << lane) - 1u))] = static_cast<int32_t>(y);
      n += __popc(m);
      __syncwarp();
    }
  } else {
    // Logical positions of the row's request -> physical slots through the page table.  Eight
    // page-table loads per lane are in flight at once; every lane has read its positions of a
    // 256-slot block before the first ballot, so compacting in place never overwrites an
    // unread entry.
    const int32_t req = paged_request_of_row(pa, row, lane);
    const int32_t kvl = paged_kv_len(pa, req);
    for (int j0 = 0; j0 < Lr; j0 += 256) {
      int64_t ps[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + 32 * u + lane;
        ps[u] = paged_slot(pa, req, kvl, j < Lr ? sl[j] : -1);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t x = ps[u];
        bool valid = x >= 0 && (n_kv_slots == 0 || x < n_kv_slots);
        const int64_t y = x * n_kvheads + kvh;
        valid = valid && y < static_cast<int64_t>(pad_row);
        const uint32_t m = __ballot_sync(0xffffffffu, valid);
        if (valid) sl[n + __popc(m & ((1u << lane) - 1u))] = static_cast<int32_t>(y);
        n += __popc(m);
      }
      __syncwarp();
    }
  }
  return n;
}

}  // namespace qsa
