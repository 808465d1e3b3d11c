// Device side of in-kernel paged addressing (PagedAddr in internal.h): the request of a row and
// the physical slot of a logical position.  Shared by the attention kernel's index warp and the
// union build.
#pragma once

#include "internal.h"

namespace qsa {

// Request of a row: the last request whose first row is <= row (warp-uniform arguments; every
// lane of the calling warp must take part).  32-ary search over cu_seqlens_q.
__device__ __forceinline__ int32_t paged_request_of_row(const PagedAddr& pa, int64_t row, int lane) {
  int32_t lo = 0, hi = pa.n_requests - 1;        // answer in [lo, hi]
  while (lo < hi) {
    const int32_t span = hi - lo + 1;
    const int32_t step = (span + 31) / 32;
    const int32_t cand = lo + lane * step;
    const bool le = cand <= hi && pa.cu_seqlens_q[cand] <= row;
    const uint32_t m = __ballot_sync(0xffffffffu, le);
    const int last = m ? 31 - __clz(m) : 0;
    lo = lo + last * step;
    hi = min(hi, lo + step - 1);
  }
  return lo;
}

// Physical slot of logical position x of request req, or -1 when x is padding: negative, at or
// past the request's KV length, past its page-table row, or on a missing / out-of-range page.
__device__ __forceinline__ int64_t paged_slot(const PagedAddr& pa, int32_t req, int32_t kv_len,
                                              int32_t x) {
  if (x < 0 || x >= kv_len) return -1;
  const int32_t page = pa.page_shift >= 0 ? (x >> pa.page_shift) : x / pa.page_size;
  if (page >= pa.pages_per_req) return -1;
  const int32_t pid = __ldg(pa.page_table + static_cast<int64_t>(req) * pa.pages_per_req + page);
  if (pid < 0 || (pa.n_pages > 0 && pid >= pa.n_pages)) return -1;
  return static_cast<int64_t>(pid) * pa.page_size + (x - page * pa.page_size);
}
__device__ __forceinline__ int32_t paged_kv_len(const PagedAddr& pa, int32_t req) {
  return pa.kv_lens ? __ldg(pa.kv_lens + req) : INT32_MAX;
}

}  // namespace qsa
