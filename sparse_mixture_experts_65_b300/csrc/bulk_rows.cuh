// bulk_rows.cuh -- block-level copy of whole token rows with bulk async
// copies (global -> shared -> global), used to build the expert-ordered copy
// of the kept token rows.  A few issuing lanes keep many kilobytes in flight
// per SM, where per-thread 16-byte loads leave the copy latency-bound.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace moe {

constexpr int kBulkIssuers = 4;   // warps whose lane 0 issues copies

// Shared memory the caller provides: `stage` (16-byte aligned, `stage_bytes`
// long) and kBulkIssuers mbarriers in `bars` (initialised here by thread 0;
// the caller synchronises the block before and after the call).  Rows are
// 16-byte aligned and `row_bytes` is a multiple of 16.  Row i of the list is
// copied from src_of(i) to dst_of(i) when dst_of(i) is not null.  Issuer w takes
// the rows i = w, w + kBulkIssuers, ... in batches of its slots.  Returns false
// if a wait ran out (the status word then carries `timeout_bit`).
template <typename SrcF, typename DstF>
__device__ __forceinline__ bool bulk_copy_rows(int n, uint32_t row_bytes, SrcF src_of, DstF dst_of,
                                               uint8_t* stage, uint32_t stage_bytes,
                                               uint64_t* bars, uint32_t* status,
                                               uint32_t timeout_bit, uint64_t timeout_ns) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kBulkIssuers; ++w) mbar_init(smem_u32(bars + w), 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool ok = true;
  if (warp < kBulkIssuers && lane == 0) {
    const uint32_t per = stage_bytes / kBulkIssuers / row_bytes;
    const uint32_t nslot = per < 16 ? per : 16;
    const uint32_t slots = smem_u32(stage) + (uint32_t)warp * nslot * row_bytes;
    const uint32_t bar = smem_u32(bars + warp);
    uint32_t phase = 0;
    int batch[16];
    int nb = 0;
    for (int i = warp;; i += kBulkIssuers) {
      const bool more = i < n;
      if (more && dst_of(i) != nullptr) batch[nb++] = i;
      if (nb > 0 && (nb == (int)nslot || !more)) {
        mbar_arrive_expect_tx(bar, (uint32_t)nb * row_bytes);
        for (int j = 0; j < nb; ++j) bulk_load(slots + j * row_bytes, src_of(batch[j]), row_bytes, bar);
        if (!mbar_wait_bounded(bar, phase, timeout_ns, nullptr)) {
          atomicOr(status, timeout_bit);
          ok = false;
          break;
        }
        phase ^= 1u;
        for (int j = 0; j < nb; ++j) bulk_store(dst_of(batch[j]), slots + j * row_bytes, row_bytes);
        bulk_commit();
        bulk_wait_read_all();   // the slots are free again
        nb = 0;
      }
      if (!more) break;
    }
    bulk_commit();
    bulk_wait_all();
  }
  return ok;
}

}  // namespace moe
