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

// Fan-out copy: source row i (i < n) goes to each non-null dst_of(i, j),
// j < fan -- a token row to the expert segments of its kept slots.  Each row
// is read once.  One issuing thread (thread 0) runs a pipeline over the
// stage's slots: row i's stores are committed as one bulk group, loads run
// nslot - kFanPend rows ahead of the stores, and a slot is refilled only once
// the group that stored it has finished reading shared memory.  `bars` holds
// kFanMaxSlots mbarriers (initialised here; the caller synchronises the block
// before and after the call).  Returns false if a wait ran out.
constexpr int kFanMaxSlots = 16;
constexpr int kFanPend = 2;   // store groups allowed to still read shared memory

template <typename SrcF, typename DstF>
__device__ __forceinline__ bool bulk_fanout_rows(int n, int fan, uint32_t row_bytes, SrcF src_of,
                                                 DstF dst_of, uint8_t* stage,
                                                 uint32_t stage_bytes, uint64_t* bars,
                                                 uint32_t* status, uint32_t timeout_bit,
                                                 uint64_t timeout_ns) {
  const uint32_t fit = stage_bytes / row_bytes;
  const int nslot = (int)(fit < (uint32_t)kFanMaxSlots ? fit : (uint32_t)kFanMaxSlots);
  if (threadIdx.x == 0) {
    for (int w = 0; w < nslot; ++w) mbar_init(smem_u32(bars + w), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0 || n <= 0) return true;
  const uint32_t base = smem_u32(stage);
  const int ahead = nslot - kFanPend;      // >= 1: the caller gives at least 3 slots
  uint32_t phases = 0;
  auto load = [&](int i) {
    const int s = i % nslot;
    mbar_arrive_expect_tx(smem_u32(bars + s), row_bytes);
    bulk_load(base + (uint32_t)s * row_bytes, src_of(i), row_bytes, smem_u32(bars + s));
  };
  int next = 0;
  for (; next < n && next < ahead; ++next) load(next);
  bool ok = true;
  int i = 0;
  for (; i < n; ++i) {
    const int s = i % nslot;
    if (!mbar_wait_bounded(smem_u32(bars + s), (phases >> s) & 1u, timeout_ns, nullptr)) {
      atomicOr(status, timeout_bit);
      ok = false;
      break;
    }
    phases ^= 1u << s;
    for (int j = 0; j < fan; ++j) {
      void* d = dst_of(i, j);
      if (d != nullptr) bulk_store(d, base + (uint32_t)s * row_bytes, row_bytes);
    }
    bulk_commit();
    bulk_wait_read<kFanPend>();           // rows <= i - kFanPend: slots free again
    if (next < n) load(next++);
  }
  if (!ok) {
    // loads issued ahead may still be landing in the stage
    for (int r = i; r < next; ++r) {
      const int s = r % nslot;
      mbar_wait_bounded(smem_u32(bars + s), (phases >> s) & 1u, timeout_ns, nullptr);
      phases ^= 1u << s;
    }
  }
  bulk_commit();
  bulk_wait_all();
  return ok;
}

// The same fan-out copy over rows handed out while the copy runs: claim()
// (called by the issuing thread only) returns the first of up to `batch`
// rows [r, r + batch) the block may copy next, or a negative value when none
// are left; `n` bounds the row indices.  Blocks that finish early take more
// rows, so that the copy ends at about the same time on every block.
template <typename ClaimF, typename SrcF, typename DstF>
__device__ __forceinline__ bool bulk_fanout_claimed(ClaimF claim, int batch, int n, int fan,
                                                    uint32_t row_bytes, SrcF src_of, DstF dst_of,
                                                    uint8_t* stage, uint32_t stage_bytes,
                                                    uint64_t* bars, uint32_t* status,
                                                    uint32_t timeout_bit, uint64_t timeout_ns) {
  const uint32_t fit = stage_bytes / row_bytes;
  const int nslot = (int)(fit < (uint32_t)kFanMaxSlots ? fit : (uint32_t)kFanMaxSlots);
  if (threadIdx.x == 0) {
    for (int w = 0; w < nslot; ++w) mbar_init(smem_u32(bars + w), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return true;
  const uint32_t base = smem_u32(stage);
  const int ahead = nslot - kFanPend;      // >= 1: the caller gives at least 3 slots
  int slot_row[kFanMaxSlots];
  uint32_t phases = 0;
  int cur = 0, end = 0;                    // rows claimed and not yet loaded
  bool more = true;
  auto next_row = [&]() -> int {
    if (cur == end && more) {
      const int r = claim();
      if (r < 0 || r >= n) {
        more = false;
      } else {
        cur = r;
        end = r + batch < n ? r + batch : n;
      }
    }
    return cur < end ? cur++ : -1;
  };
  int issued = 0;
  auto load = [&](int row) {
    const int s = issued % nslot;
    slot_row[s] = row;
    mbar_arrive_expect_tx(smem_u32(bars + s), row_bytes);
    bulk_load(base + (uint32_t)s * row_bytes, src_of(row), row_bytes, smem_u32(bars + s));
    ++issued;
  };
  while (issued < ahead) {
    const int r = next_row();
    if (r < 0) break;
    load(r);
  }
  bool ok = true;
  int done = 0;
  for (; done < issued; ++done) {
    const int s = done % nslot;
    if (!mbar_wait_bounded(smem_u32(bars + s), (phases >> s) & 1u, timeout_ns, nullptr)) {
      atomicOr(status, timeout_bit);
      ok = false;
      break;
    }
    phases ^= 1u << s;
    for (int j = 0; j < fan; ++j) {
      void* d = dst_of(slot_row[s], j);
      if (d != nullptr) bulk_store(d, base + (uint32_t)s * row_bytes, row_bytes);
    }
    bulk_commit();
    bulk_wait_read<kFanPend>();            // rows <= done - kFanPend: slots free again
    const int r = next_row();
    if (r >= 0) load(r);
  }
  if (!ok) {
    // loads issued ahead may still be landing in the stage
    for (int r = done; r < issued; ++r) {
      const int s = r % nslot;
      mbar_wait_bounded(smem_u32(bars + s), (phases >> s) & 1u, timeout_ns, nullptr);
      phases ^= 1u << s;
    }
  }
  bulk_commit();
  bulk_wait_all();
  return ok;
}

}  // namespace moe
