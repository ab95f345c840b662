// check.cuh -- the bounds-checked build.
//
// Compiled with -DMOE_CHECK=1 (the library variant libmoe_check.so), every
// index that comes out of routing -- an expert number, a position inside an
// expert's capacity, a row of the expert-ordered buffers, a token -- is tested
// against its range before the access it drives.  A failed test records
// STATUS_BOUNDS in the workspace status word (moe_check_status then reports
// MOE_ERR_BOUNDS) and the access is skipped: nothing traps and the kernel runs
// on.  In the normal build the tests compile away.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace moe {

#if defined(MOE_CHECK) && MOE_CHECK
constexpr bool kBoundsChecked = true;
#else
constexpr bool kBoundsChecked = false;
#endif

// True when the access may go ahead.  `ok` is the range test; on failure the
// status word gets STATUS_BOUNDS (when a status word is at hand).
__device__ __forceinline__ bool in_bounds(bool ok, uint32_t* status) {
  if constexpr (kBoundsChecked) {
    if (!ok && status != nullptr) atomicOr(status, STATUS_BOUNDS);
    return ok;
  } else {
    return true;
  }
}

}  // namespace moe
