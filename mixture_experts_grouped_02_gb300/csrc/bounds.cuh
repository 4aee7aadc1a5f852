// bounds.cuh -- the range checks of the checked build.  Compiled with
// -DMOE_BOUNDS_CHECK (libmoe_gb300_checked.so), every index a kernel takes
// from its inputs before a global load or store is checked against the
// buffer it addresses: gathered and scattered rows against the padded list's
// capacity, flat assignment indices against T*K, experts against the experts
// held, block counts against the block array.  A failed check records
// MOE_ERR_BOUNDS in the status word and the access is skipped, so a corrupt
// routing table or workspace shows up as a status instead of a memory fault.
// TMA loads need no check: a box outside the tensor reads the fill value.
// In the product build in_bounds() is the constant true and the checks cost
// nothing.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace moe {

#ifdef MOE_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

// `ok` in the checked build (recording MOE_ERR_BOUNDS when false), else true.
__device__ __forceinline__ bool in_bounds(bool ok, const int32_t* status) {
  if constexpr (kBoundsCheck) {
    if (!ok) report_error(const_cast<int32_t*>(status), MOE_ERR_BOUNDS);
    return ok;
  } else {
    return true;
  }
}

// An align block descriptor {expert, m, first slot, valid rows} that
// addresses only the experts held and slots below the capacity.
__device__ __forceinline__ bool block_in_bounds(const int4& bi, int n_held, long long cap,
                                                int max_rows, const int32_t* status) {
  if constexpr (kBoundsCheck) {
    return in_bounds(bi.x >= 0 && bi.x < n_held && bi.z >= 0 && bi.w >= 1 && bi.w <= max_rows &&
                         static_cast<long long>(bi.z) + bi.w <= cap,
                     status);
  } else {
    return true;
  }
}

// The number of align blocks, or 0 (with MOE_ERR_BOUNDS) when it exceeds the
// block array.
__device__ __forceinline__ int checked_num_blocks(int n, int max_blocks, const int32_t* status) {
  return in_bounds(n >= 0 && n <= max_blocks, status) ? n : 0;
}

}  // namespace moe
