// Range checks of the data-dependent indices the kernels gather from and
// scatter to (neuron indices read from TwELL / ELL columns, counts read as
// loop bounds, spill slots, row maps, per-neuron record offsets, union
// positions).  In a build with -DTWELL_BOUNDS_CHECK an index outside its
// buffer sets TWELL_FLAG_BOUNDS in the caller's status word and the access
// is skipped (a store) or redirected to element 0 (a load), so the kernel
// reports the fault instead of touching memory it does not own; in the
// normal build the checks compile to nothing.
#pragma once

#include <cstdint>

#include "../../include/twell.h"

namespace twell {

#ifdef TWELL_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

// True when 0 <= idx < n.  In the checking build a false result also sets
// TWELL_FLAG_BOUNDS in *status; in the normal build the result is always
// true.
__device__ __forceinline__ bool in_bounds(long long idx, long long n, int32_t* status) {
  if (!kBoundsCheck) return true;
  if (idx >= 0 && idx < n) return true;
  if (status) atomicOr(status, TWELL_FLAG_BOUNDS);
  return false;
}

// idx when it is in [0, n), else 0 (and TWELL_FLAG_BOUNDS in the checking
// build): for gathers whose load must still happen.
__device__ __forceinline__ long long clamp_index(long long idx, long long n, int32_t* status) {
  return in_bounds(idx, n, status) ? idx : 0;
}

// A TwELL column byte read as a column of its 128-wide tile: in the checking
// build the byte as stored (its neuron's range is checked where it is used);
// in the normal build its low seven bits, so a TwELL left undefined (by a
// gate call whose wait ran out) can give wrong values downstream but never a
// neuron outside its tile.
__device__ __forceinline__ int tile_col(uint32_t byte) {
  return static_cast<int>(kBoundsCheck ? byte : (byte & 127u));
}

}  // namespace twell
