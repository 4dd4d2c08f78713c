// bounds.cuh — index checks of the debug build (-DVSF_DEBUG_BOUNDS).
//
// Every kernel that indexes a packed buffer receives the buffer's extent (the
// elements of the plan's rank window) and the plan's device error word. In a
// debug build each range a kernel is about to touch (a tensor segment, a ring
// chunk, a quantisation block, an 8-element group, a matrix) is checked
// first: a range outside [0, limit) sets bit 4 of the error word and the
// access is skipped, so no stray access is ever made and no trap is raised.
// In a normal build the check is a constant and compiles away.
#pragma once

#include <cstdint>

namespace vsf {

struct Bounds {
  int64_t limit;  // elements of every packed buffer
  unsigned* err;  // the plan's device error word
};

constexpr unsigned kErrBounds = 4u;  // error-word bit of a failed index check

#ifdef VSF_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(const Bounds& bd, int64_t first, int64_t last) {
  if (first >= 0 && first <= last && last <= bd.limit) return true;
  atomicOr(bd.err, kErrBounds);
  return false;
}
#else
__device__ __forceinline__ bool in_bounds(const Bounds&, int64_t, int64_t) { return true; }
#endif

}  // namespace vsf
