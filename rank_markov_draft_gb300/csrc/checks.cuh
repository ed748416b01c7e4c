// checks.cuh -- range predicates of the optional on-chip offset checks.
//
// The debug library (built with DSPARK_DEVICE_CHECKS defined) checks, before
// each access, that a TMEM address lies in the region the access belongs to
// (the accumulators or the MMA's operand columns, and the lane quadrant its
// warp may reach) and that a shared-memory offset lies in its ring.  A failed
// check records DSPARK_ERR_DEVICE_OOB in the launch's status word and replaces
// the offset with the region's first one, so the access itself stays in
// bounds: nothing traps, the launch runs to its end, and the host reads the
// status.  The release library compiles every check away.
//
// The predicates are host-callable so that they can be tested without a GPU.
#pragma once

#include <cstdint>

namespace dspark {

#ifdef DSPARK_DEVICE_CHECKS
constexpr bool kDeviceChecks = true;
#else
constexpr bool kDeviceChecks = false;
#endif

// [off, off + len) lies inside [0, limit)
__host__ __device__ constexpr bool span_ok(uint32_t off, uint32_t len, uint32_t limit) {
  return len <= limit && off <= limit - len;
}

// A TMEM address relative to the allocation's base (lane << 16 | column): `width`
// columns from its column lie inside [col_lo, col_hi), and its lane is lane0, the
// first lane of the quadrant the accessing warp owns (for an MMA, lane 0).
__host__ __device__ constexpr bool tmem_span_ok(uint32_t rel, uint32_t width, uint32_t col_lo,
                                                uint32_t col_hi, uint32_t lane0) {
  return (rel >> 16) == lane0 && (rel & 0xFFFFu) >= col_lo && col_hi >= col_lo &&
         span_ok((rel & 0xFFFFu) - col_lo, width, col_hi - col_lo);
}

// The offset to use: `off` when the check passes, else the region's first offset.
__host__ __device__ constexpr uint32_t span_or_first(uint32_t off, uint32_t len, uint32_t limit) {
  return span_ok(off, len, limit) ? off : 0u;
}

__host__ __device__ constexpr uint32_t tmem_or_first(uint32_t rel, uint32_t width, uint32_t col_lo,
                                                     uint32_t col_hi, uint32_t lane0) {
  return tmem_span_ok(rel, width, col_lo, col_hi, lane0) ? rel : ((lane0 << 16) | col_lo);
}

}  // namespace dspark
