// checks.cuh -- the bounds-checked build of the library.
//
// Compiled with -DRA_CHECKS=1 (libringattn_checked.so), every global-memory
// index in the epilogues, the merge, preprocess, decode and float32 kernels,
// and every TMA box coordinate, is checked against the extent of the tensor
// it addresses before the access.  A failed check skips the access and is
// recorded in the per-device CheckRec (count, first site, index and extent);
// a skipped TMA copy leaves its barrier incomplete, so the waiting roles time
// out within their bound and the call reports RA_ERR_TIMEOUT as well.  The
// checked build also counts kernel events that tests want to see happen (the
// forward's O rescale).  In the default build (RA_CHECKS undefined or 0) the
// macros below compile to nothing and the kernels are unchanged.
#pragma once
#include <cstdint>

#ifndef RA_CHECKS
#define RA_CHECKS 0
#endif

namespace ra {

// One per device, in device memory (host.cu).  Layout mirrors ra_check_report.
struct CheckRec {
  unsigned long long events[8];
  unsigned int violations;
  unsigned int first_site;
  long long first_index;
  long long first_extent;
};

// Event counters (CheckRec::events).
enum : int {
  EV_FWD_RESCALE_ROWS = 0,   // bf16 forward: rows whose running max jumped past the threshold after
                             // keys were folded in (O rescaled for that row)
  EV_FWD_RESCALE_WARPS = 1,  // bf16 forward: rescale passes over O in TMEM (one per warp and tile)
  EV_TMA_BOXES = 2,          // TMA boxes whose coordinates were checked (all kernels)
  EV_CHECKED = 3,            // other checked global accesses
};

// Check sites (CheckRec::first_site): kernel in the high byte, access below.
enum : unsigned int {
  SITE_FWD_TMA_Q = 0x101, SITE_FWD_TMA_K, SITE_FWD_TMA_V, SITE_FWD_O, SITE_FWD_LSE, SITE_FWD_FOLD,
  SITE_F32_Q = 0x201, SITE_F32_KV, SITE_F32_O, SITE_F32_LSE,
  SITE_PREP_IN = 0x301, SITE_PREP_LSE, SITE_PREP_OUT,
  SITE_DKV_TMA_Q = 0x401, SITE_DKV_TMA_DO, SITE_DKV_TMA_KV, SITE_DKV_VEC, SITE_DKV_OUT,
  SITE_DQ_TMA_K = 0x501, SITE_DQ_TMA_V, SITE_DQ_TMA_DO, SITE_DQ_Q, SITE_DQ_VEC, SITE_DQ_OUT,
  SITE_MERGE_LSE = 0x601, SITE_MERGE_O,
  SITE_DEC_KV = 0x701, SITE_DEC_Q, SITE_DEC_PART, SITE_DEC_OUT,
  SITE_FFN_TMA = 0x801, SITE_FFN_OUT,
};

#if RA_CHECKS
__device__ __forceinline__ void check_fail(CheckRec* r, unsigned int site, long long idx, long long extent) {
  if (atomicAdd(&r->violations, 1u) == 0u) {
    r->first_site = site;
    r->first_index = idx;
    r->first_extent = extent;
  }
}
// [idx, idx + width) inside [0, extent)?
__device__ __forceinline__ bool check_range(CheckRec* r, unsigned int site, long long idx, long long width,
                                            long long extent) {
  atomicAdd(&r->events[EV_CHECKED], 1ull);
  if (idx >= 0 && width >= 0 && idx + width <= extent) return true;
  check_fail(r, site, idx, extent);
  return false;
}
// A TMA load box's start coordinates (x innermost): x inside the row and on
// the 16-byte boundary the copy requires (x_align elements), z inside the
// tensor, and y below `ny`.  A load may start past the last row (the hardware
// fills the box with zeros there), so callers pass as `ny` the exclusive bound
// their schedule guarantees: S for tiles that start inside a block, S plus the
// rows by which a unit's later query tiles (or the upper half of a KV tile)
// may start past it.
__device__ __forceinline__ bool check_box(CheckRec* r, unsigned int site, int x, int y, int z, long long nx,
                                          long long ny, long long nz, int x_align) {
  atomicAdd(&r->events[EV_TMA_BOXES], 1ull);
  if (x >= 0 && x < nx && x % x_align == 0 && y >= 0 && y < ny && z >= 0 && z < nz) return true;
  check_fail(r, site, (static_cast<long long>(z) << 40) | (static_cast<long long>(y) << 16) | x, ny);
  return false;
}
#define RA_CHECK_RANGE(rec, site, idx, width, extent) \
  ::ra::check_range((rec), (site), static_cast<long long>(idx), static_cast<long long>(width), \
                    static_cast<long long>(extent))
#define RA_CHECK_BOX(rec, site, x, y, z, nx, ny, nz, xa) \
  ::ra::check_box((rec), (site), (x), (y), (z), static_cast<long long>(nx), static_cast<long long>(ny), \
                  static_cast<long long>(nz), (xa))
#define RA_COUNT(rec, ev, n) atomicAdd(&(rec)->events[(ev)], static_cast<unsigned long long>(n))
#else
#define RA_CHECK_RANGE(rec, site, idx, width, extent) true
#define RA_CHECK_BOX(rec, site, x, y, z, nx, ny, nz, xa) true
#define RA_COUNT(rec, ev, n) ((void)0)
#endif

}  // namespace ra
