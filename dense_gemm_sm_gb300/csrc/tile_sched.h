// tile_sched.h -- tile raster and stream-K partition shared by the host planner and the kernels.
//
// Raster: the output of each problem is cut into tiles_m x tiles_n tiles; one linear
// tile id t (batch-major) is mapped to (b, tm, tn).  Within a batch, tiles are visited
// in groups of `group` tile rows: inside a group the walk goes down the group's rows
// for one tile column, then to the next column (serpentine: odd columns walk upward),
// and successive groups sweep the columns in alternating directions.  Consecutive
// ids therefore touch few distinct A row-tiles and B column-tiles, the L2 reuse
// argument of the MUSA lesson m11-l5 "Block ID Swizzle" discussion (every 8 blocks
// change row: 64 blocks need only 8 + 8 operand tiles, an 8x amplification) and the
// "fuse the 2-D tile grid into one linear index" transform of "Operator & Runtime"
// section 5.4.2.  The walk is a bijection on [0, batch*tiles_m*tiles_n).
//
// Stream-K: the thin (decode-shaped) path flattens (output tile, K block) pairs into
// U = tiles * kblocks units and gives CTA c the contiguous range
// [floor(c*U/G), floor((c+1)*U/G)).  A tile split across CTAs is finished by the
// last CTA to arrive, which sums the partial results in CTA (= K) order, so the
// result does not depend on arrival order ("Operator & Runtime" section 5.2.4:
// split-K needs a combine step; a fixed combination order is deterministic).
#pragma once
#include <cstdint>

#if defined(__CUDACC__)
#define DG_HD __host__ __device__ __forceinline__
#else
#define DG_HD inline
#endif

namespace dg {

DG_HD void raster_tile(int64_t t, int64_t tiles_m, int64_t tiles_n, int32_t group, int64_t* b,
                       int64_t* tm, int64_t* tn) {
  const int64_t per_batch = tiles_m * tiles_n;
  const int64_t bb = t / per_batch;
  const int64_t r = t - bb * per_batch;
  const int64_t G = group < 1 ? 1 : group;
  const int64_t gsize = G * tiles_n;
  const int64_t g = r / gsize;
  const int64_t first = g * G;
  const int64_t rows = (tiles_m - first) < G ? (tiles_m - first) : G;
  const int64_t local = r - g * gsize;
  int64_t n = local / rows;
  int64_t ml = local - n * rows;
  if (n & 1) ml = rows - 1 - ml;
  if (g & 1) n = tiles_n - 1 - n;
  *b = bb;
  *tm = first + ml;
  *tn = n;
}

// The stream-K helpers are written for an index type T: int64_t in general, uint32_t when
// units * ctas < 2^32 (the kernels pick it at launch), where the divisions are 32-bit.

// First unit of CTA c's stream-K range.
template <typename T>
DG_HD T sk_start(T c, T units, T ctas) { return c * units / ctas; }

// The CTA whose range contains unit x (the largest c with sk_start(c) <= x).
template <typename T>
DG_HD T sk_cta_of(T x, T units, T ctas) { return ((x + 1) * ctas - 1) / units; }

// Number of CTAs that contribute to output tile `tile` (kblocks units per tile).
template <typename T>
DG_HD T sk_contributors(T tile, T kblocks, T units, T ctas) {
  return sk_cta_of<T>((tile + 1) * kblocks - 1, units, ctas) - sk_cta_of<T>(tile * kblocks, units, ctas) +
         1;
}

// Partial-result slot used by CTA c for tile `tile`: 0 when c's range starts inside the
// tile (its first segment), 1 when the range began in an earlier tile (its last segment).
template <typename T>
DG_HD int sk_slot(T c, T tile, T kblocks, T units, T ctas) {
  return sk_start<T>(c, units, ctas) >= tile * kblocks ? 0 : 1;
}

// True when the 32-bit helpers are exact for this partition.
inline bool sk_fits_u32(int64_t units, int64_t ctas) {
  return units > 0 && ctas > 0 && (units + 1) * (ctas + 1) < (int64_t(1) << 32);
}

}  // namespace dg
