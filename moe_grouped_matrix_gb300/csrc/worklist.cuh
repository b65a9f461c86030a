// Device-side group metadata and tile worklist.
//
// The grouped matmul needs, for every group, the row range it owns: the
// exclusive prefix sum of group_sizes (page "tpu-inference 0.12.0.dev20251213
// -> 0.13.2.dev20251230", gmm.py, make_group_metadata: group_offsets as CSR
// row offsets).  Instead of the pages' tile-aligned visits (a tile straddling
// k groups visited k times and merged), every local group here is covered by
// its own BM-row tiles starting at the group's first row; the last tile of a
// group may run past its end and is masked at the store.  So no output tile is
// shared between groups and no read-modify-write merge is needed.
//
// One warp builds both tables in shared memory in the kernel prologue, from
// group_sizes in device memory, with no host round trip.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace gmmk {

// offs[0..G]: offs[0] = 0, offs[g+1] = min(offs[g] + max(sizes[g], 0), m).
// Flags negative sizes and sum(sizes) > m in *err (one report per launch:
// only CTA 0 writes).  Must be called by all 32 lanes of one warp.
__device__ __forceinline__ void build_group_offsets(const int32_t* __restrict__ sizes, int32_t groups, int32_t m,
                                                    int32_t* offs, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  long long carry = 0;
  bool negative = false;
  if (lane == 0) offs[0] = 0;
  for (int base = 0; base < groups; base += 32) {
    const int i = base + lane;
    int v = i < groups ? __ldg(sizes + i) : 0;
    negative |= v < 0;
    long long x = v > 0 ? v : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    const long long incl = carry + x;
    if (i < groups) offs[i + 1] = int32_t(incl < m ? incl : m);
    carry = __shfl_sync(0xffffffffu, incl, 31);
  }
  const bool any_negative = __any_sync(0xffffffffu, negative);
  if (lane == 0 && blockIdx.x == 0) {
    uint32_t flags = 0;
    if (any_negative) flags |= kErrNegativeSize;
    if (carry > m) flags |= kErrSizesExceedM;
    if (flags) atomicOr(err, flags);
  }
  __syncwarp();
}

// The first local group: the host value, or the device scalar when one is given
// (the pages pass group_offset as a device array).  Every thread reads the same
// value; an out-of-range device value records kErrGroupOffset and the caller
// returns before touching shared memory, barriers or TMEM, writing nothing.
__device__ __forceinline__ bool resolve_group_offset(const int32_t* dev, int32_t host, int32_t total, int32_t local,
                                                     uint32_t* err, int32_t& go) {
  go = host;
  if (dev == nullptr) return true;
  go = __ldg(dev);
  if (go >= 0 && go <= total - local) return true;
  if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, kErrGroupOffset);
  return false;
}

// tiles[0..L]: exclusive prefix sum over local groups l of ceil(rows_l / bm),
// rows_l = offs[first + l + 1] - offs[first + l].  All 32 lanes of one warp.
__device__ __forceinline__ void build_tile_prefix(const int32_t* offs, int32_t first, int32_t local, int32_t bm,
                                                  int32_t* tiles) {
  const int lane = threadIdx.x & 31;
  int32_t carry = 0;
  if (lane == 0) tiles[0] = 0;
  for (int base = 0; base < local; base += 32) {
    const int l = base + lane;
    int32_t t = 0;
    if (l < local) {
      const int32_t rows = offs[first + l + 1] - offs[first + l];
      t = (rows + bm - 1) / bm;
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, t, d);
      if (lane >= d) t += y;
    }
    if (l < local) tiles[l + 1] = carry + t;
    carry += __shfl_sync(0xffffffffu, t, 31);
  }
  __syncwarp();
}

// Largest l in [0, local) with tiles[l] <= mt, given tiles[0] = 0 <= mt < tiles[local].
// That group is never empty (an empty group has tiles[l] == tiles[l+1]).
__device__ __forceinline__ int32_t find_group(const int32_t* tiles, int32_t local, int32_t mt) {
  int32_t lo = 0, hi = local;
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (tiles[mid] <= mt)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// One output tile of the forward grouped matmul.
struct GemmTile {
  int32_t local_group;  // index into the local rhs slice
  int32_t row0;         // first row of the tile (group start + i * BM)
  int32_t row_end;      // one past the last row of the group
  int32_t n_tile;
};

// Work item w -> tile.  With raster > 0 items are ordered in super-columns of
// `raster` n-tiles: within a super-column, m-tiles (across all groups, in row
// order) are outer and its n-tiles inner, so CTAs running at the same time
// share the same few weight tiles and lhs row blocks in L2.  With raster < 0
// they go group by group, each group in blocks of up to -raster of its m-tiles,
// and within a block the n-tiles outer and the m-tiles inner: the CTAs running
// at the same time read each weight tile once between them, and the block's
// lhs rows stay in L2 while every weight tile of the group passes (each lhs
// row block is read once per block, not once per super-column).
__device__ __forceinline__ GemmTile decode_gemm_tile(int32_t w, int32_t m_tiles, int32_t n_tiles, int32_t raster,
                                                     const int32_t* tiles, const int32_t* offs, int32_t first,
                                                     int32_t local, int32_t bm) {
  if (raster < 0) {
    GemmTile t;
    t.local_group = find_group(tiles, local, int32_t(w / n_tiles));  // tiles[g] * n_tiles <= w
    const int32_t g0 = tiles[t.local_group], mt_g = tiles[t.local_group + 1] - g0;
    const int32_t r = w - g0 * n_tiles;                              // item within the group
    const int32_t blk = -raster;
    const int32_t b0 = (r / (blk * n_tiles)) * blk;                  // first m-tile of r's block
    const int32_t width = min(blk, mt_g - b0);
    const int32_t rb = r - b0 * n_tiles;
    t.n_tile = rb / width;
    const int32_t mt = g0 + b0 + (rb - t.n_tile * width);
    t.row0 = offs[first + t.local_group] + (mt - g0) * bm;
    t.row_end = offs[first + t.local_group + 1];
    return t;
  }
  const int64_t per_col = int64_t(m_tiles) * raster;
  const int32_t sc = int32_t(w / per_col);
  const int32_t n0 = sc * raster;
  const int32_t width = min(raster, n_tiles - n0);
  const int32_t r = int32_t(w - sc * per_col);
  const int32_t mt = r / width;
  GemmTile t;
  t.n_tile = n0 + (r - mt * width);
  t.local_group = find_group(tiles, local, mt);
  t.row0 = offs[first + t.local_group] + (mt - tiles[t.local_group]) * bm;
  t.row_end = offs[first + t.local_group + 1];
  return t;
}

}  // namespace gmmk
