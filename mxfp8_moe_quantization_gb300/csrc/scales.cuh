// Destinations of MXFP8 scale bytes: row-major, the 128x4 tile layout of one
// matrix per batch, or the 128x4 layout with per-group padding of rows
// (GROUP_ROWS) or of 32-element column blocks (GROUP_COLS), as the block-scaled
// tcgen05 MMA reads them ("Accelerating Llama4 Scout training with TorchAO
// MXFP8 MoE primitives": scale factors in the 128x4 layout, grouped by the
// offsets).  Shared by the quantization kernels (internal).
#pragma once
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace fp8moe {

// Grouped layouts need, per group, its end and its padded start: built per
// CTA in shared memory with a block-wide scan of the offsets (which are also
// validated).
constexpr int QG_MAX = 1024;

struct ScaleSpec {
  uint8_t* p;
  int layout;      // FP8MOE_SCALES_ROWMAJOR, FP8MOE_NO_GROUPS, FP8MOE_GROUP_ROWS / _COLS
  int64_t Rp, Cp;  // padded geometry of one (batch's) swizzled matrix
  const int32_t* offs;
  int E;
};

struct GroupTable {
  int64_t end[QG_MAX];
  int64_t pad[QG_MAX];
  int bad;
};

FP8MOE_DEV int64_t tile_off(int64_t r, int64_t c, int64_t Cp) {
  return ((r >> 7) * (Cp >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// first group whose end is > key
FP8MOE_DEV int find_group(const int64_t* ends, int E, int64_t key) {
  int lo = 0, hi = E - 1, g = E - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (ends[mid] > key) {
      g = mid;
      hi = mid - 1;
    } else {
      lo = mid + 1;
    }
  }
  return g;
}

// What pad[] accumulates over the earlier groups:
//   GT_ROWS128: group sizes rounded up to 128 rows (scale tiles of the rows);
//   GT_COLS:    group sizes / 32 rounded up to 4 (scale tile columns; every
//               group size must be a multiple of 32);
//   GT_SUB32:   group sizes in 32-row sub-tiles, ceil(size / 32);
//   GT_BLK128:  group sizes in 128-row blocks, ceil(size / 128) (every group
//               size must be a multiple of 32).
enum { GT_ROWS128 = 0, GT_COLS = 1, GT_SUB32 = 2, GT_BLK128 = 3 };

// Call with all threads of a block of at least 256 (a multiple of 32, at most
// 1024); the groups are spread over the first 256 threads.  Ends with
// __syncthreads.
static __device__ void build_group_table(GroupTable& t, const int32_t* offs, int E, int64_t total, int mode,
                                  int* status) {
  __shared__ int64_t wsum[32];   // per warp (warps past the eighth hold no groups)
  const int tid = threadIdx.x;
  const int per = (E + 255) / 256;  // <= 4
  int64_t u[4] = {0, 0, 0, 0};
  int64_t sum = 0;
  int bad = 0;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e >= E) break;
    const int64_t end = offs[e];
    const int64_t start = e == 0 ? 0 : offs[e - 1];
    if (end < start || end > total || (e == E - 1 && end != total)) bad = 1;
    if ((mode == GT_COLS || mode == GT_BLK128) && (end % 32)) bad = 1;
    const int64_t sz = end - start;
    u[i] = mode == GT_COLS     ? ((sz / 32 + 3) / 4 * 4)
           : mode == GT_SUB32  ? (sz + 31) / 32
           : mode == GT_BLK128 ? (sz + 127) / 128
                               : ((sz + 127) / 128 * 128);
    sum += u[i];
    t.end[e] = end;
  }
  // block exclusive scan of the per-thread sums
  const int lane = tid & 31, warp = tid >> 5;
  int64_t incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  bad = __syncthreads_or(bad);
  int64_t base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  int64_t run = base + incl - sum;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e >= E) break;
    t.pad[e] = run;
    run += u[i];
  }
  if (tid == 0) {
    t.bad = bad;
    if (bad) set_status(status, FP8MOE_ERR_DEVICE_OFFSETS);
  }
  __syncthreads();
}

// Byte offset of scale (row, col) of batch b.  For GROUP_ROWS the row is an
// element row of x (grouped over R); for GROUP_COLS the column is a 32-block
// index along the grouped contracting dimension.
FP8MOE_DEV int64_t scale_offset(const ScaleSpec& s, const GroupTable* gt, int64_t b, int64_t row, int64_t col,
                                int64_t rows_per_batch, int64_t cols) {
  if (s.layout == FP8MOE_SCALES_ROWMAJOR) return (b * rows_per_batch + row) * cols + col;
  if (s.layout == FP8MOE_NO_GROUPS) return b * s.Rp * s.Cp + tile_off(row, col, s.Cp);
  if (s.layout == FP8MOE_GROUP_ROWS) {
    const int g = find_group(gt->end, s.E, row);
    const int64_t gs = g == 0 ? 0 : gt->end[g - 1];
    return tile_off(gt->pad[g] + (row - gs), col, s.Cp);
  }
  const int g = find_group(gt->end, s.E, col * 32);
  const int64_t gs = g == 0 ? 0 : gt->end[g - 1];
  return tile_off(row, gt->pad[g] + (col - gs / 32), s.Cp);
}

static inline ScaleSpec make_spec(uint8_t* p, int layout, int64_t R, int64_t Cs, const int32_t* offs, int64_t E) {
  ScaleSpec o;
  o.p = p;
  o.layout = layout;
  const bool grouped = layout == FP8MOE_GROUP_ROWS || layout == FP8MOE_GROUP_COLS;
  const SwizzleGeom g = swizzle_geom(R, Cs, grouped ? E : 0, grouped ? layout : FP8MOE_NO_GROUPS);
  o.Rp = g.Rp;
  o.Cp = g.Cp;
  o.offs = offs;
  o.E = (int)E;
  return o;
}

}  // namespace fp8moe
