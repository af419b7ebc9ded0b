// 128x4 tiled layout of e8m0 scale factors for tcgen05 block-scaled MMA.
//
// "Accelerating Llama4 Scout training with TorchAO MXFP8 MoE primitives",
// section details and the caption of its 128x4 tile layout table: a dedicated
// kernel rearranges row-major scale factors into 128x4 tiles.  The byte order
// inside a tile is the one tcgen05 consumes: 512 bytes per tile, element
// (r, c) at (r % 32) * 16 + (r / 32) * 4 + c, i.e. 32 rows of 16 bytes, each
// holding rows r, r+32, r+64, r+96 -- one 16-byte row per TMEM lane.
//
// The kernel is output-driven: each thread produces one 16-byte row of a tile
// (so every output byte, padding included, is written exactly once and the
// stores are contiguous) and gathers its 16 source bytes.  Group boundaries
// come from device offsets: each group starts a new 128-row block (rows) or
// 4-column block (columns).
#include "common.cuh"
#include "launch.h"

namespace fp8moe {

SwizzleGeom swizzle_geom(int64_t R, int64_t Cs, int64_t E, int group_axis) {
  int64_t rb = (R + 127) / 128, cb = (Cs + 3) / 4;
  if (group_axis == FP8MOE_GROUP_ROWS) rb += E;
  if (group_axis == FP8MOE_GROUP_COLS) cb += E;
  return SwizzleGeom{rb * 128, cb * 4};
}

constexpr int SWZ_MAX_GROUPS = 1024;

struct SwizzleArgs {
  const uint8_t* s;
  int64_t B, R, Cs;
  const int32_t* offs;
  int E;
  int group_axis;
  int64_t Rp, Cp;
  uint8_t* out;
  int* status;
};

__global__ void __launch_bounds__(256) k_swizzle(SwizzleArgs a) {
  // padded start / real start / size of each group, in rows (GROUP_ROWS) or
  // scale columns (GROUP_COLS)
  __shared__ int64_t gp[SWZ_MAX_GROUPS + 1];
  __shared__ int64_t gs[SWZ_MAX_GROUPS];
  __shared__ int64_t gz[SWZ_MAX_GROUPS];
  __shared__ int bad;
  const bool grouped = a.group_axis != FP8MOE_NO_GROUPS;
  if (grouped) {
    if (threadIdx.x == 0) {
      const int unit = a.group_axis == FP8MOE_GROUP_ROWS ? 128 : 4;
      const int64_t total = a.group_axis == FP8MOE_GROUP_ROWS ? a.R : a.Cs * 32;
      int64_t p = 0, prev = 0;
      int b = 0;
      for (int e = 0; e < a.E; ++e) {
        int64_t end = a.offs[e];
        if (end < prev || end > total) b = 1;
        if (a.group_axis == FP8MOE_GROUP_COLS) {
          if (end % 32) b = 1;
        }
        const int64_t sz_el = end - prev;
        const int64_t sz = a.group_axis == FP8MOE_GROUP_COLS ? sz_el / 32 : sz_el;
        gp[e] = p;
        gs[e] = a.group_axis == FP8MOE_GROUP_COLS ? prev / 32 : prev;
        gz[e] = sz;
        p += (sz + unit - 1) / unit * unit;
        prev = end;
      }
      if (prev != total) b = 1;
      gp[a.E] = p;
      bad = b;
      if (b) set_status(a.status, FP8MOE_ERR_DEVICE_OFFSETS);
    }
    __syncthreads();
  }
  const int64_t per_batch = a.Rp * a.Cp / 16;
  const int64_t total = a.B * per_batch;
  const int64_t tiles_per_rb = a.Cp / 4;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total;
       k += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = k / per_batch;
    const int64_t kk = k % per_batch;
    const int64_t tile = kk / 32;
    const int r32 = (int)(kk % 32);
    const int64_t rbk = tile / tiles_per_rb, cbk = tile % tiles_per_rb;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t prow = rbk * 128 + q * 32 + r32;
      uint32_t word = 0;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int64_t pcol = cbk * 4 + c4;
        int64_t r = -1, c = -1;
        if (!grouped) {
          r = prow;
          c = pcol;
        } else if (!bad) {
          const int64_t key = a.group_axis == FP8MOE_GROUP_ROWS ? prow : pcol;
          // last group whose padded start is <= key (skips empty groups)
          int lo = 0, hi = a.E - 1, g = -1;
          while (lo <= hi) {
            const int mid = (lo + hi) >> 1;
            if (gp[mid] <= key) {
              g = mid;
              lo = mid + 1;
            } else {
              hi = mid - 1;
            }
          }
          if (g >= 0) {
            const int64_t within = key - gp[g];
            if (within < gz[g]) {
              if (a.group_axis == FP8MOE_GROUP_ROWS) {
                r = gs[g] + within;
                c = pcol;
              } else {
                r = prow;
                c = gs[g] + within;
              }
            }
          }
        }
        uint32_t v = 0;
        if (r >= 0 && r < a.R && c >= 0 && c < a.Cs) v = a.s[(b * a.R + r) * a.Cs + c];
        word |= v << (8 * c4);
      }
      w[q] = word;
    }
    reinterpret_cast<uint4*>(a.out + b * a.Rp * a.Cp)[kk] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_swizzle(const uint8_t* s, int64_t B, int64_t R, int64_t Cs, const int32_t* offs,
                           int64_t E, int group_axis, uint8_t* out, int* status, int num_sms,
                           cudaStream_t st) {
  SwizzleArgs a;
  const SwizzleGeom g = swizzle_geom(R, Cs, group_axis == FP8MOE_NO_GROUPS ? 0 : E, group_axis);
  a.s = s;
  a.B = B;
  a.R = R;
  a.Cs = Cs;
  a.offs = offs;
  a.E = (int)E;
  a.group_axis = group_axis;
  a.Rp = g.Rp;
  a.Cp = g.Cp;
  a.out = out;
  a.status = status;
  const int64_t total = B * g.Rp * g.Cp / 16;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  k_swizzle<<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fp8moe
