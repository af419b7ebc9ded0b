// MXFP8 quantization of one bf16 tensor in both directions from a single read
// of it: dim0 (blocks of 32 along a row, codes [B, R, C]) and dim1 (blocks of
// 32 down a column, codes transposed to [B, C, R]), each with its e8m0 scales
// written straight into their final layout.  This is the operand preparation
// of the MXFP8 MoE layer ("Accelerating Llama4 Scout training with TorchAO
// MXFP8 MoE primitives": a tensor is quantized along both dimensions for the
// forward and the two backward GEMMs); doing both from one read moves 4 bytes
// per element instead of the 6 of two separate passes.
//
// Layout of the work (no shared-memory staging): a warp owns a band of up to
// 128 rows x 128 columns and sweeps it in 32-row sub-tiles, so that every
// 128-byte line of the transposed codes and of the scales is completed by one
// warp within a short time (while it is still in L2); small tensors use lower
// bands so that every warp gets work.  In a sub-tile, lane l
// holds rows 16*(l/16) .. +15 of the 8 columns 8*(l%16) .. +7 in registers
// (16 loads of 16 bytes, each warp load covering two 256-byte row segments).
//   dim0: the 32-element block of a row spans 4 lanes: two shuffles give its
//         absolute maximum; each lane encodes and stores its 8 codes, so a
//         warp store writes two 128-byte row segments.
//   dim1: a lane has 16 rows of each of its columns; one shuffle with the
//         lane holding the other 16 rows gives the column block's maximum;
//         each lane stores 16 codes per column, the two halves of a column's
//         32-byte output segment coming from the two lanes.
#include <stdlib.h>

#include "common.cuh"
#include "launch.h"
#include "mxcvt.cuh"
#include "scales.cuh"

namespace fp8moe {

namespace {

FP8MOE_DEV uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

struct DualArgs {
  const uint16_t* x;    // [B, R, C] bf16
  int64_t B, R, C;
  uint32_t n_ct, n_band, tiles;  // 128 columns x bands of `nsub` 32-row sub-tiles
  uint32_t n_rt;
  int nsub;
  uint8_t* q0;          // [B, R, C]
  uint8_t* q1;          // [B, C, R]
  ScaleSpec s0;         // [B, R, C/32] in its layout
  ScaleSpec s1;         // [B, C, R/32] in its layout
  int* status;
};

constexpr uint32_t FULL = 0xffffffffu;

// scale offsets off the fast paths (kept out of line: the unrolled loops
// would otherwise carry many copies)
__device__ __noinline__ int64_t s0_offset_slow(const ScaleSpec& s, const GroupTable* gt, int64_t b, int64_t row,
                                               int64_t col, int64_t R, int64_t cols) {
  return scale_offset(s, gt, b, row, col, R, cols);
}
__device__ __noinline__ int64_t s1_offset_slow(const ScaleSpec& s, const GroupTable* gt, int64_t b, int64_t row,
                                               int64_t col, int64_t R, int64_t cols) {
  return scale_offset(s, gt, b, row, col, R, cols);
}

// dim1 of the column pair held in word K of this lane's 16 rows: 16 codes per
// column (this half's rows); the two scale bytes are returned
template <int K>
FP8MOE_DEV void dim1_pair(const uint4 (&v)[16], uint32_t mw, bool ok, uint8_t* q1c, int64_t R, uint32_t& b_lo,
                          uint32_t& b_hi) {
  // exponent fields of the two column maxima (sign bits are clear)
  const uint32_t efl = max((mw >> 7) & 0xFFu, 8u), efh = max(mw >> 23, 8u);
  const uint32_t blo = efl - 8u, bhi = efh - 8u;
  const uint32_t p2 = ((262u - efl) << 7) | ((262u - efh) << 23);
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4& w = v[4 * k + i];
      y[i] = mul_bf16x2(K == 0 ? w.x : (K == 1 ? w.y : (K == 2 ? w.z : w.w)), p2);
    }
    lo[k] = cvt4(lo_f32(y[0]), lo_f32(y[1]), lo_f32(y[2]), lo_f32(y[3]));
    hi[k] = cvt4(hi_f32(y[0]), hi_f32(y[1]), hi_f32(y[2]), hi_f32(y[3]));
  }
  if (ok) {
    *reinterpret_cast<uint4*>(q1c + (2 * K) * R) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(q1c + (2 * K + 1) * R) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  }
  b_lo = blo;
  b_hi = bhi;
}

// D0 / D1: produce the dim0 / dim1 direction (the dim1-only instance serves
// the standalone transposed quantization)
template <bool D0, bool D1>
__global__ void __launch_bounds__(256, 2) k_mx_dual(DualArgs a) {
  __shared__ GroupTable gt0, gt1;
  if (D0 && a.s0.layout == FP8MOE_GROUP_ROWS) {
    build_group_table(gt0, a.s0.offs, a.s0.E, a.R, GT_ROWS128, a.status);
    if (gt0.bad) return;
  }
  if (D1 && a.s1.layout == FP8MOE_GROUP_COLS) {
    build_group_table(gt1, a.s1.offs, a.s1.E, a.R, GT_COLS, a.status);
    if (gt1.bad) return;
  }
  const int lane = threadIdx.x & 31, half = lane >> 4, cl = lane & 15;
  const uint32_t nwarps = gridDim.x * (blockDim.x >> 5);
  // Grouped layouts (B == 1): a warp's tiles come in increasing row order and
  // every 32-row sub-tile lies inside one routing group (offsets are
  // multiples of 32), so a forward-only cursor per table replaces the
  // binary searches: the group of row r is the first whose end exceeds r.
  int g0c = 0, g1c = 0;
  auto advance = [](const GroupTable& gt, int E, int& g, int64_t r) {
    while (g < E - 1 && gt.end[g] <= r) ++g;
  };
  for (uint32_t t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < a.tiles; t += nwarps) {
    const uint32_t ct = t % a.n_ct;
    const uint32_t rest = t / a.n_ct;
    const uint32_t rt0 = (rest % a.n_band) * a.nsub;
    const int64_t b = rest / a.n_band;
    // dim1 scale bytes of this lane's 8 columns over the band's row blocks
    // (byte `sub` of each word): the row blocks of a band are consecutive
    // scale bytes of a column in every layout, written as one word per column
    uint32_t sacc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int sub = 0; sub < a.nsub && rt0 + sub < a.n_rt; ++sub) {
      const int64_t rt = rt0 + sub;
      const int64_t r = rt * 32 + half * 16;   // first of this lane's 16 rows
      const int64_t c = (int64_t)ct * 128 + cl * 8;   // first of this lane's 8 columns
      const bool ok = c < a.C;                 // C % 32 == 0: whole 4-lane groups are in or out
      const uint16_t* xp = a.x + (b * a.R + r) * a.C + c;
      uint4 v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = ok ? ld_nc16(xp + i * a.C) : make_uint4(0, 0, 0, 0);

      if (D0) {
      // ---- dim0: blocks of 32 along each row (4 lanes x 8 columns).
      // Scale byte of row r + i: rows r .. r + 15 share a 32-row group of the
      // 128x4 layout (offset step 16) or are consecutive rows (step C/32) --
      // unless a routing group ends inside them (grouped layout only).
      int64_t s0_base = 0, s0_step = 0;
      if (a.s0.layout == FP8MOE_GROUP_ROWS) {
        // the cursor follows the sub-tile's first row; this half's group is
        // at most a few steps further.  When rows r .. r + 15 lie in one
        // routing group and start a 16-row half of the layout's 32-row group
        // (always, for 32-multiple groups) their offsets step by 16; else
        // each row's offset is computed on its own
        advance(gt0, a.s0.E, g0c, rt * 32);
        int g = g0c;
        advance(gt0, a.s0.E, g, r);
        const int64_t gs = g == 0 ? 0 : gt0.end[g - 1];
        if (gt0.end[g] >= r + 16 && ((r - gs) & 15) == 0) {
          s0_base = tile_off(gt0.pad[g] + (r - gs), c >> 5, a.s0.Cp);
          s0_step = 16;
        }
      } else if ((cl & 3) == 0 && ok) {
        s0_base = scale_offset(a.s0, &gt0, b, r, c >> 5, a.R, a.C >> 5);
        s0_step = a.s0.layout == FP8MOE_SCALES_ROWMAJOR ? (a.C >> 5) : 16;
      }
      uint8_t* q0p = a.q0 + (b * a.R + r) * a.C + c;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        uint32_t m2 = max_u16x2(max_u16x2(v[i].x & 0x7FFF7FFFu, v[i].y & 0x7FFF7FFFu),
                                max_u16x2(v[i].z & 0x7FFF7FFFu, v[i].w & 0x7FFF7FFFu));
        m2 = max_u16x2(m2, __byte_perm(m2, 0, 0x1032));   // both halves: the chunk's maximum
        m2 = max_u16x2(m2, __shfl_xor_sync(FULL, m2, 1));
        m2 = max_u16x2(m2, __shfl_xor_sync(FULL, m2, 2));
        const uint32_t ef = max((m2 >> 7) & 0xFFu, 8u);   // exponent field of the block maximum
        const uint32_t byte = ef - 8u;
        const uint32_t p2 = (262u - ef) * 0x00800080u;    // 2^-e in both bf16 halves
        if (ok) {
          *reinterpret_cast<uint2*>(q0p + i * a.C) = enc_row8(v[i], p2);
          if ((cl & 3) == 0) {
            const int64_t off =
                s0_step ? s0_base + i * s0_step : s0_offset_slow(a.s0, &gt0, b, r + i, c >> 5, a.R, a.C >> 5);
            a.s0.p[off] = (uint8_t)byte;
          }
        }
      }

      }
      if (D1) {
      // ---- dim1: blocks of 32 down each column (16 rows here + 16 in lane ^ 16)
      uint32_t mw[4] = {0, 0, 0, 0};   // column pairs (2k, 2k+1) as packed 16-bit maxima
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        mw[0] = max_u16x2(mw[0], v[i].x & 0x7FFF7FFFu);
        mw[1] = max_u16x2(mw[1], v[i].y & 0x7FFF7FFFu);
        mw[2] = max_u16x2(mw[2], v[i].z & 0x7FFF7FFFu);
        mw[3] = max_u16x2(mw[3], v[i].w & 0x7FFF7FFFu);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) mw[k] = max_u16x2(mw[k], __shfl_xor_sync(FULL, mw[k], 16));
      // q1[b][c + j][r .. r + 15]
      uint8_t* q1c = a.q1 + (b * a.C + c) * a.R + r;
      uint32_t bl, bh;
      dim1_pair<0>(v, mw[0], ok, q1c, a.R, bl, bh);
      sacc[0] |= bl << (8 * sub);
      sacc[1] |= bh << (8 * sub);
      dim1_pair<1>(v, mw[1], ok, q1c, a.R, bl, bh);
      sacc[2] |= bl << (8 * sub);
      sacc[3] |= bh << (8 * sub);
      dim1_pair<2>(v, mw[2], ok, q1c, a.R, bl, bh);
      sacc[4] |= bl << (8 * sub);
      sacc[5] |= bh << (8 * sub);
      dim1_pair<3>(v, mw[3], ok, q1c, a.R, bl, bh);
      sacc[6] |= bl << (8 * sub);
      sacc[7] |= bh << (8 * sub);
      }
    }
    if (D1) {
      // dim1 scales of the band: columns c .. c + 7 share a 32-row group of
      // the 128x4 layout (step 16) or are consecutive rows of the row-major
      // [C, R/32] scales (step R/32)
      const int64_t c = (int64_t)ct * 128 + cl * 8;
      const int nv = (int)min((uint32_t)a.nsub, a.n_rt - rt0);
      const bool gcols = a.s1.layout == FP8MOE_GROUP_COLS;
      if (gcols) advance(gt1, a.s1.E, g1c, (int64_t)rt0 * 32);
      if (half == 0 && c < a.C) {
        int64_t base;
        if (gcols) {
          const int64_t gs = g1c == 0 ? 0 : gt1.end[g1c - 1];
          base = tile_off(c, gt1.pad[g1c] + (rt0 - gs / 32), a.s1.Cp);
        } else {
          base = scale_offset(a.s1, &gt1, b, c, rt0, a.C, a.R >> 5);
        }
        const bool rowmajor = a.s1.layout == FP8MOE_SCALES_ROWMAJOR;
        const int64_t st1 = rowmajor ? (a.R >> 5) : 16;
        // the band's row blocks are consecutive scale bytes of each column:
        // always in row-major; in a 128x4 tile while they stay inside one
        // 4-column group of it (and, grouped, inside one routing group)
        bool contiguous = rowmajor || (base & 3) + nv <= 4;
        if (contiguous && gcols && nv > 1) contiguous = gt1.end[g1c] >= (int64_t)(rt0 + nv) * 32;
        uint8_t* p0 = a.s1.p + base;
        if (contiguous && nv == 4 && ((uintptr_t)p0 & 3) == 0 && (st1 & 3) == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j) *reinterpret_cast<uint32_t*>(p0 + j * st1) = sacc[j];
        } else if (contiguous && nv == 2 && ((uintptr_t)p0 & 1) == 0 && (st1 & 1) == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j) *reinterpret_cast<uint16_t*>(p0 + j * st1) = (uint16_t)sacc[j];
        } else if (contiguous) {
          for (int j = 0; j < 8; ++j)
            for (int sb = 0; sb < nv; ++sb) p0[j * st1 + sb] = (uint8_t)(sacc[j] >> (8 * sb));
        } else {
          // one offset per row block; the 8 columns step by st1 from it
          for (int sb = 0; sb < nv; ++sb) {
            uint8_t* pb = a.s1.p + s1_offset_slow(a.s1, &gt1, b, c, rt0 + sb, a.C, a.R >> 5);
#pragma unroll
            for (int j = 0; j < 8; ++j) pb[j * st1] = (uint8_t)(sacc[j] >> (8 * sb));
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_mx_dual(const void* x, int64_t B, int64_t R, int64_t C, void* q0, uint8_t* s0, int s0_layout,
                           void* q1, uint8_t* s1, int s1_layout, const int32_t* offs, int64_t E, int num_sms,
                           int* status, cudaStream_t st) {
  if (!q1) return cudaErrorInvalidValue;
  if (B == 0 || R == 0 || C == 0) return cudaSuccess;
  DualArgs a;
  a.x = (const uint16_t*)x;
  a.B = B;
  a.R = R;
  a.C = C;
  a.n_ct = (uint32_t)((C + 127) / 128);
  a.n_rt = (uint32_t)(R / 32);
  // bands of 4 sub-tiles when that leaves several bands per warp, else lower
  const int64_t warps = (int64_t)num_sms * 2 * 8;
  a.nsub = 4;
  while (a.nsub > 1 && (int64_t)a.n_ct * ((a.n_rt + a.nsub - 1) / a.nsub) * B < 4 * warps) a.nsub >>= 1;
  // FP8MOE_DUAL_BAND=1|2|4 fixes the band height (tests use it to cover every
  // band shape on small inputs)
  static const int force_band = [] {
    const char* v = getenv("FP8MOE_DUAL_BAND");
    const int n = v ? atoi(v) : 0;
    return (n == 1 || n == 2 || n == 4) ? n : 0;
  }();
  if (force_band) a.nsub = force_band;
  a.n_band = (a.n_rt + a.nsub - 1) / a.nsub;
  const int64_t tiles = (int64_t)a.n_ct * a.n_band * B;
  if (tiles >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  a.tiles = (uint32_t)tiles;
  a.q0 = (uint8_t*)q0;
  a.q1 = (uint8_t*)q1;
  a.s0 = make_spec(s0, s0_layout, R, C / 32, offs, E);
  a.s1 = make_spec(s1, s1_layout, C, R / 32, offs, E);
  a.status = status;
  int64_t grid = (a.tiles + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 2;
  if (grid > cap) grid = cap;
  if (q0) {
    k_mx_dual<true, true><<<(unsigned)grid, 256, 0, st>>>(a);
  } else {
    k_mx_dual<false, true><<<(unsigned)grid, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace fp8moe
