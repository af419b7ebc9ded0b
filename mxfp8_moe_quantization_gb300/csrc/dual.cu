// MXFP8 quantization of one bf16 tensor in both directions from a single read
// of it: dim0 (blocks of 32 along a row, codes [B, R, C]) and dim1 (blocks of
// 32 down a column, codes transposed to [B, C, R]), each with its e8m0 scales
// written straight into their final layout.  This is the operand preparation
// of the MXFP8 MoE layer ("Accelerating Llama4 Scout training with TorchAO
// MXFP8 MoE primitives": a tensor is quantized along both dimensions for the
// forward and the two backward GEMMs); doing both from one read moves 4 bytes
// per element instead of the 6 of two separate passes.
//
// Two forms.  Both directions with at least 128 columns run the
// warp-specialised kernel (k_mx_dual_ws, described where it is defined): a
// producer warp stages 32 x 128 sub-tiles in a shared-memory ring by TMA,
// and dim0 and dim1 consumer warps each take one direction, a lane one
// block.  Narrower tensors and the dim1-only call run the register-tile form
// below (k_mx_dual), which was measured faster there.
//
// Register-tile form: a warp owns a band of up to 128 rows x 128 columns and
// sweeps it in 32-row sub-tiles, so that every 128-byte line of the
// transposed codes and of the scales is completed by one warp within a short
// time (while it is still in L2); small tensors use lower bands so that every
// warp gets work.  Each warp has one 8 KB shared-memory buffer: a TMA load
// brings the next sub-tile (32 rows x 128 columns) into it while the warp
// works on the current one from registers, so every warp keeps a load in
// flight through its arithmetic.  In a sub-tile, lane l holds rows
// 16*(l/16) .. +15 of the 8 columns 8*(l%16) .. +7 in registers (16
// conflict-free 16-byte shared loads).
//   dim0: the 32-element block of a row spans 4 lanes: two shuffles give its
//         absolute maximum; each lane encodes and stores its 8 codes, so a
//         warp store writes two 128-byte row segments.
//   dim1: a lane has 16 rows of each of its columns; one shuffle with the
//         lane holding the other 16 rows gives the column block's maximum;
//         each lane stores 16 codes per column, the two halves of a column's
//         32-byte output segment coming from the two lanes.
#include <stdlib.h>

#include <string.h>

#include <atomic>
#include <type_traits>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "mxcvt.cuh"
#include "scales.cuh"
#include "tma.cuh"

namespace fp8moe {

namespace {

FP8MOE_DEV uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

FP8MOE_DEV uint4 lds16(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(saddr));
  return v;
}

constexpr int DUAL_WARPS = 8;                 // warps per CTA
constexpr int SUB_ROWS = 32;                  // rows of a sub-tile
constexpr int SUB_BYTES = SUB_ROWS * 128 * 2; // one sub-tile of bf16 (128 columns at most)
constexpr size_t DUAL_SMEM = (size_t)DUAL_WARPS * SUB_BYTES + DUAL_WARPS * sizeof(uint64_t);

struct DualArgs {
  const uint16_t* x;    // [B, R, C] bf16
  int64_t B, R, C;
  uint32_t n_ct, n_band, tiles;  // 128 columns x bands of `nsub` 32-row sub-tiles
  uint32_t n_rt;
  int nsub;
  int boxc;             // columns of the TMA box: min(128, C)
  uint8_t* q0;          // [B, R, C]
  uint8_t* q1;          // [B, C, R]
  ScaleSpec s0;         // [B, R, C/32] in its layout
  ScaleSpec s1;         // [B, C, R/32] in its layout
  int* status;
  int stall_test;       // warp-specialised form: CTA 0 never loads its first sub-tile (timeout-path test)
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
  const uint32_t efl = max((mw >> 7) & 0xFFu, 8u), efh = max((mw >> 23) & 0xFFu, 8u);
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
// the standalone transposed quantization).  PF: sub-tiles come through the
// warp's shared-memory buffer, loaded one ahead by TMA; otherwise each lane
// loads its 16 rows straight into registers when the sub-tile starts.
template <bool D0, bool D1, bool PF>
__global__ void __launch_bounds__(32 * DUAL_WARPS, 2) k_mx_dual(const __grid_constant__ CUtensorMap tx, DualArgs a) {
  __shared__ GroupTable gt0, gt1;
  extern __shared__ __align__(1024) uint8_t dsm[];
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
  // this warp's sub-tile buffer and the barrier its loads complete on
  const int wib = threadIdx.x >> 5;
  uint8_t* wbuf = dsm + wib * SUB_BYTES;
  uint64_t* wbar = reinterpret_cast<uint64_t*>(dsm + DUAL_WARPS * SUB_BYTES) + wib;
  if (PF && lane == 0) {
    mbar_init(wbar, 1);
    mbar_fence_init();
  }
  __syncwarp();
  const uint32_t box_bytes = (uint32_t)a.boxc * SUB_ROWS * 2;
  // a band tile's column tile, first row block, batch and first row of x
  struct Tile {
    uint32_t ct, rt0;
    int64_t b, row0;
  };
  auto tile_of = [&](uint32_t t) {
    Tile u;
    u.ct = t % a.n_ct;
    const uint32_t rest = t / a.n_ct;
    u.rt0 = (rest % a.n_band) * a.nsub;
    u.b = rest / a.n_band;
    u.row0 = u.b * a.R + (int64_t)u.rt0 * SUB_ROWS;
    return u;
  };
  // load the sub-tile at (row, column) of x into the buffer (one lane)
  auto issue = [&](int64_t row, uint32_t ct) {
    mbar_expect_tx(wbar, box_bytes);
    tma_load_2d(wbuf, &tx, wbar, (int)(ct * 128), (int)row);
  };
  uint32_t parity = 0;
  bool live = true;  // false after a wait ran out: no further loads or waits
  uint32_t lost = 0; // the phase whose wait ran out (its load may be in flight)
  const uint32_t t_first = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  Tile cur;
  if (t_first < a.tiles) {
    cur = tile_of(t_first);
    if (PF && lane == 0) issue(cur.row0, cur.ct);
  }
  // this lane's 16 rows x 16 bytes in the buffer
  const uint32_t lbase = smem_u32(wbuf) + (uint32_t)(half * 16 * a.boxc * 2 + cl * 16);
  const uint32_t lpitch = (uint32_t)a.boxc * 2;
  // Grouped layouts (B == 1): a warp's tiles come in increasing row order and
  // every 32-row sub-tile lies inside one routing group (offsets are
  // multiples of 32), so a forward-only cursor per table replaces the
  // binary searches: the group of row r is the first whose end exceeds r.
  int g0c = 0, g1c = 0;
  auto advance = [](const GroupTable& gt, int E, int& g, int64_t r) {
    while (g < E - 1 && gt.end[g] <= r) ++g;
  };
  for (uint32_t t = t_first; t < a.tiles; t += nwarps) {
    if (!PF) cur = tile_of(t);
    const uint32_t ct = cur.ct, rt0 = cur.rt0;
    const int64_t b = cur.b;
    const bool more = PF && t + nwarps < a.tiles;
    const Tile nxt = more ? tile_of(t + nwarps) : cur;
    // dim1 scale bytes of this lane's 8 columns over the band's row blocks
    // (byte `sub` of each word): the row blocks of a band are consecutive
    // scale bytes of a column in every layout, written as one word per column
    uint32_t sacc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int sub = 0; sub < a.nsub && rt0 + sub < a.n_rt; ++sub) {
      const int64_t rt = rt0 + sub;
      const int64_t r = rt * 32 + half * 16;   // first of this lane's 16 rows
      const int64_t c = (int64_t)ct * 128 + cl * 8;   // first of this lane's 8 columns
      const bool ok = c < a.C;                 // C % 32 == 0: whole 4-lane groups are in or out
      uint4 v[16];
      if (!PF) {
        const uint16_t* xp = a.x + (b * a.R + r) * a.C + c;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = ok ? ld_nc16(xp + i * a.C) : make_uint4(0, 0, 0, 0);
      } else {
      if (live && !mbar_wait(wbar, parity, nullptr)) {
        set_status(a.status, FP8MOE_ERR_TIMEOUT);
        live = false;
        lost = parity;
      }
      parity ^= 1;
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = ok ? lds16(lbase + i * lpitch) : make_uint4(0, 0, 0, 0);
      // the buffer is free again: the next sub-tile of this warp's sequence
      // starts loading while this one is worked on
      __syncwarp();
      }
      if (PF && lane == 0 && live) {
        fence_proxy_async_smem();
        if (sub + 1 < a.nsub && rt0 + sub + 1 < a.n_rt)
          issue(cur.row0 + (int64_t)(sub + 1) * SUB_ROWS, ct);
        else if (more)
          issue(nxt.row0, nxt.ct);
      }

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
        // magnitudes (the sign bits of m2 are meaningless; the exponent
        // field below drops them)
        uint32_t m2 = max_abs_bf16x2(max_abs_bf16x2(v[i].x, v[i].y), max_abs_bf16x2(v[i].z, v[i].w));
        m2 = max_abs_bf16x2(m2, __byte_perm(m2, 0, 0x1032));   // both halves: the chunk's maximum
        m2 = max_abs_bf16x2(m2, __shfl_xor_sync(FULL, m2, 1));
        m2 = max_abs_bf16x2(m2, __shfl_xor_sync(FULL, m2, 2));
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
        mw[0] = max_abs_bf16x2(mw[0], v[i].x);
        mw[1] = max_abs_bf16x2(mw[1], v[i].y);
        mw[2] = max_abs_bf16x2(mw[2], v[i].z);
        mw[3] = max_abs_bf16x2(mw[3], v[i].w);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) mw[k] = max_abs_bf16x2(mw[k], __shfl_xor_sync(FULL, mw[k], 16));
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
    if (PF) cur = nxt;
  }
  // after a wait that ran out, wait (bounded) once more for that load, the
  // only one that can be in flight, before the warp's buffer goes away
  if (PF && !live && lane == 0) (void)mbar_wait(wbar, lost, nullptr);
}

// ---------------------------------------------------------------------------
// Warp-specialised form of both directions (C >= 128).  The CTA walks its
// band tiles (the same enumeration as above, tiles blockIdx.x, + gridDim.x,
// ...) sub-tile by sub-tile; a producer warp brings each 32-row x 128-column
// sub-tile into a four-slot shared-memory ring by TMA (two 64-column boxes,
// 128-byte swizzle: 16-byte chunk c of row r at r * 128 + (c ^ (r % 8)) * 16)
// and eight consumer warps work on it from there:
//   dim0 warps 0-3: a lane owns one 32-element block of a row (row
//         8w + lane / 4, block lane % 4): four 16-byte reads, its maximum
//         without shuffles, 32 codes as two 16-byte stores (the four lanes of
//         a row write its 128 bytes) and the block's scale byte;
//   dim1 warps 4-7: a lane owns a column pair for 16 rows (pair
//         16 (w - 4) + lane % 16, rows 16 (lane / 16) ...): sixteen 4-byte
//         reads, one shuffle with the lane holding the other 16 rows for the
//         column maxima, and 16 codes per column as one 16-byte store.
// Per element this is about half the instruction count of the register-tile
// form (whose dim0 block spans four lanes: two shuffles and the scale work
// four times per block), and with under 80 registers three CTAs fit per SM.
constexpr int WS_SLOTS = 4;
constexpr int WS_SUB_BYTES = 32 * 128 * 2;   // one sub-tile: two 64-column x 32-row boxes of 4 KB
constexpr size_t WS_SMEM = (size_t)WS_SLOTS * WS_SUB_BYTES + 1024;   // + room to align the ring to 1 KB
// consumer warps: 4 dim0 + 4 dim1, or (dim1 alone) 4 dim1; one producer warp
template <bool D0>
__host__ __device__ constexpr int ws_consumers() { return D0 ? 8 : 4; }
template <bool D0>
__host__ __device__ constexpr int ws_threads() { return 32 * (ws_consumers<D0>() + 1); }

FP8MOE_DEV uint32_t lds32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
  return v;
}

template <bool D0>
__global__ void __launch_bounds__(ws_threads<D0>(), 3) k_mx_dual_ws(const __grid_constant__ CUtensorMap tx, DualArgs a) {
  constexpr int WS_CONSUMERS = ws_consumers<D0>();
  __shared__ std::conditional_t<D0, GroupTable, char> gt0_s;
  __shared__ GroupTable gt1;
  __shared__ uint64_t full[WS_SLOTS], empty[WS_SLOTS];
  __shared__ int abort_s;
  // grouped layouts, per slot: the row shift into the padded scale matrix of
  // the sub-tile's group (dim0: padded row = row + shift0, or NO_SHIFT when
  // a group ends inside the sub-tile; dim1: padded 32-block column = block +
  // shift1), set by the producer before it issues the slot's load
  __shared__ int64_t shift0_s[WS_SLOTS], shift1_s[WS_SLOTS];
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  if constexpr (D0) {
    if (a.s0.layout == FP8MOE_GROUP_ROWS) {
      build_group_table(gt0_s, a.s0.offs, a.s0.E, a.R, GT_ROWS128, a.status);
      if (gt0_s.bad) return;
    }
  }
  if (a.s1.layout == FP8MOE_GROUP_COLS) {
    build_group_table(gt1, a.s1.offs, a.s1.E, a.R, GT_COLS, a.status);
    if (gt1.bad) return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < WS_SLOTS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], WS_CONSUMERS);
    }
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  auto tile_of = [&](uint32_t t, uint32_t& ct, uint32_t& rt0, int64_t& b) {
    ct = t % a.n_ct;
    const uint32_t rest = t / a.n_ct;
    rt0 = (rest % a.n_band) * a.nsub;
    b = rest / a.n_band;
  };
  const uint32_t ring_s = smem_u32(ring);

  constexpr int64_t NO_SHIFT = -((int64_t)1 << 62);   // no shift: rows of two groups
  if (warp == WS_CONSUMERS) {
    // ======================= producer =======================
    if (lane == 0) {
      uint32_t k = 0;
      int pg0 = 0, pg1 = 0;   // group cursors (the CTA's rows only grow: B == 1 for grouped layouts)
      for (uint32_t t = blockIdx.x; t < a.tiles && !abort_s; t += gridDim.x) {
        uint32_t ct, rt0;
        int64_t b;
        tile_of(t, ct, rt0, b);
        const int nv = (int)min((uint32_t)a.nsub, a.n_rt - rt0);
        for (int sub = 0; sub < nv; ++sub, ++k) {
          const uint32_t s = k % WS_SLOTS, round = k / WS_SLOTS;
          if (k >= WS_SLOTS && !mbar_wait(&empty[s], (round - 1) & 1u, &abort_s)) {
            if (!abort_s) set_status(a.status, FP8MOE_ERR_TIMEOUT);
            abort_s = 1;
            break;
          }
          const int64_t r = (int64_t)(rt0 + sub) * 32;
          if constexpr (D0) {
            if (a.s0.layout == FP8MOE_GROUP_ROWS) {
              const GroupTable& gt0 = gt0_s;
              while (pg0 < a.s0.E - 1 && gt0.end[pg0] <= r) ++pg0;
              const int64_t gs = pg0 == 0 ? 0 : gt0.end[pg0 - 1];
              shift0_s[s] = gt0.end[pg0] >= r + 32 ? gt0.pad[pg0] - gs : NO_SHIFT;
            }
          }
          if (a.s1.layout == FP8MOE_GROUP_COLS) {
            while (pg1 < a.s1.E - 1 && gt1.end[pg1] <= r) ++pg1;
            const int64_t gs = pg1 == 0 ? 0 : gt1.end[pg1 - 1];
            shift1_s[s] = gt1.pad[pg1] - gs / 32;
          }
          const int row = (int)(b * a.R + r);
          // test hook: CTA 0's first sub-tile is never loaded, so its
          // consumers' bounded wait runs out
          if (a.stall_test && blockIdx.x == 0 && k == 0) continue;
          // (the arrive below releases the shifts to the consumers' wait)
          mbar_expect_tx(&full[s], WS_SUB_BYTES);
          tma_load_2d(ring + s * WS_SUB_BYTES, &tx, &full[s], (int)(ct * 128), row);
          tma_load_2d(ring + s * WS_SUB_BYTES + WS_SUB_BYTES / 2, &tx, &full[s], (int)(ct * 128 + 64), row);
        }
      }
      // the loads still in flight land before the CTA can leave: the last
      // fill of each slot (the consumers may have stopped early)
      for (uint32_t j = k > WS_SLOTS ? k - WS_SLOTS : 0; j < k; ++j)
        (void)mbar_wait(&full[j % WS_SLOTS], (j / WS_SLOTS) & 1u, nullptr);
    }
    return;
  }

  // ======================= consumers =======================
  const bool d0w = D0 && warp < 4;
  // dim0 lane: row rl of the sub-tile, 32-column block bq
  const int bq = lane & 3, rl = warp * 8 + (lane >> 2);
  // dim1 lane: column pair cp (columns 2cp, 2cp + 1), rows 16 * half ...
  const int half = lane >> 4, cp = (warp & 3) * 16 + (lane & 15);
  int g0c = 0;   // forward-only group cursor for rows whose sub-tile holds two groups
  auto advance = [](const GroupTable& gt, int E, int& g, int64_t r) {
    while (g < E - 1 && gt.end[g] <= r) ++g;
  };
  uint32_t k = 0;
  bool ok = true;
  for (uint32_t t = blockIdx.x; t < a.tiles && ok; t += gridDim.x) {
    uint32_t ct, rt0;
    int64_t b;
    tile_of(t, ct, rt0, b);
    const int nv = (int)min((uint32_t)a.nsub, a.n_rt - rt0);
    const int64_t c0 = (int64_t)ct * 128;
    for (int sub = 0; sub < nv; ++sub, ++k) {
      const uint32_t s = k % WS_SLOTS;
      if (!mbar_wait(&full[s], (k / WS_SLOTS) & 1u, &abort_s)) {
        if (!abort_s) set_status(a.status, FP8MOE_ERR_TIMEOUT);
        abort_s = 1;
        ok = false;
        break;
      }
      const int64_t r = (int64_t)(rt0 + sub) * 32;   // first row of the sub-tile (in batch b)
      const uint32_t slot = ring_s + s * WS_SUB_BYTES;
      if constexpr (D0) {
      if (d0w) {
        const GroupTable& gt0 = gt0_s;
        // ---- dim0: the block of 32 at (row r + rl, columns c0 + 32 bq ...)
        const int64_t col = c0 + 32 * bq;
        const uint32_t rb = slot + (uint32_t)((bq >> 1) * (WS_SUB_BYTES / 2) + rl * 128);
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = lds16(rb + (uint32_t)(((((bq & 1) * 4 + j) ^ (rl & 7))) << 4));
        const int64_t sh0 = a.s0.layout == FP8MOE_GROUP_ROWS ? shift0_s[s] : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        uint32_t m2 = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          m2 = max_abs_bf16x2(m2, max_abs_bf16x2(max_abs_bf16x2(v[j].x, v[j].y), max_abs_bf16x2(v[j].z, v[j].w)));
        m2 = max_abs_bf16x2(m2, __byte_perm(m2, 0, 0x1032));
        uint32_t p2;
        const uint32_t byte = mx_block_scale(m2 & 0xFFFFu, p2);
        if (col < a.C) {
          const uint2 e0 = enc_row8(v[0], p2), e1 = enc_row8(v[1], p2), e2 = enc_row8(v[2], p2),
                      e3 = enc_row8(v[3], p2);
          uint8_t* qp = a.q0 + (b * a.R + r + rl) * a.C + col;
          *reinterpret_cast<uint4*>(qp) = make_uint4(e0.x, e0.y, e1.x, e1.y);
          *reinterpret_cast<uint4*>(qp + 16) = make_uint4(e2.x, e2.y, e3.x, e3.y);
          int64_t off;
          if (a.s0.layout == FP8MOE_GROUP_ROWS) {
            if (sh0 != NO_SHIFT) {
              off = tile_off(r + rl + sh0, col >> 5, a.s0.Cp);
            } else {
              // a group ends inside this sub-tile: this row's own group
              advance(gt0, a.s0.E, g0c, r + rl);
              const int64_t gs = g0c == 0 ? 0 : gt0.end[g0c - 1];
              off = tile_off(gt0.pad[g0c] + (r + rl - gs), col >> 5, a.s0.Cp);
            }
          } else if (a.s0.layout == FP8MOE_NO_GROUPS) {
            off = b * a.s0.Rp * a.s0.Cp + tile_off(r + rl, col >> 5, a.s0.Cp);
          } else {
            off = (b * a.R + r + rl) * (a.C >> 5) + (col >> 5);
          }
          a.s0.p[off] = (uint8_t)byte;
        }
        continue;
      }
      }
      {
        // ---- dim1: columns (2cp, 2cp + 1) over rows r + 16 half ... + 15
        const uint32_t cb = slot + (uint32_t)((cp >> 5) * (WS_SUB_BYTES / 2) + (cp & 3) * 4);
        const uint32_t cc = (uint32_t)((cp & 31) >> 2);
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t row = (uint32_t)(half * 16 + i);
          v[i] = lds32(cb + row * 128 + ((cc ^ (row & 7)) << 4));
        }
        const int64_t sh1 = a.s1.layout == FP8MOE_GROUP_COLS ? shift1_s[s] : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        uint32_t mw = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) mw = max_abs_bf16x2(mw, v[i]);
        mw = max_abs_bf16x2(mw, __shfl_xor_sync(FULL, mw, 16));
        const uint32_t efl = max((mw >> 7) & 0xFFu, 8u), efh = max((mw >> 23) & 0xFFu, 8u);
        const uint32_t p2 = ((262u - efl) << 7) | ((262u - efh) << 23);
        const int64_t col = c0 + 2 * cp;
        if (col < a.C) {
          if (half == 0) {
            // the two columns' scale bytes of row block r / 32 (the sub-tile
            // lies inside one routing group: offsets are multiples of 32)
            const int64_t rb = r >> 5;
            int64_t off, step;
            if (a.s1.layout == FP8MOE_GROUP_COLS) {
              off = tile_off(col, rb + sh1, a.s1.Cp);
              step = 16;
            } else if (a.s1.layout == FP8MOE_NO_GROUPS) {
              off = b * a.s1.Rp * a.s1.Cp + tile_off(col, rb, a.s1.Cp);
              step = 16;
            } else {
              off = (b * a.C + col) * (a.R >> 5) + rb;
              step = a.R >> 5;
            }
            a.s1.p[off] = (uint8_t)(efl - 8u);
            a.s1.p[off + step] = (uint8_t)(efh - 8u);
          }
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t y0 = mul_bf16x2(v[4 * q], p2), y1 = mul_bf16x2(v[4 * q + 1], p2);
            const uint32_t y2 = mul_bf16x2(v[4 * q + 2], p2), y3 = mul_bf16x2(v[4 * q + 3], p2);
            lo[q] = cvt4(lo_f32(y0), lo_f32(y1), lo_f32(y2), lo_f32(y3));
            hi[q] = cvt4(hi_f32(y0), hi_f32(y1), hi_f32(y2), hi_f32(y3));
          }
          uint8_t* qp = a.q1 + (b * a.C + col) * a.R + r + half * 16;
          *reinterpret_cast<uint4*>(qp) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint4*>(qp + a.R) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
      }
    }
    if (!ok) break;
  }
}

}  // namespace

// One-shot test hook of the warp-specialised quantizers (this file and the
// jagged colwise kernel): armed by fp8moe_testing_stall_next_quant_ring,
// consumed by the next such launch.
static std::atomic<int> g_ring_stall{0};
void arm_ring_stall_hook() { g_ring_stall.store(1, std::memory_order_relaxed); }
int take_ring_stall_hook() { return g_ring_stall.exchange(0, std::memory_order_relaxed); }

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
  // FP8MOE_DUAL_BAND=1|2|4 fixes the band height (tests use it to cover every
  // band shape on small inputs)
  static const int force_band = [] {
    const char* v = getenv("FP8MOE_DUAL_BAND");
    const int n = v ? atoi(v) : 0;
    return (n == 1 || n == 2 || n == 4) ? n : 0;
  }();
  // both directions with at least one whole 128-column tile: the
  // warp-specialised kernel (FP8MOE_DUAL_WS=0 keeps the register-tile form,
  // for comparison).  Its dim1-only instance (four dim1 warps) measured
  // slower than the register-tile form (Scout W1 412 against 387 us, the
  // activation 57 against 49 us), which keeps that case; FP8MOE_DUAL_WS=1
  // selects it anyway.
  static const int ws_env = [] {
    const char* v = getenv("FP8MOE_DUAL_WS");
    return v ? atoi(v) : -1;
  }();
  if (C >= 128 && (q0 ? ws_env != 0 : ws_env == 1)) {
    static std::atomic<int> per_sm_ws[2];
    static std::once_flag ws_once;
    std::call_once(ws_once, [] {
      cudaFuncSetAttribute(k_mx_dual_ws<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)WS_SMEM);
      cudaFuncSetAttribute(k_mx_dual_ws<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)WS_SMEM);
    });
    const bool both = q0 != nullptr;
    const int per = both ? blocks_per_sm(per_sm_ws[1], k_mx_dual_ws<true>, ws_threads<true>(), WS_SMEM, 2)
                         : blocks_per_sm(per_sm_ws[0], k_mx_dual_ws<false>, ws_threads<false>(), WS_SMEM, 2);
    const int64_t ctas = (int64_t)num_sms * per;
    // bands of 4 sub-tiles while every CTA gets 16 band tiles or more
    a.nsub = 4;
    while (a.nsub > 1 && (int64_t)a.n_ct * ((a.n_rt + a.nsub - 1) / a.nsub) * B < 16 * ctas) a.nsub >>= 1;
    if (force_band) a.nsub = force_band;
    a.n_band = (a.n_rt + a.nsub - 1) / a.nsub;
    const int64_t tiles = (int64_t)a.n_ct * a.n_band * B;
    if (tiles >= ((int64_t)1 << 31) || B * R >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    a.tiles = (uint32_t)tiles;
    a.boxc = 64;
    a.q0 = (uint8_t*)q0;
    a.q1 = (uint8_t*)q1;
    a.s0 = make_spec(s0, both ? s0_layout : FP8MOE_SCALES_ROWMAJOR, R, C / 32, offs, E);
    a.s1 = make_spec(s1, s1_layout, C, R / 32, offs, E);
    a.status = status;
    a.stall_test = take_ring_stall_hook();
    CUtensorMap tx;
    memset(&tx, 0, sizeof(tx));
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(B * R)};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {64, 32};
    if (!make_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 2, dims, strides, box)) return cudaErrorInvalidValue;
    const int64_t grid = tiles < ctas ? tiles : ctas;
    if (both)
      k_mx_dual_ws<true><<<(unsigned)grid, ws_threads<true>(), WS_SMEM, st>>>(tx, a);
    else
      k_mx_dual_ws<false><<<(unsigned)grid, ws_threads<false>(), WS_SMEM, st>>>(tx, a);
    return cudaGetLastError();
  }
  // bands of 4 sub-tiles when that leaves several bands per warp, else lower
  const int64_t warps = (int64_t)num_sms * 2 * 8;
  a.nsub = 4;
  while (a.nsub > 1 && (int64_t)a.n_ct * ((a.n_rt + a.nsub - 1) / a.nsub) * B < 4 * warps) a.nsub >>= 1;
  if (force_band) a.nsub = force_band;
  a.n_band = (a.n_rt + a.nsub - 1) / a.nsub;
  const int64_t tiles = (int64_t)a.n_ct * a.n_band * B;
  if (tiles >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  a.tiles = (uint32_t)tiles;
  a.boxc = (int)(C < 128 ? C : 128);
  a.q0 = (uint8_t*)q0;
  a.q1 = (uint8_t*)q1;
  a.s0 = make_spec(s0, s0_layout, R, C / 32, offs, E);
  a.s1 = make_spec(s1, s1_layout, C, R / 32, offs, E);
  a.status = status;
  a.stall_test = 0;
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(k_mx_dual<true, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DUAL_SMEM);
    cudaFuncSetAttribute(k_mx_dual<false, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DUAL_SMEM);
  });
  int64_t grid = (a.tiles + DUAL_WARPS - 1) / DUAL_WARPS;
  const int64_t cap = (int64_t)num_sms * 2;
  if (grid > cap) grid = cap;
  // the prefetching form for the dim1-only kernel and, for both directions,
  // where every warp has few sub-tiles (its loads would otherwise wait in
  // the open); plain loads where each warp has many sub-tiles of both
  // directions' arithmetic (measured faster there: Scout W1 530 against 545
  // us, DeepSeek-V3 W1 2951 against 3185 us; the activations 82 against 88).
  // FP8MOE_DUAL_PREFETCH=0|1 fixes the form (tests cover both).
  const int64_t subs_per_warp = (int64_t)a.tiles * a.nsub / (grid * DUAL_WARPS);
  static const int pf_env = [] {
    const char* v = getenv("FP8MOE_DUAL_PREFETCH");
    return v ? atoi(v) : -1;
  }();
  const bool pf = pf_env >= 0 ? pf_env != 0 : (!q0 || subs_per_warp < 32);
  // x as a 2D [B*R, C] bf16 tensor; one box is a sub-tile (columns past C
  // read as zero)
  CUtensorMap tx;
  memset(&tx, 0, sizeof(tx));
  {
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(B * R)};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {(cuuint32_t)a.boxc, (cuuint32_t)SUB_ROWS};
    if (pf && !make_tmap(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  const size_t smem = pf ? DUAL_SMEM : 0;
  if (q0) {
    if (pf)
      k_mx_dual<true, true, true><<<(unsigned)grid, 32 * DUAL_WARPS, smem, st>>>(tx, a);
    else
      k_mx_dual<true, true, false><<<(unsigned)grid, 32 * DUAL_WARPS, smem, st>>>(tx, a);
  } else {
    if (pf)
      k_mx_dual<false, true, true><<<(unsigned)grid, 32 * DUAL_WARPS, smem, st>>>(tx, a);
    else
      k_mx_dual<false, true, false><<<(unsigned)grid, 32 * DUAL_WARPS, smem, st>>>(tx, a);
  }
  return cudaGetLastError();
}

}  // namespace fp8moe
