// Colwise FP8 quantization: one scale per (expert, column), over the rows of
// a dense expert weight [E, R, C] or over each group of routed rows [R, C]
// delimited by offsets ("FP8-обучение на AMD", sections "MoE: почему
// DeepSeek-V3 ломал пайплайн" and "Три уровня оптимизации": column scales
// per expert, the transposed output written without a separate copy).
//
// Three streaming passes instead of one strip held on chip:
//   1. k_cw_amax  reads x once, coalesced (128 bytes of a row per 8 lanes),
//                 and folds per-column maxima into the scale buffer with
//                 atomicMax on the bf16 bit patterns (order-preserving for
//                 non-negative values);
//   2. k_cw_cast  reads x again, in the reverse tile order so that its first
//                 tiles are the last ones the amax pass left in L2, and
//                 writes the codes: untransposed rows, or 8-byte column
//                 runs transposed in registers (no shared-memory staging;
//                 4 lanes fill 32 contiguous bytes of an output row);
//   3. k_cw_finish turns each maximum into fl(1 / fl(fp8_max / amax)) in
//                 place and zeroes the slack after the last group of the
//                 jagged transposed layout.
// Work is cut into warp sub-tiles of 32 rows x 64 columns aligned to the
// groups, so no sub-tile straddles two groups; a lane holds 8 rows x 8
// columns (few registers: many warps per SM keep enough loads in flight).  In the jagged transposed layout a group's last sub-tile covers
// exactly its zero padding up to the next multiple of 32.
#include <cuda_runtime.h>
#include <stdint.h>

#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "launch.h"
#include "scales.cuh"

namespace fp8moe {
namespace {

constexpr int CW_SUB = 32;            // rows of a warp sub-tile
constexpr int CW_LR = 8;              // rows held by a lane
constexpr int CW_NRQ = CW_SUB / CW_LR;  // lanes along the rows of a sub-tile
constexpr int CW_NCL = 32 / CW_NRQ;   // lanes along the columns, 8 columns each
constexpr int CW_TC = CW_NCL * 8;     // columns of a tile
constexpr int CW_WARPS = 8;           // sub-tiles (warps) per CTA unit

struct CwArgs {
  const uint16_t* x;
  int64_t R, C;            // dense: rows per expert; jagged: total rows
  int E;
  const int32_t* offs;     // null: dense
  int64_t nsub;            // dense: sub-tiles per expert, ceil(R / 32)
  int64_t n_units;         // row blocks x column tiles
  int n_ct;                // column tiles
  int64_t ldt;             // jagged transposed row length
  uint8_t* q;
  uint32_t* amax;          // [E, C] column maxima as bf16 bit patterns
  const uint32_t* fixed;   // tensorwise: one maximum for every column
  int* status;
};

struct Sub {
  int g;                   // group, -1 past the last sub-tile
  int64_t j;               // sub-tile index inside the group
  int64_t r0, r1;          // first row of the sub-tile, end row of the group
};

// Sub-tile s of the group-aligned sequence.  Jagged: pad[g] is the number of
// sub-tiles before group g; the owner of s is the last group with pad <= s
// (an empty group shares its first sub-tile index with its successor).
template <bool JAG>
FP8MOE_DEV Sub locate(const CwArgs& a, const GroupTable& gt, int64_t total, int64_t s) {
  Sub o{-1, 0, 0, 0};
  if (s >= total) return o;
  if constexpr (!JAG) {
    const int64_t g = s / a.nsub;
    o.g = (int)g;
    o.j = s - g * a.nsub;
    o.r0 = g * a.R + o.j * CW_SUB;
    o.r1 = g * a.R + a.R;
  } else {
    int lo = 0, hi = a.E - 1, g = 0;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (gt.pad[mid] <= s) {
        g = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    o.g = g;
    o.j = s - gt.pad[g];
    o.r0 = (g == 0 ? 0 : gt.end[g - 1]) + o.j * CW_SUB;
    o.r1 = gt.end[g];
  }
  return o;
}

// Sub-tiles in the sequence (jagged: after the table is built).
template <bool JAG>
FP8MOE_DEV int64_t total_subs(const CwArgs& a, const GroupTable& gt) {
  if constexpr (!JAG) {
    return (int64_t)a.E * a.nsub;
  } else {
    const int64_t last = gt.end[a.E - 1] - (a.E > 1 ? gt.end[a.E - 2] : 0);
    return gt.pad[a.E - 1] + (last + 31) / 32;
  }
}

FP8MOE_DEV uint4 ld16(const uint16_t* p) { return ld_nc16(p); }

// The rows of a lane (rows at or past r1 read as zeros); all loads are
// issued before any is consumed.
FP8MOE_DEV void load_rows(const CwArgs& a, int64_t rr, int64_t r1, int64_t c, uint4 (&v)[CW_LR]) {
  const uint16_t* p = a.x + rr * a.C + c;
  if (rr + CW_LR <= r1) {
#pragma unroll
    for (int k = 0; k < CW_LR; ++k) v[k] = ld16(p + k * a.C);
  } else {
    const int64_t n = r1 - rr;
#pragma unroll
    for (int k = 0; k < CW_LR; ++k) v[k] = k < n ? ld16(p + k * a.C) : make_uint4(0, 0, 0, 0);
  }
}

FP8MOE_DEV void flush_max(const CwArgs& a, int g, int64_t col, uint32_t acc) {
  if (g < 0) return;
  uint32_t* p = a.amax + (int64_t)g * a.C + col;
  if (acc & 0xFFFFu) atomicMax(p, acc & 0xFFFFu);
  if (acc >> 16) atomicMax(p + 1, acc >> 16);
}

template <bool JAG>
__global__ void __launch_bounds__(256) k_cw_amax(CwArgs a) {
  __shared__ GroupTable gt;
  __shared__ uint4 red[CW_WARPS][CW_NCL];
  __shared__ int gsel[CW_WARPS];
  if constexpr (JAG) {
    build_group_table(gt, a.offs, a.E, a.R, GT_SUB32, a.status);
    if (gt.bad) return;
  }
  const int64_t total = total_subs<JAG>(a, gt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cl = lane % CW_NCL, rq = lane / CW_NCL;
  for (int64_t u = blockIdx.x; u < a.n_units; u += gridDim.x) {
    const int ct = (int)(u % a.n_ct);
    const Sub sb = locate<JAG>(a, gt, total, (u / a.n_ct) * CW_WARPS + warp);
    const int64_t c = (int64_t)ct * CW_TC + cl * 8;
    uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    if (sb.g >= 0 && c < a.C) {
      uint4 v[CW_LR];
      load_rows(a, sb.r0 + rq * CW_LR, sb.r1, c, v);
#pragma unroll
      for (int k = 0; k < CW_LR; ++k) {
        m0 = umax16x2(m0, v[k].x & 0x7FFF7FFFu);
        m1 = umax16x2(m1, v[k].y & 0x7FFF7FFFu);
        m2 = umax16x2(m2, v[k].z & 0x7FFF7FFFu);
        m3 = umax16x2(m3, v[k].w & 0x7FFF7FFFu);
      }
    }
    // the row groups of a column sit in lanes cl, cl + NCL, ...
#pragma unroll
    for (int o = CW_NCL; o < 32; o <<= 1) {
      m0 = umax16x2(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = umax16x2(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      m2 = umax16x2(m2, __shfl_xor_sync(0xffffffffu, m2, o));
      m3 = umax16x2(m3, __shfl_xor_sync(0xffffffffu, m3, o));
    }
    if (lane < CW_NCL) red[warp][lane] = make_uint4(m0, m1, m2, m3);
    if (lane == 0) gsel[warp] = sb.g;
    __syncthreads();
    if (threadIdx.x < CW_NCL * 4) {
      // one column pair per thread; consecutive warps of the same group are
      // combined before the atomic
      const int l = threadIdx.x >> 2, wi = threadIdx.x & 3;
      const int64_t col = (int64_t)ct * CW_TC + l * 8 + wi * 2;
      if (col < a.C) {
        int cur = -1;
        uint32_t acc = 0;
        for (int w = 0; w < CW_WARPS; ++w) {
          const int gw = gsel[w];
          if (gw != cur) {
            flush_max(a, cur, col, acc);
            cur = gw;
            acc = 0;
          }
          acc = umax16x2(acc, reinterpret_cast<const uint32_t*>(&red[w][l])[wi]);
        }
        flush_max(a, cur, col, acc);
      }
    }
    __syncthreads();
  }
}


template <bool JAG, bool TRANS, bool FNUZ>
__global__ void __launch_bounds__(256) k_cw_cast(CwArgs a) {
  __shared__ GroupTable gt;
  if constexpr (JAG) {
    build_group_table(gt, a.offs, a.E, a.R, GT_SUB32, a.status);
    if (gt.bad) return;
  }
  const int64_t total = total_subs<JAG>(a, gt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cl = lane % CW_NCL, rq = lane / CW_NCL;
  const bool fixed = a.fixed != nullptr;
  const uint32_t fixed_bits = fixed ? *a.fixed : 0u;
  for (int64_t i = blockIdx.x; i < a.n_units; i += gridDim.x) {
    const int64_t u = a.n_units - 1 - i;
    const int ct = (int)(u % a.n_ct);
    const Sub sb = locate<JAG>(a, gt, total, (u / a.n_ct) * CW_WARPS + warp);
    const int64_t c = (int64_t)ct * CW_TC + cl * 8;
    if (sb.g < 0 || c >= a.C) continue;
    float sv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t bits = fixed ? fixed_bits : a.amax[(int64_t)sb.g * a.C + c + t];
      float inv;
      rowwise_scale<FNUZ>(bf16bits_to_float(bits), sv[t], inv);
      sv[t] = enc_mul<FNUZ>(sv[t]);
    }
    const int64_t rr = sb.r0 + rq * CW_LR;
    uint4 v[CW_LR];
    load_rows(a, rr, sb.r1, c, v);
    uint32_t w0[CW_LR], w1[CW_LR];
#pragma unroll
    for (int k = 0; k < CW_LR; ++k) {
      w0[k] = enc4_pre<FNUZ>(__fmul_rn(bf16_lo(v[k].x), sv[0]), __fmul_rn(bf16_hi(v[k].x), sv[1]),
                         __fmul_rn(bf16_lo(v[k].y), sv[2]), __fmul_rn(bf16_hi(v[k].y), sv[3]));
      w1[k] = enc4_pre<FNUZ>(__fmul_rn(bf16_lo(v[k].z), sv[4]), __fmul_rn(bf16_hi(v[k].z), sv[5]),
                         __fmul_rn(bf16_lo(v[k].w), sv[6]), __fmul_rn(bf16_hi(v[k].w), sv[7]));
    }
    if constexpr (!TRANS) {
#pragma unroll
      for (int k = 0; k < CW_LR; ++k)
        if (rr + k < sb.r1) *reinterpret_cast<uint2*>(a.q + (rr + k) * a.C + c) = make_uint2(w0[k], w1[k]);
    } else {
      // 8 consecutive rows of each of the 8 columns as one 8-byte store
      uint8_t* base;
      int64_t pitch;
      if constexpr (JAG) {
        pitch = a.ldt;
        base = a.q + c * pitch + (gt.pad[sb.g] + sb.j) * CW_SUB + rq * CW_LR;
      } else {
        pitch = a.R;
        const int64_t off = sb.j * CW_SUB + rq * CW_LR;
        if (off >= a.R) continue;  // R % 8 == 0: a lane's rows are all in or all out
        base = a.q + ((int64_t)sb.g * a.C + c) * pitch + off;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t* W = h ? w1 : w0;
        uint32_t q0[4], q1[4];
        transpose4x4(W[0], W[1], W[2], W[3], q0);
        transpose4x4(W[4], W[5], W[6], W[7], q1);
#pragma unroll
        for (int t = 0; t < 4; ++t) *reinterpret_cast<uint2*>(base + (h * 4 + t) * pitch) = make_uint2(q0[t], q1[t]);
      }
    }
  }
}

// Blocks [0, n_a): column maxima -> dequantization scales, in place.
// Blocks [n_a, gridDim.x): zero columns [32 * sub-tiles, ldt) of every row of
// the jagged transposed output (the slack after the last group).
template <bool FNUZ>
__global__ void __launch_bounds__(256) k_cw_finish(CwArgs a, int64_t n_inv, int n_a) {
  if ((int)blockIdx.x < n_a) {
    float* inv = reinterpret_cast<float*>(a.amax);
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n_inv; i += (int64_t)n_a * 256) {
      float s, iv;
      rowwise_scale<FNUZ>(bf16bits_to_float(a.amax[i]), s, iv);
      inv[i] = iv;
    }
    return;
  }
  __shared__ int64_t part[8];
  int64_t subs = 0;
  int bad = 0;
  for (int e = threadIdx.x; e < a.E; e += 256) {
    const int64_t end = a.offs[e], start = e == 0 ? 0 : a.offs[e - 1];
    if (end < start || end > a.R || (e == a.E - 1 && end != a.R)) bad = 1;
    subs += (end - start + 31) / 32;
  }
  for (int o = 16; o > 0; o >>= 1) subs += __shfl_xor_sync(0xffffffffu, subs, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = subs;
  if (__syncthreads_or(bad)) return;  // the cast pass reports the offsets
  int64_t total = 0;
  for (int w = 0; w < 8; ++w) total += part[w];
  const int64_t from = total * CW_SUB;
  const int64_t chunks = (a.ldt - from) / 16;
  if (chunks <= 0) return;
  const int nb = (int)gridDim.x - n_a;
  for (int64_t k = (int64_t)(blockIdx.x - n_a) * 256 + threadIdx.x; k < a.C * chunks; k += (int64_t)nb * 256) {
    const int64_t row = k / chunks, ch = k - row * chunks;
    *reinterpret_cast<uint4*>(a.q + row * a.ldt + from + ch * 16) = make_uint4(0, 0, 0, 0);
  }
}

template <typename K>
static int resident(K kern, int num_sms) {
  int per = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, 256, 0) != cudaSuccess || per < 1) {
    (void)cudaGetLastError();
    per = 1;
  }
  return per * num_sms;
}

template <bool JAG>
static cudaError_t launch_amax(const CwArgs& a, int num_sms, cudaStream_t st) {
  static int cap = 0;
  if (!cap) cap = resident(k_cw_amax<JAG>, num_sms);
  const int64_t grid = a.n_units < cap ? a.n_units : cap;
  k_cw_amax<JAG><<<(unsigned)grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <bool JAG, bool TRANS, bool FNUZ>
static cudaError_t launch_cast(const CwArgs& a, int num_sms, cudaStream_t st) {
  static int cap = 0;
  if (!cap) cap = resident(k_cw_cast<JAG, TRANS, FNUZ>, num_sms);
  const int64_t grid = a.n_units < cap ? a.n_units : cap;
  k_cw_cast<JAG, TRANS, FNUZ><<<(unsigned)grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <bool JAG, bool TRANS>
static cudaError_t launch_cast_k(const CwArgs& a, bool fnuz, int num_sms, cudaStream_t st) {
  return fnuz ? launch_cast<JAG, TRANS, true>(a, num_sms, st) : launch_cast<JAG, TRANS, false>(a, num_sms, st);
}

static cudaError_t run_colwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                               int transpose_out, int kind, int64_t ldt, void* q, float* inv,
                               const uint32_t* fixed, int* status, int num_sms, cudaStream_t st) {
  if (E == 0 || C == 0) return cudaSuccess;
  CwArgs a;
  a.x = (const uint16_t*)x;
  a.R = R;
  a.C = C;
  a.E = (int)E;
  a.offs = offs;
  a.nsub = offs ? 0 : (R + CW_SUB - 1) / CW_SUB;
  const int64_t subs = offs ? (R + CW_SUB - 1) / CW_SUB + E : E * a.nsub;  // jagged: an upper bound
  a.n_ct = (int)((C + CW_TC - 1) / CW_TC);
  a.n_units = (subs + CW_WARPS - 1) / CW_WARPS * a.n_ct;
  a.ldt = ldt;
  a.q = (uint8_t*)q;
  a.amax = (uint32_t*)inv;
  a.fixed = fixed;
  a.status = status;
  const bool jag = offs != nullptr, fnuz = kind == FP8MOE_E4M3FNUZ;
  cudaError_t err;
  if (!fixed) {
    if ((err = cudaMemsetAsync(inv, 0, (size_t)(E * C) * sizeof(float), st)) != cudaSuccess) return err;
    if (a.n_units > 0) {
      err = jag ? launch_amax<true>(a, num_sms, st) : launch_amax<false>(a, num_sms, st);
      if (err != cudaSuccess) return err;
    }
  }
  if (a.n_units > 0) {
    if (jag) {
      err = transpose_out ? launch_cast_k<true, true>(a, fnuz, num_sms, st)
                          : launch_cast_k<true, false>(a, fnuz, num_sms, st);
    } else {
      err = transpose_out ? launch_cast_k<false, true>(a, fnuz, num_sms, st)
                          : launch_cast_k<false, false>(a, fnuz, num_sms, st);
    }
    if (err != cudaSuccess) return err;
  }
  const int64_t n_inv = fixed ? 0 : E * C;
  int64_t n_a = (n_inv + 255) / 256;
  if (n_a > 4 * num_sms) n_a = 4 * num_sms;
  int64_t n_b = 0;
  if (jag && transpose_out) {
    const int64_t slack = C * ((ldt - R) / 16 + 1);
    n_b = (slack + 255) / 256;
    if (n_b > 2 * num_sms) n_b = 2 * num_sms;
  }
  if (n_a + n_b == 0) return cudaSuccess;
  if (fnuz) {
    k_cw_finish<true><<<(unsigned)(n_a + n_b), 256, 0, st>>>(a, n_inv, (int)n_a);
  } else {
    k_cw_finish<false><<<(unsigned)(n_a + n_b), 256, 0, st>>>(a, n_inv, (int)n_a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_colwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs, int transpose_out,
                           int kind, int64_t ldt, void* q, float* inv, int* status, int num_sms, cudaStream_t st) {
  // transposed output (the dgrad operand of dense weights, the wgrad operand
  // of routed rows): one pass
  if (!offs && transpose_out && colwise_cluster_supported(E, R, C))
    return launch_colwise_cluster(x, E, R, C, kind, q, inv, status, num_sms, st);
  if (offs && transpose_out && R > 0 && colwise_cluster_jagged_supported(E, R, C)) {
    // one persistent CTA per SM holding whole group strips; FP8MOE_CW_JAGGED=cluster
    // selects the two-CTA cluster kernel instead (for comparison)
    static const bool cluster = [] {
      const char* v = getenv("FP8MOE_CW_JAGGED");
      return v && strcmp(v, "cluster") == 0;
    }();
    if (cluster) return launch_colwise_cluster_jagged(x, E, R, C, offs, kind, ldt, q, inv, status, num_sms, st);
    return launch_colwise_jagged_ws(x, E, R, C, offs, kind, ldt, q, inv, status, num_sms, st);
  }
  return run_colwise(x, E, R, C, offs, transpose_out, kind, ldt, q, inv, nullptr, status, num_sms, st);
}

cudaError_t launch_colwise_fixed(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs, int kind,
                                 int64_t ldt, void* q, const uint32_t* amax_bits, int* status, int num_sms,
                                 cudaStream_t st) {
  return run_colwise(x, E, R, C, offs, 1, kind, ldt, q, nullptr, amax_bits, status, num_sms, st);
}

}  // namespace fp8moe
