// Blockwise FP8 quantization: one fp32 scale per tile ("FP8-обучение на
// AMD", section "Скейлы: от тензора до микроблока": a scale per tile of fixed
// size, between rowwise and MXFP8).  The tile arithmetic is the rowwise one
// (s = fp8_max / max(amax, 1e-12), q = enc(x * s), scale_inv = 1 / s, fp32).
//   k_bw_rows    1 x 128 tiles along the rows of x [R, C]: a half-warp per
//                tile, scales [C/128, R] (tile-index major);
//   k_bw_weight  128 x 128 tiles of w [E, N, K]: a CTA per tile, codes in
//                w's layout and / or transposed [E, K, N] (the dgrad
//                operand) from one read, scales [E, N/128, K/128];
//   k_bw_tokens  128 x 1 tiles along the routed tokens of x [M, C], cut per
//                group (32-multiple offsets), codes transposed [C, M],
//                scales [blocks, C].
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "scales.cuh"

namespace fp8moe {
namespace {

constexpr int TILE = 128;

// max over the 16 lanes of a half-warp
FP8MOE_DEV uint32_t half_max(uint32_t m, unsigned mask) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(mask, m, o));
  return m;
}

// One row per half-warp, 4 tiles in flight per lane.
template <bool FNUZ>
__global__ void __launch_bounds__(256) k_bw_rows(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                 uint8_t* __restrict__ q, float* __restrict__ inv) {
  const int half = threadIdx.x >> 4, hl = threadIdx.x & 15;
  const int64_t r = (int64_t)blockIdx.x * 16 + half;
  if (r >= R) return;  // the whole half-warp leaves together
  const unsigned mask = 0xFFFFu << (threadIdx.x & 16);
  const int nb = (int)(C / TILE);
  const uint16_t* xr = x + r * C + hl * 8;
  uint8_t* qr = q + r * C + hl * 8;
  for (int b0 = 0; b0 < nb; b0 += 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = b0 + u < nb ? ld_nc16(xr + (b0 + u) * TILE) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (b0 + u >= nb) break;
      const uint32_t m = half_max(absmax8_bits(v[u]), mask);
      float s, iv;
      rowwise_scale<FNUZ>(bf16bits_to_float(m), s, iv);
      *reinterpret_cast<uint2*>(qr + (b0 + u) * TILE) = enc8_bf16<FNUZ>(v[u], s);
      if (hl == 0) inv[(int64_t)(b0 + u) * R + r] = iv;
    }
  }
}

// A 128 x 128 tile per CTA; thread t holds rows 8*(t/16) .. +7 and columns
// 8*(t%16) .. +7 of the tile.
template <bool FNUZ>
__global__ void __launch_bounds__(256) k_bw_weight(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                   uint8_t* __restrict__ q, uint8_t* __restrict__ qt,
                                                   float* __restrict__ inv) {
  __shared__ uint32_t red[8];
  const int64_t nkb = K / TILE, nnb = N / TILE;
  const int64_t tile = blockIdx.x;
  const int64_t e = tile / (nnb * nkb);
  const int64_t nb = (tile / nkb) % nnb, kb = tile % nkb;
  const int rg = threadIdx.x >> 4, cg = threadIdx.x & 15;
  const int64_t row0 = nb * TILE + rg * 8, col0 = kb * TILE + cg * 8;
  const uint16_t* src = w + (e * N + row0) * K + col0;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_nc16(src + i * K);
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, absmax8_bits(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) m = max(m, red[i]);
  float s, iv;
  rowwise_scale<FNUZ>(bf16bits_to_float(m), s, iv);
  if (threadIdx.x == 0) inv[tile] = iv;
  uint32_t w0[8], w1[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint2 o = enc8_bf16<FNUZ>(v[i], s);
    w0[i] = o.x;
    w1[i] = o.y;
  }
  if (q) {
    uint8_t* dst = q + (e * N + row0) * K + col0;
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(dst + i * K) = make_uint2(w0[i], w1[i]);
  }
  if (qt) {
    // column j of the thread's 8 x 8 block is 8 consecutive bytes of row
    // col0 + j of the transposed weight
    uint8_t* dst = qt + (e * K + col0) * N + row0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t* W = h ? w1 : w0;
      uint32_t lo[4], hi[4];
      transpose4x4(W[0], W[1], W[2], W[3], lo);
      transpose4x4(W[4], W[5], W[6], W[7], hi);
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<uint2*>(dst + (h * 4 + j) * N) = make_uint2(lo[j], hi[j]);
    }
  }
}

// Units of one token block (<= 128 rows of one group) x 128 columns; a
// persistent CTA builds the group table once and loops over units.  Warp w:
// rows 32*(w&3) .. +31 of the block, columns 64*(w>>2) .. +63; lane: 8 rows x
// 8 columns.
template <bool FNUZ>
__global__ void __launch_bounds__(256, 4) k_bw_tokens(const uint16_t* __restrict__ x, int64_t M, int64_t C,
                                                   const int32_t* __restrict__ offs, int E, int n_ct,
                                                   uint8_t* __restrict__ qt, float* __restrict__ inv, int* status) {
  __shared__ GroupTable gt;
  __shared__ uint4 red[4][2][8];
  build_group_table(gt, offs, E, M, GT_BLK128, status);
  if (gt.bad) return;
  const int64_t last = gt.end[E - 1] - (E > 1 ? gt.end[E - 2] : 0);
  const int64_t total = gt.pad[E - 1] + (last + TILE - 1) / TILE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rq4 = warp & 3, ch = warp >> 2, cl = lane & 7, rq = lane >> 3;
  for (int64_t u = blockIdx.x; u < total * n_ct; u += gridDim.x) {
    const int64_t blk = u / n_ct;
    const int ct = (int)(u % n_ct);
    // owner: the last group whose first block is <= blk
    int lo = 0, hi = E - 1, g = 0;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (gt.pad[mid] <= blk) {
        g = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    const int64_t r0 = (g == 0 ? 0 : gt.end[g - 1]) + (blk - gt.pad[g]) * TILE;
    const int64_t r1 = min(gt.end[g], r0 + TILE);
    const int64_t c = (int64_t)ct * TILE + ch * 64 + cl * 8;
    const int64_t rr = r0 + rq4 * 32 + rq * 8;
    // block sizes are multiples of 32: a lane's 8 rows are all in or all out
    const bool rows_ok = rr < r1, col_ok = c < C;
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = rows_ok && col_ok ? ld_nc16(x + (rr + k) * C + c) : make_uint4(0, 0, 0, 0);
    uint32_t m[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      m[0] = umax16x2(m[0], v[k].x & 0x7FFF7FFFu);
      m[1] = umax16x2(m[1], v[k].y & 0x7FFF7FFFu);
      m[2] = umax16x2(m[2], v[k].z & 0x7FFF7FFFu);
      m[3] = umax16x2(m[3], v[k].w & 0x7FFF7FFFu);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[i] = umax16x2(m[i], __shfl_xor_sync(0xffffffffu, m[i], 8));
      m[i] = umax16x2(m[i], __shfl_xor_sync(0xffffffffu, m[i], 16));
    }
    __syncthreads();  // the previous unit's reads of red are done
    if (rq == 0) red[rq4][ch][cl] = make_uint4(m[0], m[1], m[2], m[3]);
    __syncthreads();
    uint32_t cm[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t* p0 = reinterpret_cast<const uint32_t*>(&red[0][ch][cl]);
      const uint32_t* p1 = reinterpret_cast<const uint32_t*>(&red[1][ch][cl]);
      const uint32_t* p2 = reinterpret_cast<const uint32_t*>(&red[2][ch][cl]);
      const uint32_t* p3 = reinterpret_cast<const uint32_t*>(&red[3][ch][cl]);
      cm[i] = umax16x2(umax16x2(p0[i], p1[i]), umax16x2(p2[i], p3[i]));
    }
    float sv[8], iv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      rowwise_scale<FNUZ>(bf16bits_to_float(cm[i] & 0xFFFFu), sv[2 * i], iv[2 * i]);
      rowwise_scale<FNUZ>(bf16bits_to_float(cm[i] >> 16), sv[2 * i + 1], iv[2 * i + 1]);
    }
    if (rq4 == 0 && rq == 0 && col_ok) {
      float* ip = inv + blk * C + c;
      *reinterpret_cast<float4*>(ip) = make_float4(iv[0], iv[1], iv[2], iv[3]);
      *reinterpret_cast<float4*>(ip + 4) = make_float4(iv[4], iv[5], iv[6], iv[7]);
    }
    if (!rows_ok || !col_ok) continue;
#pragma unroll
    for (int t = 0; t < 8; ++t) sv[t] = enc_mul<FNUZ>(sv[t]);
    uint32_t w0[8], w1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      w0[k] = enc4_pre<FNUZ>(__fmul_rn(bf16_lo(v[k].x), sv[0]), __fmul_rn(bf16_hi(v[k].x), sv[1]),
                         __fmul_rn(bf16_lo(v[k].y), sv[2]), __fmul_rn(bf16_hi(v[k].y), sv[3]));
      w1[k] = enc4_pre<FNUZ>(__fmul_rn(bf16_lo(v[k].z), sv[4]), __fmul_rn(bf16_hi(v[k].z), sv[5]),
                         __fmul_rn(bf16_lo(v[k].w), sv[6]), __fmul_rn(bf16_hi(v[k].w), sv[7]));
    }
    uint8_t* dst = qt + c * M + rr;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t* W = h ? w1 : w0;
      uint32_t a[4], b[4];
      transpose4x4(W[0], W[1], W[2], W[3], a);
      transpose4x4(W[4], W[5], W[6], W[7], b);
#pragma unroll
      for (int j = 0; j < 4; ++j) *reinterpret_cast<uint2*>(dst + (h * 4 + j) * M) = make_uint2(a[j], b[j]);
    }
  }
}

}  // namespace

cudaError_t launch_bw_rows(const void* x, int64_t R, int64_t C, int kind, void* q, float* inv, cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((R + 15) / 16);
  if (kind == FP8MOE_E4M3FNUZ) {
    k_bw_rows<true><<<grid, 256, 0, st>>>((const uint16_t*)x, R, C, (uint8_t*)q, inv);
  } else {
    k_bw_rows<false><<<grid, 256, 0, st>>>((const uint16_t*)x, R, C, (uint8_t*)q, inv);
  }
  return cudaGetLastError();
}

cudaError_t launch_bw_weight(const void* w, int64_t E, int64_t N, int64_t K, int kind, void* q, void* qt,
                             float* inv, cudaStream_t st) {
  const int64_t tiles = E * (N / TILE) * (K / TILE);
  if (tiles == 0) return cudaSuccess;
  if (kind == FP8MOE_E4M3FNUZ) {
    k_bw_weight<true><<<(unsigned)tiles, 256, 0, st>>>((const uint16_t*)w, N, K, (uint8_t*)q, (uint8_t*)qt, inv);
  } else {
    k_bw_weight<false><<<(unsigned)tiles, 256, 0, st>>>((const uint16_t*)w, N, K, (uint8_t*)q, (uint8_t*)qt, inv);
  }
  return cudaGetLastError();
}

cudaError_t launch_bw_tokens(const void* x, int64_t M, int64_t C, const int32_t* offs, int64_t E, int kind,
                             void* qt, float* inv, int num_sms, int* status, cudaStream_t st) {
  if (C == 0) return cudaSuccess;
  const int n_ct = (int)((C + TILE - 1) / TILE);
  // persistent CTAs, one wave: as many as are resident, at most one per unit
  // (the unit count is an upper bound here; the exact one needs the offsets)
  static std::atomic<int> per_sm_fn{0}, per_sm_fnuz{0};
  const bool fnuz = kind == FP8MOE_E4M3FNUZ;
  const int per_sm = fnuz ? blocks_per_sm(per_sm_fnuz, k_bw_tokens<true>, 256, 0, 4)
                          : blocks_per_sm(per_sm_fn, k_bw_tokens<false>, 256, 0, 4);
  const int64_t units = ((M + TILE - 1) / TILE + E) * n_ct;
  const int64_t cap = (int64_t)per_sm * num_sms;
  const int64_t blocks = units < cap ? units : cap;
  if (fnuz) {
    k_bw_tokens<true><<<(unsigned)blocks, 256, 0, st>>>((const uint16_t*)x, M, C, offs, (int)E, n_ct,
                                                        (uint8_t*)qt, inv, status);
  } else {
    k_bw_tokens<false><<<(unsigned)blocks, 256, 0, st>>>((const uint16_t*)x, M, C, offs, (int)E, n_ct,
                                                         (uint8_t*)qt, inv, status);
  }
  return cudaGetLastError();
}

}  // namespace fp8moe
