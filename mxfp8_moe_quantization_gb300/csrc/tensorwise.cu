// Tensorwise FP8 quantization: one scale for a whole tensor, the coarsest of
// the four scaling granularities ("FP8-обучение на AMD", section "Скейлы: от
// тензора до микроблока").  The arithmetic is the rowwise one (fp32:
// s = fmax / max(amax, 1e-12), q = RNE_sat(x * s), stored inv = 1 / s) with
// the absolute maximum taken over every element.
//
// Three stream-ordered launches around the caller's one-float scale buffer,
// which holds the maximum's bf16 bit pattern until the last one replaces it
// by the dequantization scale:
//   1. k_tw_amax: grid-stride 16-byte loads (four in flight per thread; six
//      256-thread CTAs per SM, the grid one wave of them),
//      warp / block maxima, one atomicMax per block (bit patterns of
//      non-negative values order like the values);
//   2. the cast: k_tw_cast for the plain layout, or the colwise kernel in its
//      fixed-scale mode for the transposed / jagged layouts;
//   3. k_tw_finalize: one thread writes fl(1 / s).
#include "common.cuh"
#include "launch.h"

namespace fp8moe {

namespace {

FP8MOE_DEV uint4 ld_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Four 16-byte chunks in flight per thread and loop trip.
constexpr int TW_U = 4;

__global__ void __launch_bounds__(256, 6) k_tw_amax(const uint16_t* __restrict__ x, int64_t n,
                                                 uint32_t* __restrict__ amax_bits) {
  __shared__ uint32_t wmax[8];
  const int64_t nch = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t m = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nch; i += stride * TW_U) {
    uint4 v[TW_U];
    if (i + (TW_U - 1) * stride < nch) {  // all in range: unconditional loads, all in flight
#pragma unroll
      for (int u = 0; u < TW_U; ++u) v[u] = ld_nc(x + (i + u * stride) * 8);
    } else {
#pragma unroll
      for (int u = 0; u < TW_U; ++u)
        v[u] = i + u * stride < nch ? ld_nc(x + (i + u * stride) * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < TW_U; ++u) m = max(m, absmax8_bits(v[u]));
  }
  // tail elements (n % 8)
  for (int64_t i = nch * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    m = max(m, (uint32_t)x[i] & 0x7FFFu);
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, wmax[w]);
    if (m) atomicMax(amax_bits, m);
  }
}

template <bool FNUZ>
__global__ void __launch_bounds__(256, 6) k_tw_cast(const uint16_t* __restrict__ x, int64_t n, uint8_t* __restrict__ q,
                                                 const uint32_t* __restrict__ amax_bits) {
  float s, inv;
  rowwise_scale<FNUZ>(bf16bits_to_float(*amax_bits), s, inv);
  const int64_t nch = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // chunks in the reverse of the amax pass's order: the first reads find
  // the tensor's tail still in L2
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nch; i += stride * TW_U) {
    uint4 v[TW_U];
    if (i + (TW_U - 1) * stride < nch) {
#pragma unroll
      for (int u = 0; u < TW_U; ++u) v[u] = ld_nc(x + (nch - 1 - (i + u * stride)) * 8);
#pragma unroll
      for (int u = 0; u < TW_U; ++u)
        *reinterpret_cast<uint2*>(q + (nch - 1 - (i + u * stride)) * 8) = enc8_bf16<FNUZ>(v[u], s);
    } else {
#pragma unroll
      for (int u = 0; u < TW_U; ++u)
        if (i + u * stride < nch) {
          v[u] = ld_nc(x + (nch - 1 - (i + u * stride)) * 8);
          *reinterpret_cast<uint2*>(q + (nch - 1 - (i + u * stride)) * 8) = enc8_bf16<FNUZ>(v[u], s);
        }
    }
  }
  for (int64_t i = nch * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    q[i] = (uint8_t)(enc2<FNUZ>(__fmul_rn(bf16bits_to_float(x[i]), s), 0.0f) & 0xFFu);
}

template <bool FNUZ>
__global__ void k_tw_finalize(float* scale) {
  float s, inv;
  rowwise_scale<FNUZ>(bf16bits_to_float(*reinterpret_cast<const uint32_t*>(scale)), s, inv);
  *scale = inv;
}

// CTAs of `kern` resident on the whole GPU at once: the grid-stride kernels
// run as a single wave (a second wave would repeat the ramp and the tail)
template <typename K>
int resident_ctas(K kern, int num_sms) {
  int per = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, 256, 0) != cudaSuccess || per < 1) {
    (void)cudaGetLastError();
    per = 4;
  }
  return per * num_sms;
}

}  // namespace

cudaError_t launch_tensorwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                              int transpose_out, int kind, void* q, float* scale_inv, int num_sms, int* status,
                              cudaStream_t st) {
  const int64_t n = (offs ? 1 : E) * R * C;
  cudaError_t e = cudaMemsetAsync(scale_inv, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  const bool fnuz = kind == FP8MOE_E4M3FNUZ;
  static int cap_amax = 0, cap_fn = 0, cap_fnuz = 0;
  if (!cap_amax) {
    cap_amax = resident_ctas(k_tw_amax, num_sms);
    cap_fn = resident_ctas(k_tw_cast<false>, num_sms);
    cap_fnuz = resident_ctas(k_tw_cast<true>, num_sms);
  }
  if (n > 0) {
    const int64_t want = (n / 8 + 255) / 256;
    auto grid = [&](int cap) -> unsigned { return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap)); };
    k_tw_amax<<<grid(cap_amax), 256, 0, st>>>((const uint16_t*)x, n, (uint32_t*)scale_inv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (!transpose_out) {
      if (fnuz) {
        k_tw_cast<true><<<grid(cap_fnuz), 256, 0, st>>>((const uint16_t*)x, n, (uint8_t*)q,
                                                        (const uint32_t*)scale_inv);
      } else {
        k_tw_cast<false><<<grid(cap_fn), 256, 0, st>>>((const uint16_t*)x, n, (uint8_t*)q,
                                                       (const uint32_t*)scale_inv);
      }
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  if (transpose_out) {
    // the transposed (and, jagged, group-padded) layout of the colwise
    // kernel, with the tensor's maximum in place of per-column maxima
    const int64_t ldt = offs ? fp8moe_jagged_t_cols(R, E) : 0;
    e = launch_colwise_fixed(x, E, R, C, offs, kind, ldt, q, (const uint32_t*)scale_inv, status, num_sms, st);
    if (e != cudaSuccess) return e;
  }
  if (fnuz) {
    k_tw_finalize<true><<<1, 1, 0, st>>>(scale_inv);
  } else {
    k_tw_finalize<false><<<1, 1, 0, st>>>(scale_inv);
  }
  return cudaGetLastError();
}

}  // namespace fp8moe
