// Fused FP8 / MXFP8 quantization kernels (sm_103a).
//
// Every kernel reads its bf16 input once from HBM and writes codes and scales
// once: absmax, scale, clamp and cast happen in one pass ("FP8 Training on AMD
// GPUs with TorchTitan and TorchAO", aihirek.info section "A Triton-kernelok
// csökkentették a kvantálás költségét"; aixai.ru section "Три уровня
// оптимизации Triton-ядер": the unfused chain with HBM intermediates is what
// the pages remove).  The colwise kernels live in colwise.cu.

#include "common.cuh"
#include "launch.h"
#include "scales.cuh"

namespace fp8moe {

FP8MOE_DEV uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}


// ============================================================================
// Rowwise: TPR threads per row, each holding V 16-byte chunks in registers.
// ============================================================================
template <int TPR, int V, bool FNUZ>
__global__ void __launch_bounds__(256) k_quant_rowwise(const uint16_t* __restrict__ x, int64_t R,
                                                       int C, int64_t ldx, uint8_t* __restrict__ q,
                                                       float* __restrict__ inv_out) {
  constexpr int RPB = 256 / TPR;
  const int t = threadIdx.x % TPR;
  const int rloc = threadIdx.x / TPR;
  const int64_t row = (int64_t)blockIdx.x * RPB + rloc;
  const bool active = row < R;
  const int nch = C / 8;
  const uint16_t* xr = x + (active ? row : 0) * ldx;
  uint4 v[V];
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int ch = t + i * TPR;
    if (active && ch < nch) {
      v[i] = ld_stream(xr + (int64_t)ch * 8);
    } else {
      v[i] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) m = max(m, absmax8_bits(v[i]));
#pragma unroll
  for (int o = (TPR < 32 ? TPR : 32) / 2; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if constexpr (TPR > 32) {
    __shared__ uint32_t red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    constexpr int WPR = TPR / 32;
    m = 0;
#pragma unroll
    for (int w = 0; w < WPR; ++w) m = max(m, red[rloc * WPR + w]);
  }
  float s, inv;
  rowwise_scale<FNUZ>(bf16bits_to_float(m), s, inv);
  if (!active) return;
  uint8_t* qr = q + row * (int64_t)C;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int ch = t + i * TPR;
    if (ch < nch) *reinterpret_cast<uint2*>(qr + (int64_t)ch * 8) = enc8_bf16<FNUZ>(v[i], s);
  }
  if (t == 0) inv_out[row] = inv;
}

// Rows too long for registers: two passes over the row (the second re-reads
// it from L2), one row per 256-thread block.
template <bool FNUZ>
__global__ void __launch_bounds__(256) k_quant_rowwise_long(const uint16_t* __restrict__ x, int64_t R,
                                                            int C, int64_t ldx, uint8_t* __restrict__ q,
                                                            float* __restrict__ inv_out) {
  const int64_t row = blockIdx.x;
  const uint16_t* xr = x + row * ldx;
  const int nch = C / 8;
  uint32_t m = 0;
  for (int ch = threadIdx.x; ch < nch; ch += 256) m = max(m, absmax8_bits(ld_stream(xr + (int64_t)ch * 8)));
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0;
  for (int w = 0; w < 8; ++w) m = max(m, red[w]);
  float s, inv;
  rowwise_scale<FNUZ>(bf16bits_to_float(m), s, inv);
  uint8_t* qr = q + row * (int64_t)C;
  for (int ch = threadIdx.x; ch < nch; ch += 256) {
    uint4 v = *reinterpret_cast<const uint4*>(xr + (int64_t)ch * 8);
    *reinterpret_cast<uint2*>(qr + (int64_t)ch * 8) = enc8_bf16<FNUZ>(v, s);
  }
  if (threadIdx.x == 0) inv_out[row] = inv;
}

template <int TPR, int V, bool FNUZ>
static cudaError_t launch_rowwise_t(const void* x, int64_t R, int C, int64_t ldx, void* q, float* inv,
                                    cudaStream_t st) {
  constexpr int RPB = 256 / TPR;
  const int64_t blocks = (R + RPB - 1) / RPB;
  k_quant_rowwise<TPR, V, FNUZ><<<(unsigned)blocks, 256, 0, st>>>(
      (const uint16_t*)x, R, C, ldx, (uint8_t*)q, inv);
  return cudaGetLastError();
}

template <bool FNUZ>
static cudaError_t launch_rowwise_k(const void* x, int64_t R, int C, int64_t ldx, void* q, float* inv,
                                    cudaStream_t st) {
  const int nch = C / 8;
  int tpr = 32;
  while (tpr < 256 && tpr * 8 < nch) tpr *= 2;
  const int v = (nch + tpr - 1) / tpr;
#define FP8MOE_RW(T, VV) \
  if (tpr == T && v <= VV) return launch_rowwise_t<T, VV, FNUZ>(x, R, C, ldx, q, inv, st);
  FP8MOE_RW(32, 1) FP8MOE_RW(32, 2) FP8MOE_RW(32, 4) FP8MOE_RW(32, 8)
  FP8MOE_RW(64, 8) FP8MOE_RW(128, 8) FP8MOE_RW(256, 8)
#undef FP8MOE_RW
  k_quant_rowwise_long<FNUZ><<<(unsigned)R, 256, 0, st>>>((const uint16_t*)x, R, C, ldx, (uint8_t*)q, inv);
  return cudaGetLastError();
}

cudaError_t launch_quant_rowwise(const void* x, int64_t R, int64_t C, int64_t ldx, int kind, void* q,
                                 float* inv, cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  return kind == FP8MOE_E4M3FNUZ ? launch_rowwise_k<true>(x, R, (int)C, ldx, q, inv, st)
                                 : launch_rowwise_k<false>(x, R, (int)C, ldx, q, inv, st);
}

// ============================================================================
// MXFP8 dim0: four lanes per 32-element block, 8 bf16 (16 bytes) per lane.
// ============================================================================
// IDX32: every chunk index fits 32 bits, so the row / column of a scale come
// from a 32-bit division (a 64-bit division per scale costs a third of the
// kernel's time).  Row-major scales need no division at all.
template <int U, bool IDX32>
__global__ void __launch_bounds__(256) k_mx_dim0(const uint16_t* __restrict__ x, int64_t nch, int64_t R, int64_t C,
                                                 uint8_t* __restrict__ q, ScaleSpec sc, int* status) {
  __shared__ GroupTable gt;
  if (sc.layout == FP8MOE_GROUP_ROWS) {
    build_group_table(gt, sc.offs, sc.E, R, GT_ROWS128, status);
    if (gt.bad) return;
  }
  const int64_t Cs = C / 32, cpr = C / 8;  // scale columns, 16-byte chunks per row
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t warp0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int64_t wb = warp0 * 32 * U; wb < nch; wb += warps_total * 32 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t ch = wb + u * 32 + lane;
      v[u] = ch < nch ? ld_stream(x + ch * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t ch = wb + u * 32 + lane;
      uint32_t m = absmax8_bits(v[u]);
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const int e = e8m0_exponent(m);
      const float p = exp2_neg(e);
      if (ch < nch) {
        *reinterpret_cast<uint2*>(q + ch * 8) = enc8_bf16<false>(v[u], p);
        if ((lane & 3) == 0) {
          int64_t off;
          if (sc.layout == FP8MOE_SCALES_ROWMAJOR) {
            off = ch >> 2;
          } else {
            int64_t row, cb;
            if (IDX32) {
              const uint32_t c32 = (uint32_t)ch, p32 = (uint32_t)cpr;
              const uint32_t r32 = c32 / p32;
              row = r32;
              cb = (c32 - r32 * p32) >> 2;
            } else {
              row = ch / cpr;
              cb = (ch % cpr) >> 2;
            }
            int64_t b = 0;
            if (sc.layout != FP8MOE_GROUP_ROWS) b = IDX32 ? (int64_t)((uint32_t)row / (uint32_t)R) : row / R;
            off = scale_offset(sc, &gt, b, row - b * R, cb, R, Cs);
          }
          sc.p[off] = (uint8_t)(e + 127);
        }
      }
    }
  }
}

cudaError_t launch_mx_dim0(const void* x, int64_t B, int64_t R, int64_t C, void* q, uint8_t* s, int layout,
                           const int32_t* offs, int64_t E, int num_sms, int* status, cudaStream_t st) {
  const int64_t nch = B * R * C / 8;
  if (nch == 0) return cudaSuccess;
  constexpr int U = 4;
  int64_t blocks = (nch + 256 * U - 1) / (256 * U);
  const int64_t cap = (int64_t)num_sms * 8 * 4;
  if (blocks > cap) blocks = cap;
  const ScaleSpec spec = make_spec(s, layout, R, C / 32, offs, E);
  if (nch < ((int64_t)1 << 32)) {
    k_mx_dim0<U, true><<<(unsigned)blocks, 256, 0, st>>>((const uint16_t*)x, nch, R, C, (uint8_t*)q, spec, status);
  } else {
    k_mx_dim0<U, false><<<(unsigned)blocks, 256, 0, st>>>((const uint16_t*)x, nch, R, C, (uint8_t*)q, spec, status);
  }
  return cudaGetLastError();
}

}  // namespace fp8moe
