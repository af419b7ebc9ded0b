// Fused FP8 / MXFP8 quantization kernels (sm_103a).
//
// Every kernel reads its bf16 input once from HBM and writes codes and scales
// once: absmax, scale, clamp and cast happen in one pass ("FP8 Training on AMD
// GPUs with TorchTitan and TorchAO", aihirek.info section "A Triton-kernelok
// csökkentették a kvantálás költségét"; aixai.ru section "Три уровня
// оптимизации Triton-ядер": the unfused chain with HBM intermediates is what
// the pages remove).  Transposed outputs are staged through shared memory so
// that global stores are contiguous (same pages: the colwise-scales kernel
// whose lanes wrote K bytes apart).
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "scales.cuh"
#include "tma.cuh"

namespace cg = cooperative_groups;

namespace fp8moe {

FP8MOE_DEV uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

FP8MOE_DEV void cp_async16(void* smem, const void* gmem) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem));
}
FP8MOE_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

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
    build_group_table(gt, sc.offs, sc.E, R, false, status);
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

// ============================================================================
// Colwise (per expert, per column) FP8: a 32-column strip of one group stays
// resident in shared memory between the absmax and the cast.  Strips taller
// than one CTA's shared memory are split over a thread-block cluster whose
// CTAs exchange their partial column maxima through distributed shared
// memory; groups taller than the whole cluster fall back to re-reading the
// overflow from L2.
// ============================================================================
constexpr int CW_COLS = 32, CW_PITCH = 80;      // 64 B of bf16 + 16 B pad per row
constexpr int CW_TCHUNK = 256;                  // rows per transposed output chunk
constexpr int CW_TPITCH = CW_TCHUNK + 16;

struct ColwiseArgs {
  const uint16_t* x;
  int64_t C;
  int64_t R;          // dense: rows per expert; jagged: total rows
  int E;
  const int32_t* offs;  // NULL: dense
  int transpose_out;
  int64_t ldt;        // jagged transposed width
  uint8_t* q;
  float* inv;
  int cap_rows;       // rows of the strip resident per CTA
  int* status;
  // tensorwise mode: the bf16 bit pattern of the whole tensor's maximum
  // replaces the per-column maxima, and no per-column scale is written
  const uint32_t* fixed_amax;
};

template <bool FNUZ>
__global__ void __launch_bounds__(256) k_colwise(ColwiseArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* buf = smem;                                        // cap_rows x CW_PITCH
  uint8_t* tbuf = smem + (size_t)a.cap_rows * CW_PITCH;       // 32 x CW_TPITCH
  __shared__ uint32_t red[256][4];
  __shared__ float s_col[CW_COLS];
  __shared__ uint32_t amax_part[CW_COLS];
  __shared__ int64_t grp[3];                                  // start, end, padded start

  cg::cluster_group cluster = cg::this_cluster();
  const int CL = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t nstrips = (a.C + CW_COLS - 1) / CW_COLS;
  const int64_t unit = blockIdx.x / CL;
  const int e = (int)(unit / nstrips);
  const int64_t c0 = (unit % nstrips) * CW_COLS;
  const int tid = threadIdx.x;

  if (tid < 32) {
    // group bounds and the padded start of group e: warp 0 reads offsets
    // 0..e 32 at a time (coalesced) and scans the 32-padded sizes with
    // shuffles, validating 0 <= start <= end <= R on the way
    int64_t g0 = 0, g1 = 0, P = 0;
    bool bad = false;
    if (a.offs == nullptr) {
      g0 = (int64_t)e * a.R;
      g1 = g0 + a.R;
    } else {
      int64_t carry = 0, prev_end = 0;
      for (int base = 0; base <= e; base += 32) {
        const int j = base + tid;
        const int64_t end = j <= e ? (int64_t)a.offs[j] : 0;
        const int64_t start = __shfl_up_sync(0xffffffffu, end, 1);
        const int64_t st = tid == 0 ? prev_end : start;
        int64_t padded = 0;
        if (j <= e) {
          if (end < st || end > a.R) bad = true;
          if (j < e) padded = (end - st + 31) / 32 * 32;
          if (j == e) {
            g0 = st;
            g1 = end;
          }
        }
        // inclusive scan of padded sizes over the lanes
        int64_t incl = padded;
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += u;
        }
        if (j == e) P = carry + incl - padded;
        carry += __shfl_sync(0xffffffffu, incl, 31);
        prev_end = __shfl_sync(0xffffffffu, end, 31);
      }
      // the lane that held group e has its bounds; share them
      const int owner = e % 32;
      g0 = __shfl_sync(0xffffffffu, g0, owner);
      g1 = __shfl_sync(0xffffffffu, g1, owner);
      P = __shfl_sync(0xffffffffu, P, owner);
      bad = __any_sync(0xffffffffu, bad);
      if (e == a.E - 1 && g1 != a.R) bad = true;
    }
    if (tid == 0) {
      if (bad) {
        set_status(a.status, FP8MOE_ERR_DEVICE_OFFSETS);
        g0 = g1 = P = -1;
      }
      grp[0] = g0;
      grp[1] = g1;
      grp[2] = P;
    }
  }
  __syncthreads();
  if (grp[2] < 0) return;  // invalid offsets: nothing is written (uniform across the cluster)
  const int64_t g0 = grp[0], g1 = grp[1], P = grp[2];
  const int64_t gsz = g1 - g0;
  int64_t per = (gsz + CL - 1) / CL;
  per = (per + 15) / 16 * 16;
  const int64_t rb = g0 + rank * per < g1 ? g0 + rank * per : g1;
  const int64_t re = rb + per < g1 ? rb + per : g1;
  const int64_t nrows = re - rb;
  const int cap = a.cap_rows;
  const int nwin = nrows == 0 ? 1 : (int)((nrows + cap - 1) / cap);

  // ---- phase 1: column absmax over this CTA's rows, window by window ----
  // load mapping: 4 threads per row (16 B each), 64 rows per pass
  const int lsub = tid & 3, lrow = tid >> 2;
  const bool col_ok = c0 + lsub * 8 < a.C;
  uint4 mx = make_uint4(0, 0, 0, 0);
  auto load_window = [&](int w) {
    const int64_t wr0 = rb + (int64_t)w * cap;
    const int64_t wn = (re - wr0) < cap ? (re - wr0) : cap;
    for (int64_t r = lrow; r < wn; r += 64) {
      uint8_t* d = buf + r * CW_PITCH + lsub * 16;
      if (col_ok) {
        cp_async16(d, a.x + (wr0 + r) * a.C + c0 + lsub * 8);
      } else {
        *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_wait_all();
    __syncthreads();
    return wn;
  };
  int64_t wn = 0;
  const bool fixed = a.fixed_amax != nullptr;
  for (int w = 0; w < (fixed ? 0 : nwin); ++w) {
    if (w > 0) __syncthreads();
    wn = load_window(w);
    for (int64_t r = lrow; r < wn; r += 64) {
      const uint4 v = *reinterpret_cast<const uint4*>(buf + r * CW_PITCH + lsub * 16);
      mx.x = __vmaxu2(mx.x, v.x & 0x7FFF7FFFu);
      mx.y = __vmaxu2(mx.y, v.y & 0x7FFF7FFFu);
      mx.z = __vmaxu2(mx.z, v.z & 0x7FFF7FFFu);
      mx.w = __vmaxu2(mx.w, v.w & 0x7FFF7FFFu);
    }
  }
  red[tid][0] = mx.x;
  red[tid][1] = mx.y;
  red[tid][2] = mx.z;
  red[tid][3] = mx.w;
  __syncthreads();
  if (tid < CW_COLS) {
    // column tid lives in thread-sub tid/8, halfword tid%8
    const int sub = tid >> 3, hw = tid & 7;
    uint32_t m = 0;
    for (int k = 0; k < 64; ++k) {
      const uint32_t w2 = red[k * 4 + sub][hw >> 1];
      m = max(m, (hw & 1) ? (w2 >> 16) : (w2 & 0xFFFFu));
    }
    amax_part[tid] = fixed ? *a.fixed_amax : m;
  }
  if (CL > 1 && !fixed) {
    cluster.sync();
    if (tid < CW_COLS) {
      uint32_t m = 0;
      for (int k = 0; k < CL; ++k) m = max(m, *cluster.map_shared_rank(&amax_part[tid], k));
      red[tid][0] = m;
    }
    cluster.sync();
    if (tid < CW_COLS) amax_part[tid] = red[tid][0];
  }
  __syncthreads();
  if (tid < CW_COLS) {
    float s, inv;
    rowwise_scale<FNUZ>(bf16bits_to_float(amax_part[tid]), s, inv);
    s_col[tid] = s;
    if (!fixed && rank == 0 && c0 + tid < a.C) a.inv[(int64_t)e * a.C + c0 + tid] = inv;
  }
  __syncthreads();

  // ---- phase 2: cast and store, last window first (it is still resident) ----
  const int qsub = tid >> 6, qrow = tid & 63;      // quantize mapping: 8 columns (qsub) per 64 threads
  const bool qcol_ok = c0 + qsub * 8 < a.C;
  float sv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sv[i] = s_col[(qsub * 8 + i) & 31];
  for (int w = nwin - 1; w >= 0; --w) {
    if (w != nwin - 1 || fixed) {   // (phase 1 left the last window resident)
      __syncthreads();
      wn = load_window(w);
    }
    const int64_t wr0 = rb + (int64_t)w * cap;
    if (!a.transpose_out) {
      for (int64_t r = qrow; r < wn; r += 64) {
        if (!qcol_ok) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(buf + r * CW_PITCH + qsub * 16);
        uint2 o;
        o.x = enc4<FNUZ>(__fmul_rn(bf16_lo(v.x), sv[0]), __fmul_rn(bf16_hi(v.x), sv[1]),
                         __fmul_rn(bf16_lo(v.y), sv[2]), __fmul_rn(bf16_hi(v.y), sv[3]));
        o.y = enc4<FNUZ>(__fmul_rn(bf16_lo(v.z), sv[4]), __fmul_rn(bf16_hi(v.z), sv[5]),
                         __fmul_rn(bf16_lo(v.w), sv[6]), __fmul_rn(bf16_hi(v.w), sv[7]));
        *reinterpret_cast<uint2*>(a.q + (wr0 + r) * a.C + c0 + qsub * 8) = o;
      }
      continue;
    }
    // transposed: chunks of CW_TCHUNK rows through the byte-transposed tbuf
    for (int64_t t0 = 0; t0 < wn; t0 += CW_TCHUNK) {
      const int64_t tn = (wn - t0) < CW_TCHUNK ? (wn - t0) : CW_TCHUNK;
      __syncthreads();
      {
        // 4 consecutive rows x 8 columns per thread: each column's 4 codes
        // go to the transposed tile as one word (consecutive words across a
        // warp: conflict-free); rows past tn encode zeros that are never
        // copied out
        const int r = qrow * 4;
        if (r < tn) {
          uint32_t col[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = r + k < tn ? *reinterpret_cast<const uint4*>(buf + (t0 + r + k) * CW_PITCH + qsub * 16)
                                       : make_uint4(0, 0, 0, 0);
            const uint32_t o0 = enc4<FNUZ>(__fmul_rn(bf16_lo(v.x), sv[0]), __fmul_rn(bf16_hi(v.x), sv[1]),
                                           __fmul_rn(bf16_lo(v.y), sv[2]), __fmul_rn(bf16_hi(v.y), sv[3]));
            const uint32_t o1 = enc4<FNUZ>(__fmul_rn(bf16_lo(v.z), sv[4]), __fmul_rn(bf16_hi(v.z), sv[5]),
                                           __fmul_rn(bf16_lo(v.w), sv[6]), __fmul_rn(bf16_hi(v.w), sv[7]));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              col[i] |= ((o0 >> (8 * i)) & 0xFFu) << (8 * k);
              col[4 + i] |= ((o1 >> (8 * i)) & 0xFFu) << (8 * k);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) *reinterpret_cast<uint32_t*>(tbuf + (qsub * 8 + i) * CW_TPITCH + r) = col[i];
        }
      }
      __syncthreads();
      // write 32 output rows of tn bytes; tn is a multiple of 16 except at the
      // end of a group, where the tail is written bytewise
      const int64_t row_begin = wr0 + t0 - g0;  // offset inside the group
      const int nv = (int)(tn / 16);
      for (int k = tid; k < CW_COLS * nv; k += 256) {
        const int cc = k / nv, j = k % nv;
        if (c0 + cc >= a.C) continue;
        uint8_t* dst = a.offs == nullptr ? a.q + ((int64_t)e * a.C + c0 + cc) * a.R + row_begin
                                         : a.q + (c0 + cc) * a.ldt + P + row_begin;
        reinterpret_cast<uint4*>(dst)[j] = *reinterpret_cast<const uint4*>(tbuf + cc * CW_TPITCH + j * 16);
      }
      const int tail = (int)(tn - nv * 16);
      for (int k = tid; k < CW_COLS * tail; k += 256) {
        const int cc = k / tail, j = nv * 16 + k % tail;
        if (c0 + cc >= a.C) continue;
        uint8_t* dst = a.offs == nullptr ? a.q + ((int64_t)e * a.C + c0 + cc) * a.R + row_begin
                                         : a.q + (c0 + cc) * a.ldt + P + row_begin;
        dst[j] = tbuf[cc * CW_TPITCH + j];
      }
    }
  }
  // jagged transposed: zero the group's padding columns (and the tail after
  // the last group)
  if (a.transpose_out && a.offs != nullptr && rank == CL - 1) {
    const int64_t pad_end = (e == a.E - 1) ? a.ldt : P + (gsz + 31) / 32 * 32;
    const int64_t pad0 = P + gsz;
    const int64_t npad = pad_end - pad0;
    for (int64_t k = tid; k < CW_COLS * npad; k += 256) {
      const int cc = (int)(k / npad);
      if (c0 + cc < a.C) a.q[(c0 + cc) * a.ldt + pad0 + k % npad] = 0;
    }
  }
  if (CL > 1) cluster.sync();
}

template <typename K>
static cudaError_t launch_colwise_cl8(ColwiseArgs a, K kern, int64_t R, int64_t E, int64_t nstrips, int64_t max_cap,
                                      cudaStream_t st) {
  const int CL = 8;
  const size_t tbytes = (size_t)CW_COLS * CW_TPITCH;
  int64_t cap = (((R + CL - 1) / CL + 15) / 16 * 16 + 63) / 64 * 64;
  if (cap > max_cap) cap = max_cap;
  a.cap_rows = (int)cap;
  const size_t smem = (size_t)cap * CW_PITCH + tbytes;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(E * nstrips * CL));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

static cudaError_t launch_colwise_impl(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                                       int transpose_out, int kind, int64_t ldt, void* q, float* inv,
                                       const uint32_t* fixed_amax, int* status, int max_smem, cudaStream_t st) {
  ColwiseArgs a;
  a.fixed_amax = fixed_amax;
  a.x = (const uint16_t*)x;
  a.C = C;
  a.R = R;
  a.E = (int)E;
  a.offs = offs;
  a.transpose_out = transpose_out;
  a.ldt = ldt;
  a.q = (uint8_t*)q;
  a.inv = inv;
  a.status = status;
  const int64_t nstrips = (C + CW_COLS - 1) / CW_COLS;
  if (E == 0 || nstrips == 0) return cudaSuccess;
  const size_t fixed = sizeof(uint32_t) * 256 * 4 + 1024;  // static shared memory + slack
  const size_t tbytes = (size_t)CW_COLS * CW_TPITCH;
  const int64_t max_cap = (int64_t)((max_smem - fixed - tbytes) / CW_PITCH) / 64 * 64;
  // ~640 resident rows per CTA keeps 3+ CTAs per SM, so one CTA's loads overlap
  // another's casts and stores; taller strips are split over a cluster.
  constexpr int64_t kTargetRows = 640;
  int CL = 1;
  int64_t cap;
  if (offs == nullptr) {
    while (CL < 16 && (R + CL - 1) / CL > kTargetRows) CL *= 2;
    const int64_t per = ((R + CL - 1) / CL + 15) / 16 * 16;
    cap = (per + 63) / 64 * 64;
  } else {
    // jagged: groups up to ~3x the average size stay single-pass
    const int64_t avg = R / (E > 0 ? E : 1);
    while (CL < 8 && 3 * avg > CL * kTargetRows) CL *= 2;
    cap = kTargetRows;
  }
  if (cap > max_cap) cap = max_cap;
  if (cap < 64) cap = 64;
  a.cap_rows = (int)cap;
  const size_t smem = (size_t)cap * CW_PITCH + tbytes;
  auto kern = kind == FP8MOE_E4M3FNUZ ? k_colwise<true> : k_colwise<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (CL > 8) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(E * nstrips * CL));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (CL > 8) {
    // a 16-CTA cluster may not fit next to other work; fall back to 8 with more rows each
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg) != cudaSuccess || ncl < 1) {
      (void)cudaGetLastError();
      return launch_colwise_cl8(a, kern, R, E, nstrips, max_cap, st);
    }
  }
  return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_colwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                           int transpose_out, int kind, int64_t ldt, void* q, float* inv, int* status,
                           int max_smem, cudaStream_t st) {
  return launch_colwise_impl(x, E, R, C, offs, transpose_out, kind, ldt, q, inv, nullptr, status, max_smem, st);
}

cudaError_t launch_colwise_fixed(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs, int kind,
                                 int64_t ldt, void* q, const uint32_t* amax_bits, int* status, int max_smem,
                                 cudaStream_t st) {
  return launch_colwise_impl(x, E, R, C, offs, 1, kind, ldt, q, nullptr, amax_bits, status, max_smem, st);
}

}  // namespace fp8moe
