// Token routing into expert groups (permute) and back (unpermute): the step
// that puts routed rows at the offsets the grouped GEMM consumes ("FP8-обучение
// на AMD", section "MoE: почему DeepSeek-V3 ломал пайплайн": tokens are
// routed by offsets), with every group padded to a multiple of 32 rows as the
// MXFP8 layer configurations are.
//
// Permute, four launches, no host synchronization:
//   1. k_route_count: per chunk of 1024 (token, slot) entries, a shared-memory
//      histogram of expert ids -> counts[chunk][e]; ids out of range set the
//      device status and are skipped;
//   2. k_route_scan (one CTA): per expert, the exclusive prefix over chunks
//      and the padded group starts; offs; the end of each group's real rows;
//   3. k_route_scatter: warp 0 ranks the chunk's entries stably (a warp-wide
//      match of expert ids, per-expert running counts in shared memory), then
//      all warps copy the routed rows with 16-byte accesses, optionally
//      weighted (bf16(fp32(w) * x));
//   4. k_route_zero: the padding rows of every group (and the slack of the
//      last one) are zeroed.
// Unpermute: one warp per token sums its k rows in slot order in fp32.
#include "common.cuh"
#include "launch.h"

namespace fp8moe {

namespace {

constexpr int RT_CHUNK = 1024;
constexpr int RT_MAXE = 1024;

FP8MOE_DEV uint32_t bf16x2_scaled(uint32_t v, float w) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(bf16_lo(v), w), __fmul_rn(bf16_hi(v), w));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(256) k_route_count(const int32_t* __restrict__ idx, int64_t n, int E,
                                                     int32_t* __restrict__ counts, int* status) {
  __shared__ int hist[RT_MAXE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t c0 = (int64_t)blockIdx.x * RT_CHUNK;
  for (int i = threadIdx.x; i < RT_CHUNK && c0 + i < n; i += blockDim.x) {
    const int e = idx[c0 + i];
    if (e < 0 || e >= E) {
      set_status(status, FP8MOE_ERR_DEVICE_OFFSETS);
      continue;
    }
    atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// counts [nchunks][E] -> in place the first row of each (chunk, expert);
// offs [E]; real_end [E] (end of the real rows of each group)
__global__ void __launch_bounds__(1024) k_route_scan(int32_t* __restrict__ counts, int nchunks, int E,
                                                     int64_t rows, int32_t* __restrict__ offs,
                                                     int32_t* __restrict__ real_end) {
  __shared__ int64_t part[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // one expert per thread (E <= 1024): its total and the prefix over chunks
  int64_t total = 0;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = counts[(int64_t)c * E + tid];
      counts[(int64_t)c * E + tid] = (int)total;
      total += v;
    }
  }
  const int64_t padded = (total + 31) / 32 * 32;
  // block-wide exclusive scan of the padded sizes
  int64_t incl = padded;
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) part[warp] = incl;
  __syncthreads();
  int64_t base = 0;
  for (int w = 0; w < warp; ++w) base += part[w];
  const int64_t start = base + incl - padded;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) counts[(int64_t)c * E + tid] += (int)start;
    offs[tid] = tid == E - 1 ? (int32_t)rows : (int32_t)(start + padded);
    real_end[tid] = (int32_t)(start + total);
  }
}

__global__ void __launch_bounds__(256) k_route_scatter(const uint16_t* __restrict__ x, int64_t H,
                                                       const int32_t* __restrict__ idx, const float* __restrict__ w,
                                                       int64_t n, int k, int E, const int32_t* __restrict__ first,
                                                       uint16_t* __restrict__ a, int32_t* __restrict__ row_of) {
  __shared__ int next[RT_MAXE];
  __shared__ int dst[RT_CHUNK];
  const int64_t c0 = (int64_t)blockIdx.x * RT_CHUNK;
  for (int e = threadIdx.x; e < E; e += blockDim.x) next[e] = first[(int64_t)blockIdx.x * E + e];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cn = (int)((n - c0) < RT_CHUNK ? (n - c0) : RT_CHUNK);
  if (warp == 0) {
    // stable ranks: batches of 32 entries in order; lanes with the same
    // expert take consecutive rows in lane order
    for (int b = 0; b < cn; b += 32) {
      const int i = b + lane;
      int e = i < cn ? idx[c0 + i] : -1;
      if (e >= E) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int row = -1;
      if (e >= 0) row = next[e] + rank;
      __syncwarp();
      if (e >= 0 && rank == 0) next[e] += __popc(peers);
      __syncwarp();
      if (i < cn) {
        dst[i] = row;
        row_of[c0 + i] = row;
      }
    }
  }
  __syncthreads();
  // copy: one warp per routed row, 16 bytes per lane access
  const int64_t nv = H / 8;
  for (int i = warp; i < cn; i += blockDim.x >> 5) {
    const int r = dst[i];
    if (r < 0) continue;
    const int64_t t = (c0 + i) / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4* out = reinterpret_cast<uint4*>(a + (int64_t)r * H);
    if (w == nullptr) {
      for (int64_t v = lane; v < nv; v += 32) out[v] = src[v];
    } else {
      const float wt = w[c0 + i];
      for (int64_t v = lane; v < nv; v += 32) {
        const uint4 s = src[v];
        out[v] = make_uint4(bf16x2_scaled(s.x, wt), bf16x2_scaled(s.y, wt), bf16x2_scaled(s.z, wt),
                            bf16x2_scaled(s.w, wt));
      }
    }
  }
}

// zero rows [real_end[e], offs[e]) of every group: one CTA per group
__global__ void __launch_bounds__(256) k_route_zero(uint16_t* __restrict__ a, int64_t H,
                                                    const int32_t* __restrict__ offs,
                                                    const int32_t* __restrict__ real_end) {
  const int e = blockIdx.x;
  const int64_t r0 = real_end[e], r1 = offs[e];
  const int64_t nv = (r1 - r0) * H / 8;
  uint4* p = reinterpret_cast<uint4*>(a + r0 * H);
  for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) p[v] = make_uint4(0, 0, 0, 0);
}

__global__ void __launch_bounds__(256) k_route_unpermute(const uint16_t* __restrict__ y, int64_t N,
                                                         const int32_t* __restrict__ row_of,
                                                         const float* __restrict__ w, int64_t T, int k,
                                                         uint16_t* __restrict__ out) {
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int64_t nv = N / 8;
  for (int64_t v = lane; v < nv; v += 32) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j = 0; j < k; ++j) {
      const int r = row_of[t * k + j];
      if (r < 0) continue;
      const float wt = w ? w[t * k + j] : 1.0f;
      const uint4 s = reinterpret_cast<const uint4*>(y + (int64_t)r * N)[v];
      const uint32_t q[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        acc[2 * h] = __fadd_rn(acc[2 * h], w ? __fmul_rn(wt, bf16_lo(q[h])) : bf16_lo(q[h]));
        acc[2 * h + 1] = __fadd_rn(acc[2 * h + 1], w ? __fmul_rn(wt, bf16_hi(q[h])) : bf16_hi(q[h]));
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * h], acc[2 * h + 1]);
      o[h] = *reinterpret_cast<const uint32_t*>(&b);
    }
    reinterpret_cast<uint4*>(out + t * N)[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

int64_t route_workspace_bytes(int64_t T, int64_t k, int64_t E) {
  const int64_t n = T * k;
  const int64_t nchunks = (n + RT_CHUNK - 1) / RT_CHUNK;
  return (nchunks * E + E) * (int64_t)sizeof(int32_t);
}

cudaError_t launch_route_permute(const void* x, int64_t T, int64_t H, const int32_t* idx, const float* w, int64_t k,
                                 int64_t E, int64_t rows, void* a, int32_t* offs, int32_t* row_of, void* workspace,
                                 int* status, cudaStream_t st) {
  if (E < 1 || E > RT_MAXE) return cudaErrorInvalidValue;
  const int64_t n = T * k;
  const int64_t nchunks = (n + RT_CHUNK - 1) / RT_CHUNK;
  int32_t* counts = (int32_t*)workspace;
  int32_t* real_end = counts + nchunks * E;
  cudaError_t e;
  if (nchunks > 0) {
    k_route_count<<<(unsigned)nchunks, 256, 0, st>>>(idx, n, (int)E, counts, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_route_scan<<<1, 1024, 0, st>>>(counts, (int)nchunks, (int)E, rows, offs, real_end);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nchunks > 0) {
    k_route_scatter<<<(unsigned)nchunks, 256, 0, st>>>((const uint16_t*)x, H, idx, w, n, (int)k, (int)E, counts,
                                                        (uint16_t*)a, row_of);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_route_zero<<<(unsigned)E, 256, 0, st>>>((uint16_t*)a, H, offs, real_end);
  return cudaGetLastError();
}

cudaError_t launch_route_unpermute(const void* y, int64_t N, const int32_t* row_of, const float* w, int64_t T,
                                   int64_t k, void* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int64_t blocks = (T + 7) / 8;
  k_route_unpermute<<<(unsigned)blocks, 256, 0, st>>>((const uint16_t*)y, N, row_of, w, T, (int)k, (uint16_t*)out);
  return cudaGetLastError();
}

}  // namespace fp8moe
