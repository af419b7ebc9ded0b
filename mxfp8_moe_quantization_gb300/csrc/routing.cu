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
//   3. k_route_rank: per chunk, one warp ranks the entries stably (a warp-wide
//      match of expert ids, per-expert running counts in shared memory) and
//      writes each entry's row;
//   4. k_route_copy: the routed rows, one warp per row over the whole GPU,
//      16-byte accesses, optionally weighted (bf16(fp32(w) * x)), and the
//      padding rows of every group (and the slack of the last one) zeroed.
// Unpermute: one warp per token sums its k rows in slot order in fp32.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace fp8moe {

// Scratch of the routing permute for callers that cannot allocate device
// memory (fp8moe_route_permute_noalloc): a file-scope device array that every
// device loading the library holds until the process exits.  Its size is
// ROUTE_STATIC_SCRATCH_BYTES (1 MiB, declared in include/fp8moe.h as
// FP8MOE_ROUTE_STATIC_SCRATCH_BYTES); all calls on a device share it.
constexpr int64_t ROUTE_STATIC_SCRATCH_BYTES = FP8MOE_ROUTE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) int32_t g_route_scratch[ROUTE_STATIC_SCRATCH_BYTES / 4];

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
// offs [E]; real_end [E] (end of the real rows of each group); pad_prefix
// [E + 1] (padding rows of the groups before e, and the total)
__global__ void __launch_bounds__(1024) k_route_scan(int32_t* __restrict__ counts, int nchunks, int E,
                                                     int64_t rows, int32_t* __restrict__ offs,
                                                     int32_t* __restrict__ real_end, int32_t* __restrict__ pad_prefix) {
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
  const int64_t end = tid == E - 1 ? rows : start + padded;
  if (tid < E) {
    for (int c = 0; c < nchunks; ++c) counts[(int64_t)c * E + tid] += (int)start;
    offs[tid] = (int32_t)end;
    real_end[tid] = (int32_t)(start + total);
  }
  // exclusive scan of the padding row counts
  const int64_t pad = tid < E ? end - (start + total) : 0;
  __syncthreads();
  int64_t pincl = pad;
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, pincl, o);
    if (lane >= o) pincl += u;
  }
  if (lane == 31) part[warp] = pincl;
  __syncthreads();
  int64_t pbase = 0;
  for (int w = 0; w < warp; ++w) pbase += part[w];
  if (tid < E) pad_prefix[tid] = (int32_t)(pbase + pincl - pad);
  if (tid == E - 1) pad_prefix[E] = (int32_t)(pbase + pincl);
}

__global__ void __launch_bounds__(32) k_route_rank(const int32_t* __restrict__ idx, int64_t n, int E,
                                                   const int32_t* __restrict__ first, int32_t* __restrict__ row_of) {
  __shared__ int next[RT_MAXE];
  const int64_t c0 = (int64_t)blockIdx.x * RT_CHUNK;
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) next[e] = first[(int64_t)blockIdx.x * E + e];
  __syncwarp();
  const int cn = (int)((n - c0) < RT_CHUNK ? (n - c0) : RT_CHUNK);
  // the chunk's ids, loaded up front (one per lane and batch)
  int ids[RT_CHUNK / 32];
#pragma unroll
  for (int b = 0; b < RT_CHUNK / 32; ++b) ids[b] = b * 32 + lane < cn ? idx[c0 + b * 32 + lane] : -1;
  // batches of 32 entries in order; lanes with the same expert take
  // consecutive rows in lane order (a stable placement)
#pragma unroll
  for (int bb = 0; bb < RT_CHUNK / 32; ++bb) {
    const int b = bb * 32;
    if (b >= cn) break;
    const int i = b + lane;
    int e = ids[bb];
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int row = -1;
    if (e >= 0) row = next[e] + rank;
    __syncwarp();
    if (e >= 0 && rank == 0) next[e] += __popc(peers);
    __syncwarp();
    if (i < cn) row_of[c0 + i] = row;
  }
}

// one warp per routed row (then one per padding row), 16 bytes per access
__global__ void __launch_bounds__(256) k_route_copy(const uint16_t* __restrict__ x, int64_t H, const float* __restrict__ w,
                                                    int64_t n, int k, int E, const int32_t* __restrict__ row_of,
                                                    const int32_t* __restrict__ real_end,
                                                    const int32_t* __restrict__ pad_prefix, uint16_t* __restrict__ a) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t nv = H / 8;
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < n; i += nw) {
    const int r = row_of[i];
    if (r < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + (i / k) * H);
    uint4* out = reinterpret_cast<uint4*>(a + (int64_t)r * H);
    const float wt = w ? w[i] : 1.0f;
    // four 16-byte loads in flight per lane
    int64_t v = lane;
    for (; v + 96 < nv; v += 128) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = src[v + 32 * u];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        out[v + 32 * u] = w ? make_uint4(bf16x2_scaled(q[u].x, wt), bf16x2_scaled(q[u].y, wt),
                                         bf16x2_scaled(q[u].z, wt), bf16x2_scaled(q[u].w, wt))
                            : q[u];
    }
    for (; v < nv; v += 32) {
      const uint4 q = src[v];
      out[v] = w ? make_uint4(bf16x2_scaled(q.x, wt), bf16x2_scaled(q.y, wt), bf16x2_scaled(q.z, wt),
                              bf16x2_scaled(q.w, wt))
                 : q;
    }
  }
  // padding rows: the p-th one overall belongs to the group g whose
  // pad_prefix[g] <= p < pad_prefix[g + 1], at row real_end[g] + p - pad_prefix[g]
  const int64_t npad = pad_prefix[E];
  for (int64_t pr = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pr < npad; pr += nw) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pad_prefix[mid] <= pr) {
        lo = mid;
      } else {
        hi = mid - 1;
      }
    }
    uint4* out = reinterpret_cast<uint4*>(a + ((int64_t)real_end[lo] + (pr - pad_prefix[lo])) * H);
    for (int64_t v = lane; v < nv; v += 32) out[v] = make_uint4(0, 0, 0, 0);
  }
}

// UK source rows at a time, VU 16-byte column chunks per lane and trip: UK x
// VU loads in flight per lane (about 8 for every k).
template <int UK, int VU>
__global__ void __launch_bounds__(256) k_route_unpermute(const uint16_t* __restrict__ y, int64_t N,
                                                         const int32_t* __restrict__ row_of,
                                                         const float* __restrict__ w, int64_t T, int k,
                                                         uint16_t* __restrict__ out) {
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int64_t nv = N / 8;
  // the token's first UK source rows and weights, once (rows past k: -1)
  int r0[UK];
  float w0[UK];
#pragma unroll
  for (int j = 0; j < UK; ++j) {
    r0[j] = j < k ? row_of[t * k + j] : -1;
    w0[j] = (w && j < k) ? w[t * k + j] : 1.0f;
  }
  for (int64_t vb = lane; vb < nv; vb += 32 * VU) {
    float acc[VU][8];
#pragma unroll
    for (int u = 0; u < VU; ++u)
#pragma unroll
      for (int h = 0; h < 8; ++h) acc[u][h] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += UK) {
      int rj[UK];
      float wj[UK];
#pragma unroll
      for (int j = 0; j < UK; ++j) {
        rj[j] = j0 == 0 ? r0[j] : (j0 + j < k ? row_of[t * k + j0 + j] : -1);
        wj[j] = j0 == 0 ? w0[j] : ((w && j0 + j < k) ? w[t * k + j0 + j] : 1.0f);
      }
      // every load of the group first, then the sums in slot order
      uint4 sv[VU][UK];
#pragma unroll
      for (int u = 0; u < VU; ++u)
#pragma unroll
        for (int j = 0; j < UK; ++j)
          sv[u][j] = (rj[j] >= 0 && vb + 32 * u < nv) ? ld_nc16(y + (int64_t)rj[j] * N + (vb + 32 * u) * 8)
                                                      : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < VU; ++u)
#pragma unroll
        for (int j = 0; j < UK; ++j) {
          if (rj[j] < 0) continue;
          const uint32_t q[4] = {sv[u][j].x, sv[u][j].y, sv[u][j].z, sv[u][j].w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            acc[u][2 * h] = __fadd_rn(acc[u][2 * h], w ? __fmul_rn(wj[j], bf16_lo(q[h])) : bf16_lo(q[h]));
            acc[u][2 * h + 1] =
                __fadd_rn(acc[u][2 * h + 1], w ? __fmul_rn(wj[j], bf16_hi(q[h])) : bf16_hi(q[h]));
          }
        }
    }
#pragma unroll
    for (int u = 0; u < VU; ++u) {
      if (vb + 32 * u >= nv) break;
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[u][2 * h], acc[u][2 * h + 1]);
        o[h] = *reinterpret_cast<const uint32_t*>(&b);
      }
      reinterpret_cast<uint4*>(out + t * N)[vb + 32 * u] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

int64_t route_workspace_bytes(int64_t T, int64_t k, int64_t E) {
  const int64_t n = T * k;
  const int64_t nchunks = (n + RT_CHUNK - 1) / RT_CHUNK;
  return (nchunks * E + 2 * E + 1) * (int64_t)sizeof(int32_t);
}

cudaError_t launch_route_permute(const void* x, int64_t T, int64_t H, const int32_t* idx, const float* w, int64_t k,
                                 int64_t E, int64_t rows, void* a, int32_t* offs, int32_t* row_of, void* workspace,
                                 int num_sms, int* status, cudaStream_t st) {
  if (E < 1 || E > RT_MAXE) return cudaErrorInvalidValue;
  const int64_t n = T * k;
  const int64_t nchunks = (n + RT_CHUNK - 1) / RT_CHUNK;
  int32_t* counts = (int32_t*)workspace;
  int32_t* real_end = counts + nchunks * E;
  int32_t* pad_prefix = real_end + E;
  cudaError_t e;
  if (nchunks > 0) {
    k_route_count<<<(unsigned)nchunks, 256, 0, st>>>(idx, n, (int)E, counts, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_route_scan<<<1, 1024, 0, st>>>(counts, (int)nchunks, (int)E, rows, offs, real_end, pad_prefix);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (nchunks > 0) {
    k_route_rank<<<(unsigned)nchunks, 32, 0, st>>>(idx, n, (int)E, counts, row_of);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // rows to copy or zero: about n + 31 E; 8 warps per CTA, several CTAs per SM
  int64_t blocks = (n + 31 * E + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  k_route_copy<<<(unsigned)blocks, 256, 0, st>>>((const uint16_t*)x, H, w, n, (int)k, (int)E, row_of, real_end,
                                                 pad_prefix, (uint16_t*)a);
  return cudaGetLastError();
}

int64_t route_static_scratch_bytes() { return ROUTE_STATIC_SCRATCH_BYTES; }

// Device address of g_route_scratch on the current device.  Host code only
// holds a stand-in for the array's name, so the address is looked up once
// per device (with that device current) and cached.
cudaError_t route_static_scratch(void** out) {
  constexpr int kMaxDev = 128;
  static std::mutex mu;
  static void* addr[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_route_unpermute(const void* y, int64_t N, const int32_t* row_of, const float* w, int64_t T,
                                   int64_t k, void* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int64_t blocks = (T + 7) / 8;
  const uint16_t* yp = (const uint16_t*)y;
  uint16_t* op = (uint16_t*)out;
  if (k <= 1)
    k_route_unpermute<1, 8><<<(unsigned)blocks, 256, 0, st>>>(yp, N, row_of, w, T, (int)k, op);
  else if (k <= 2)
    k_route_unpermute<2, 4><<<(unsigned)blocks, 256, 0, st>>>(yp, N, row_of, w, T, (int)k, op);
  else if (k <= 4)
    k_route_unpermute<4, 2><<<(unsigned)blocks, 256, 0, st>>>(yp, N, row_of, w, T, (int)k, op);
  else
    k_route_unpermute<8, 1><<<(unsigned)blocks, 256, 0, st>>>(yp, N, row_of, w, T, (int)k, op);
  return cudaGetLastError();
}

}  // namespace fp8moe
