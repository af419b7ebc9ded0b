// Tensorwise FP8 quantization: one scale for a whole tensor, the coarsest of
// the four scaling granularities ("FP8-обучение на AMD", section "Скейлы: от
// тензора до микроблока").  The arithmetic is the rowwise one (fp32:
// s = fmax / max(amax, 1e-12), q = RNE_sat(x * s), stored inv = 1 / s) with
// the absolute maximum taken over every element.
//
// Plain layout: one cooperative launch, one CTA per SM (k_tw_stream).  Each
// CTA streams its contiguous slice of the tensor through a shared-memory
// ring for the maximum, keeping the slice's last tiles resident; the CTAs
// meet on the caller's one-float scale buffer (zeroed first: the maxima are
// folded into its low 16 bits and the CTAs count themselves in its high 16
// bits); then each casts its resident tiles from shared memory and re-reads
// the rest, newest first, from L2.  A second count after the maximum has
// been read tells the last CTA to write fl(1/s) in the word's place.
//
// Transposed layouts: three stream-ordered launches around the same buffer,
// which holds the maximum's bf16 bit pattern until the last one replaces it
// by the dequantization scale:
//   1. k_tw_amax: grid-stride 16-byte loads (four in flight per thread; six
//      256-thread CTAs per SM, the grid one wave of them),
//      warp / block maxima, one atomicMax per block (bit patterns of
//      non-negative values order like the values);
//   2. the cast: k_tw_cast for the plain layout, or the colwise kernel in its
//      fixed-scale mode for the transposed / jagged layouts;
//   3. k_tw_finalize: one thread writes fl(1 / s).
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace fp8moe {

// One-shot test hook: armed by fp8moe_testing_stall_next_tensorwise,
// consumed by the next launch of the one-launch tensorwise kernel.
static std::atomic<int> g_tw_stall{0};
void arm_tensorwise_stall_hook() { g_tw_stall.store(1, std::memory_order_relaxed); }

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

FP8MOE_DEV uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

FP8MOE_DEV uint4 lds16(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// The streaming kernel's ring: SLOTS tiles of TILE bytes of bf16 input.
constexpr int TWS_TILE = 16384;
constexpr int TWS_CW = 16;                       // consumer warps (one producer warp besides)
constexpr int TWS_THREADS = 32 * (TWS_CW + 1);
template <int SLOTS>
constexpr size_t tws_smem() {
  return (size_t)SLOTS * TWS_TILE + 2 * SLOTS * sizeof(uint64_t);
}

// A consumer thread's 8 words of a tile (its chunks ct and ct + 512) to and
// from its TMEM lane: 32 lanes x 8 columns per warp.
FP8MOE_DEV void tmem_st8(uint32_t taddr, uint4 a, uint4 b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
FP8MOE_DEV void tmem_ld8(uint32_t taddr, uint4& a, uint4& b) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "r"(taddr)
               : "memory");
}

// One CTA per SM, every CTA resident (cooperative launch).  CTA b owns the
// contiguous tiles [nt*b/G, nt*(b+1)/G) of the tensor's whole 16-byte
// chunks (m of them).  A producer thread streams them through the
// shared-memory ring with bulk async copies; the consumer warps take each
// tile's maximum.  The tensor is held on chip across the grid-wide meeting
// as far as it fits: the last SLOTS tiles stay in their ring slots, the
// first TMEM_TILES (of those whose slot is reused) are copied to TMEM, each
// consumer thread keeping its own 8 words of a tile in its TMEM lane.
// After the meeting the consumers cast the resident tiles, then the TMEM
// tiles while the producer re-reads the rest (newest first: the likeliest
// to be in L2) into the freed slots, and cast those last.
//
// Items k = 0 .. m-1 are the phase-one loads of local tiles 0 .. m-1 (slot
// k % SLOTS); with r = max(0, m - SLOTS) and T = min(TMEM_TILES, r), items
// k = m .. m+r-T-1 re-read local tiles r-1 down to T.  Slot s holds items
// s, s+SLOTS, ... in order, so item k's fill completes the full barrier's
// phase k / SLOTS and its release the empty barrier's phase k / SLOTS.
template <bool FNUZ, int TWS_SLOTS, int TWS_TMEM_COLS, int MINB>
__global__ void __launch_bounds__(TWS_THREADS, MINB)
    k_tw_stream(const uint8_t* __restrict__ x, int64_t n, uint8_t* __restrict__ q, uint32_t* word, int* status,
                int stall_test) {
  constexpr int TWS_TMEM_TILES = TWS_TMEM_COLS / 32;
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)TWS_SLOTS * TWS_TILE);
  uint64_t* empty = full + TWS_SLOTS;
  __shared__ uint32_t wmax[TWS_CW];
  __shared__ uint32_t amax_s, tmem_s;
  __shared__ int abort_s;

  const int64_t nbytes = (n / 8) * 16;
  const int64_t nt = (nbytes + TWS_TILE - 1) / TWS_TILE;
  const int64_t t_lo = nt * blockIdx.x / gridDim.x;
  const int m = (int)(nt * (blockIdx.x + 1) / gridDim.x - t_lo);
  const int r = m > TWS_SLOTS ? m - TWS_SLOTS : 0;
  const int T = r < TWS_TMEM_TILES ? r : TWS_TMEM_TILES;
  const int total = m + r - T;
  auto local_tile = [&](int k) { return k < m ? k : r - 1 - (k - m); };
  auto gtile = [&](int j) { return t_lo + j; };  // global index of local tile j
  auto tile_bytes = [&](int k) {
    const int64_t off = gtile(local_tile(k)) * TWS_TILE;
    return (int)min((int64_t)TWS_TILE, nbytes - off);
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // a ring wait that ran out: the pipeline is broken, later ring waits
  // return at once
  auto fail = [&]() {
    set_status(status, FP8MOE_ERR_TIMEOUT);
    abort_s = 1;
  };
  // producer: fill the slot of item k once its previous occupant is released
  // (filled / fill_par: the slots filled and the phase bit of their last fill)
  uint32_t filled = 0, fill_par = 0;
  auto issue = [&](int k) {
    const int s = k % TWS_SLOTS;
    if (k >= TWS_SLOTS && !mbar_wait(&empty[s], (k / TWS_SLOTS - 1) & 1, &abort_s)) fail();
    filled |= 1u << s;
    fill_par = (fill_par & ~(1u << s)) | ((uint32_t)((k / TWS_SLOTS) & 1) << s);
    const int bytes = tile_bytes(k);
    mbar_expect_tx(&full[s], (uint32_t)bytes);
    bulk_load(sm + (size_t)s * TWS_TILE, x + gtile(local_tile(k)) * TWS_TILE, (uint32_t)bytes, &full[s]);
  };
  // the first ring fills leave as soon as the barriers exist, ahead of the
  // TMEM allocation and the block-wide barrier
  const int pre = m < TWS_SLOTS ? m : TWS_SLOTS;
  if (threadIdx.x == 0) {
    abort_s = 0;
    for (int i = 0; i < TWS_SLOTS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], TWS_CW);
    }
    mbar_fence_init();
    for (int k = 0; k < pre; ++k) issue(k);
  }
  if (warp == 1 && T > 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_s)),
                 "r"(TWS_TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();

  const int ct = threadIdx.x - 32;  // consumer thread index
  constexpr int CT = 32 * TWS_CW;   // consumer threads; a full tile is 2 * CT chunks
  static_assert(2 * CT * 16 == TWS_TILE, "two chunks per consumer thread per tile");
  // this thread's TMEM words of local tile j: lane quarter warp % 4, 8
  // columns per (quarter, warp) pair, 32 columns per tile
  const uint32_t tq = (uint32_t)(32 * (warp & 3)) << 16;
  auto taddr = [&](int j) { return tmem_s + tq + (uint32_t)(j * 32 + ((warp - 1) >> 2) * 8); };

  // ---- phase one: every element's magnitude
  uint32_t mx = 0;
  if (warp == 0) {
    if (lane == 0)
      for (int k = pre; k < m; ++k) issue(k);
  } else {
    for (int k = 0; k < m; ++k) {
      const int s = k % TWS_SLOTS;
      if (!mbar_wait(&full[s], (k / TWS_SLOTS) & 1, &abort_s)) fail();
      const uint8_t* src = sm + (size_t)s * TWS_TILE;
      const int chunks = tile_bytes(k) >> 4;
      if (chunks == 2 * CT) {
        const uint4 v0 = lds16(src + ct * 16), v1 = lds16(src + (ct + CT) * 16);
        mx = max(mx, max(absmax8_bits(v0), absmax8_bits(v1)));
        if (k < T) tmem_st8(taddr(k), v0, v1);
      } else {
        for (int c = ct; c < chunks; c += CT) mx = max(mx, absmax8_bits(lds16(src + c * 16)));
      }
      if (k < r) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    if (blockIdx.x == gridDim.x - 1)
      for (int64_t i = (n / 8) * 8 + ct; i < n; i += CT) {
        uint16_t b;
        asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(b) : "l"(x + 2 * i));
        mx = max(mx, (uint32_t)b & 0x7FFFu);
      }
    if (T > 0) asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) wmax[warp - 1] = mx;
  }
  __syncthreads();

  // ---- the grid-wide meeting on the caller's scale word
  if (threadIdx.x == 0) {
    for (int w = 0; w < TWS_CW; ++w) mx = max(mx, wmax[w]);
    // count this CTA in and fold its maximum in: a plain add when the
    // maximum already there is at least this CTA's, a compare-and-swap
    // otherwise
    uint32_t seen = ld_acquire(word);
    // test hook: CTA 0 of this launch never counts itself in, so every
    // CTA's bounded wait below runs out
    for (; !(stall_test && blockIdx.x == 0);) {
      if ((seen & 0xFFFFu) >= mx) {
        atomicAdd(word, 1u << 16);
        break;
      }
      const uint32_t old = atomicCAS(word, seen, ((seen + (1u << 16)) & 0xFFFF0000u) | mx);
      if (old == seen) break;
      seen = old;
    }
    // every CTA's maximum is in once the count is complete (bounded wait,
    // polling with loads so as not to queue behind the other CTAs' atomics)
    const uint64_t t0 = globaltimer();
    uint32_t cur = ld_acquire(word);
    while ((cur >> 16) < gridDim.x) {
      if (globaltimer() - t0 > WAIT_LIMIT_NS) {
        // the meeting ran out: the status says the result is not valid; the
        // ring's loads do not depend on the meeting and still complete and
        // are waited for, so no copy is in flight when the CTA exits
        set_status(status, FP8MOE_ERR_TIMEOUT);
        break;
      }
      __nanosleep(32);
      cur = ld_acquire(word);
    }
    amax_s = cur & 0xFFFFu;
  }
  __syncthreads();

  // ---- phase two: the cast (ring-resident tiles, TMEM tiles, re-reads)
  if (warp == 0) {
    if (lane == 0)
      for (int k = m; k < total; ++k) issue(k);
  } else {
    float sc, inv;
    rowwise_scale<FNUZ>(bf16bits_to_float(amax_s), sc, inv);
    auto cast_slot = [&](int k) {
      const int s = k % TWS_SLOTS;
      const uint8_t* src = sm + (size_t)s * TWS_TILE;
      uint8_t* dst = q + gtile(local_tile(k)) * (TWS_TILE / 2);
      const int chunks = tile_bytes(k) >> 4;
      if (chunks == 2 * CT) {
        const uint4 v0 = lds16(src + ct * 16), v1 = lds16(src + (ct + CT) * 16);
        *reinterpret_cast<uint2*>(dst + ct * 8) = enc8_bf16<FNUZ>(v0, sc);
        *reinterpret_cast<uint2*>(dst + (ct + CT) * 8) = enc8_bf16<FNUZ>(v1, sc);
      } else {
        for (int c = ct; c < chunks; c += CT)
          *reinterpret_cast<uint2*>(dst + c * 8) = enc8_bf16<FNUZ>(lds16(src + c * 16), sc);
      }
      if (k + TWS_SLOTS < total) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    };
    for (int k = r; k < m; ++k) cast_slot(k);
    for (int j = 0; j < T; ++j) {
      uint4 v0, v1;
      tmem_ld8(taddr(j), v0, v1);
      tmem_ld_wait();
      uint8_t* dst = q + gtile(j) * (TWS_TILE / 2);
      *reinterpret_cast<uint2*>(dst + ct * 8) = enc8_bf16<FNUZ>(v0, sc);
      *reinterpret_cast<uint2*>(dst + (ct + CT) * 8) = enc8_bf16<FNUZ>(v1, sc);
    }
    for (int k = m; k < total; ++k) {
      if (!mbar_wait(&full[k % TWS_SLOTS], (k / TWS_SLOTS) & 1, &abort_s)) fail();
      cast_slot(k);
    }
    if (blockIdx.x == gridDim.x - 1)
      for (int64_t i = (n / 8) * 8 + ct; i < n; i += CT) {
        uint16_t b;
        asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(b) : "l"(x + 2 * i));
        q[i] = (uint8_t)(enc2<FNUZ>(__fmul_rn(bf16bits_to_float(b), sc), 0.0f) & 0xFFu);
      }
  }
  // the second count, off the critical path: once every CTA has read the
  // maximum (each counts itself only after its own read), the last one
  // writes the dequantization scale in the word's place
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(word, 1u << 16);
    if ((prev >> 16) + 1u == 2u * gridDim.x) {
      float sc, inv;
      rowwise_scale<FNUZ>(bf16bits_to_float(amax_s), sc, inv);
      *reinterpret_cast<volatile float*>(word) = inv;
    }
  }
  // after a ring wait that ran out (in any thread: read after the barrier),
  // the producer waits (bounded) for the last fill of every slot, so no copy
  // is in flight when the CTA exits
  __syncthreads();
  if (threadIdx.x == 0 && abort_s)
    for (int s = 0; s < TWS_SLOTS; ++s)
      if (filled & (1u << s)) (void)mbar_wait(&full[s], (fill_par >> s) & 1u, nullptr);
  tc_fence_before();
  __syncthreads();
  if (warp == 1 && T > 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_s), "r"(TWS_TMEM_COLS));
  }
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
  static std::atomic<int> per_amax{0}, per_fn{0}, per_fnuz{0}, per_stream_fn{0}, per_stream_fnuz{0};
  const int cap_amax = num_sms * blocks_per_sm(per_amax, k_tw_amax, 256, 0, 4);
  const int cap_fn = num_sms * blocks_per_sm(per_fn, k_tw_cast<false>, 256, 0, 4);
  const int cap_fnuz = num_sms * blocks_per_sm(per_fnuz, k_tw_cast<true>, 256, 0, 4);
  if (n > 0 && !transpose_out) {
    // ring depth, TMEM columns and CTAs per SM of the launched shape
    constexpr int SLOTS = 8, TCOLS = 512, PER = 1;
    constexpr size_t SMEM = tws_smem<SLOTS>();
    auto kern = fnuz ? k_tw_stream<true, SLOTS, TCOLS, PER> : k_tw_stream<false, SLOTS, TCOLS, PER>;
    static std::once_flag attr_once;
    std::call_once(attr_once, [] {
      cudaFuncSetAttribute(k_tw_stream<false, SLOTS, TCOLS, PER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM);
      cudaFuncSetAttribute(k_tw_stream<true, SLOTS, TCOLS, PER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SMEM);
    });
    const int per = blocks_per_sm(fnuz ? per_stream_fnuz : per_stream_fn, kern, TWS_THREADS, SMEM, 0);
    if (per > 0) {
      // one cooperative launch: the runtime refuses it rather than queue
      // CTAs that the resident ones would wait for.  More CTAs per SM than
      // the shape was sized for would overcommit TMEM, so the grid is PER
      // CTAs per SM at most.
      unsigned grid = (unsigned)(num_sms * (per < PER ? per : PER));
      if (grid > 32767u) grid = 32767u;  // two counts of the grid fit the word's 16 bits
      const uint8_t* xp = (const uint8_t*)x;
      uint8_t* qp = (uint8_t*)q;
      uint32_t* wp = (uint32_t*)scale_inv;
      int64_t nn = n;
      int stall = g_tw_stall.exchange(0, std::memory_order_relaxed);
      void* args[] = {(void*)&xp, (void*)&nn, (void*)&qp, (void*)&wp, (void*)&status, (void*)&stall};
      return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(TWS_THREADS), args, SMEM, st);
    }
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
