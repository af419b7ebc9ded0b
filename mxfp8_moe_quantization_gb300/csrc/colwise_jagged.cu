// Colwise FP8 quantization of routed rows grouped by offsets, codes written
// transposed into the group-padded layout, in one pass over HBM and without
// cross-CTA exchanges ("FP8-обучение на AMD", sections "MoE: почему
// DeepSeek-V3 ломал пайплайн" (a column scale per expert) and "Три уровня
// оптимизации Triton-ядер" (the backward colwise-scales kernel: the columns
// staged on chip, a single pass, the transposed output written directly)).
//
// x [R, C] bf16 in E groups (offsets) -> q [C, ldt] (group g's rows at
// columns 32 * (its 32-row blocks before it) ..., its padding up to the next
// multiple of 32 and the slack after the last group zero), scale_inv [E, C].
//
// A unit is one group's 64-column strip.  One persistent CTA per SM takes
// units one after another from a device-wide counter over the units ordered
// largest group first, so that the CTAs finish together whatever the group
// sizes (a fixed assignment, e.g. a snake order over the CTAs, left the
// slowest CTA ~20% above the mean on a skewed routing):
//   * a producer warp streams the units' TMA boxes (128 rows x 64 columns,
//     128-byte swizzle, 16 KB) through a ring of CJ_NS slots, running ahead
//     into the next units while slots are free;
//   * two groups of eight consumer warps take alternate units (one group's
//     maxima pass overlaps the other's cast): a group takes its unit's
//     column maxima as the boxes land, combines them in shared memory,
//     derives the 64 scales and casts.  A
//     unit of at most CJ_NS boxes stays resident from its maxima to its cast
//     (its slots are released by the cast, box by box, so the next unit's
//     boxes load meanwhile); a longer unit is loaded twice: its boxes are
//     released after the maxima and loaded again for the cast (from L2:
//     read moments before).
// The whole group's column maximum is on one CTA, so no cluster exchange and
// no waiting on a slower peer.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "scales.cuh"
#include "tma.cuh"

namespace fp8moe {
namespace {

constexpr int CJ_COLS = 64;                          // columns of a unit: 128 bytes of a bf16 row
constexpr int CJ_BOXR = 128;                         // rows of one TMA box
constexpr int CJ_BOX_BYTES = CJ_BOXR * CJ_COLS * 2;  // 16 KB
constexpr int CJ_NS = 12;                            // ring slots: 192 KB
constexpr int CJ_CONS = 16;                          // consumer warps
constexpr int CJ_GW = CJ_CONS / 2;                   // warps of each of the two consumer groups
constexpr int CJ_THREADS = 32 * (CJ_CONS + 1);
constexpr size_t CJ_SMEM = (size_t)CJ_NS * CJ_BOX_BYTES + 1024;   // + room to align the ring to 1 KB
constexpr int CJ_UQ = 32;                            // entries of the producer's unit queue
constexpr int CJ_SLOTS = 16;                         // work-counter slots, one per launch in flight

// The work counters.  A launch with generation `gen` (a per-process launch
// count, never 0) uses slot gen % CJ_SLOTS: word = gen << 32 | units taken.
// Every CTA first raises the word to gen << 32 (a no-op once another CTA of
// the launch has), then takes units with atomicAdd; a word whose top half
// is not `gen` means that another launch in flight holds the slot, which
// the launch reports as FP8MOE_ERR_CONCURRENT.  The `units` word sums the
// units each CTA handed to its consumers and the `done` word counts the
// CTAs that have finished taking units (same tags); the last CTA checks that
// the launch took every unit exactly once (another launch's takes from the
// slot would have consumed some of its counts: FP8MOE_ERR_CONCURRENT, never
// a silent gap) and returns the three words to zero, so a replay of the same
// launch (a CUDA graph) starts clean.
__device__ unsigned long long g_cj_work[CJ_SLOTS];
__device__ unsigned long long g_cj_units[CJ_SLOTS];
__device__ unsigned long long g_cj_done[CJ_SLOTS];

struct CjArgs {
  int64_t E, R, C;
  int64_t n_ct;    // 64-column strips
  int64_t units;   // E * n_ct
  int64_t ldt;     // row length of q
  const int32_t* offs;
  uint8_t* q;
  float* inv;
  int* status;
  int stall_test;  // the first box of unit 0 is never loaded (timeout-path test)
  uint32_t gen;    // launch generation (work-counter tag), slot = gen % CJ_SLOTS
};

// A unit queue entry: the unit's index in the size-ordered list (-1: no
// more units, -2: the launch stopped) and the fill of its first box.
struct CjEntry {
  long long u;
  uint32_t f0;
};

FP8MOE_DEV void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

template <bool FNUZ>
__global__ void __launch_bounds__(CJ_THREADS, 1) k_cw_jag_ws(const __grid_constant__ CUtensorMap tmX, CjArgs a) {
  __shared__ GroupTable gt;
  __shared__ int order[QG_MAX];
  __shared__ uint64_t full[CJ_NS], empty[CJ_NS];
  __shared__ uint4 wmax[2][CJ_GW][8];   // per group, warp and 16-byte column chunk: 8 maxima as bf16 pairs
  __shared__ float scol[2][CJ_COLS];
  __shared__ int abort_s;
  __shared__ uint32_t issued_s;   // fills the producer has issued
  __shared__ CjEntry uq[CJ_UQ];   // units in the order the producer took them
  __shared__ int nq_s;            // entries published
  __shared__ int read_s[2];       // per consumer group: 1 + the last entry it took
  __shared__ CjEntry ubc[2];      // per consumer group: the entry its elected thread took
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // every CTA builds the same table, so bad offsets send every CTA home here
  build_group_table(gt, a.offs, (int)a.E, a.R, GT_SUB32, a.status);
  if (gt.bad) return;
  // groups by size, largest first (equal sizes by index)
  for (int g = tid; g < (int)a.E; g += CJ_THREADS) {
    const int64_t sg = gt.end[g] - (g ? gt.end[g - 1] : 0);
    int rk = 0;
    for (int h = 0; h < (int)a.E; ++h) {
      const int64_t sh = gt.end[h] - (h ? gt.end[h - 1] : 0);
      rk += (sh > sg || (sh == sg && h < g)) ? 1 : 0;
    }
    order[rk] = g;
  }
  if (tid == 0) {
    for (int i = 0; i < CJ_NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CJ_GW);
    }
    abort_s = 0;
    issued_s = 0;
    nq_s = 0;
    read_s[0] = read_s[1] = 0;
    mbar_fence_init();
  }
  __syncthreads();

  // unit u of the size-ordered list: group order[u / n_ct], strip u % n_ct
  struct U {
    int64_t g, gs, rg, rpad, qcol0;
    int col0, nbox;
  };
  auto unit_of = [&](int64_t u, U& o) {
    const int64_t gi = u / a.n_ct;
    o.col0 = (int)((u - gi * a.n_ct) * CJ_COLS);
    o.g = order[gi];
    o.gs = o.g ? gt.end[o.g - 1] : 0;
    o.rg = gt.end[o.g] - o.gs;
    o.rpad = (o.rg + 31) / 32 * 32;
    o.qcol0 = 32 * gt.pad[o.g];
    o.nbox = (int)((o.rg + CJ_BOXR - 1) / CJ_BOXR);
  };

  if (warp == CJ_CONS) {
    // ======================= producer =======================
    if (lane == 0) {
      unsigned long long* wk = &g_cj_work[a.gen % CJ_SLOTS];
      unsigned long long* dn = &g_cj_done[a.gen % CJ_SLOTS];
      unsigned long long* pu = &g_cj_units[a.gen % CJ_SLOTS];
      const unsigned long long tag = (unsigned long long)a.gen << 32;
      atomicMax(wk, tag);
      atomicMax(dn, tag);
      atomicMax(pu, tag);
      uint32_t handed = 0;   // units this CTA published to its consumers
      // the next unit's index: taken one unit ahead, so that the atomic's
      // round trip overlaps the issue of the current unit's boxes
      unsigned long long taken = atomicAdd(wk, 1ull);
      uint32_t f = 0;   // boxes issued so far (fill f goes to slot f % CJ_NS)
      bool live = true;
      auto stop = [&](int code) {
        if (!abort_s) set_status(a.status, code);
        abort_s = 1;
        live = false;
      };
      // room for entry n: entry n - CJ_UQ has been taken by its group
      auto room = [&](int n) -> bool {
        if (n < CJ_UQ) return true;
        const volatile int* rd = &read_s[(n - CJ_UQ) & 1];
        const uint64_t t0 = globaltimer();
        while (*rd <= n - CJ_UQ) {
          if (abort_s || globaltimer() - t0 > WAIT_LIMIT_NS) return false;
        }
        return true;
      };
      auto publish = [&](int n, long long u) {
        volatile CjEntry* e = &uq[n % CJ_UQ];
        e->u = u;
        e->f0 = f;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&nq_s) = n + 1;
      };
      int n = 0;
      for (; live; ++n) {
        long long k;
        if ((taken >> 32) != a.gen) {
          stop(FP8MOE_ERR_CONCURRENT);
          break;
        }
        k = (long long)(taken & 0xFFFFFFFFull);
        if (k >= a.units) break;
        taken = atomicAdd(wk, 1ull);
        if (!room(n)) {
          stop(FP8MOE_ERR_TIMEOUT);
          break;
        }
        U u;
        unit_of(k, u);
        publish(n, k);
        ++handed;
        const int passes = u.nbox <= CJ_NS ? 1 : 2;
        for (int p = 0; p < passes && live; ++p)
          for (int b = 0; b < u.nbox; ++b, ++f) {
            const uint32_t s = f % CJ_NS;
            if (f >= CJ_NS && !mbar_wait(&empty[s], ((f / CJ_NS) - 1) & 1u, &abort_s)) {
              stop(FP8MOE_ERR_TIMEOUT);
              break;
            }
            // test hook: the first box of unit 0 (whichever CTA takes it) is
            // never loaded (but counted as issued), so its consumers'
            // bounded wait runs out
            if (!(a.stall_test && k == 0 && p == 0 && b == 0)) {
              mbar_expect_tx(&full[s], CJ_BOX_BYTES);
              tma_load_2d(ring + s * CJ_BOX_BYTES, &tmX, &full[s], u.col0, (int)(u.gs + (int64_t)b * CJ_BOXR));
            }
            // publish the fill (after the release of fill f - CJ_NS that it waited for)
            __threadfence_block();
            *reinterpret_cast<volatile uint32_t*>(&issued_s) = f + 1;
          }
      }
      // no more units: one end entry for each group (after a stop the
      // consumers leave on abort_s instead)
      for (int e = 0; e < 2 && live; ++e) {
        if (room(n + e))
          publish(n + e, -1);
        else
          stop(FP8MOE_ERR_TIMEOUT);
      }
      // the loads still in flight land before the CTA can leave (the
      // consumers may have stopped early): the last fill of each slot
      for (uint32_t j = f > CJ_NS ? f - CJ_NS : 0; j < f; ++j)
        (void)mbar_wait(&full[j % CJ_NS], (j / CJ_NS) & 1u, nullptr);
      // the last CTA to finish taking units checks the sum and clears the slot
      atomicAdd(pu, (unsigned long long)handed);
      __threadfence();
      const unsigned long long d = atomicAdd(dn, 1ull);
      if ((d >> 32) == a.gen && (d & 0xFFFFFFFFull) == gridDim.x - 1) {
        __threadfence();
        const unsigned long long pv = atomicAdd(pu, 0ull);
        if ((pv >> 32) != a.gen || (pv & 0xFFFFFFFFull) != (unsigned long long)a.units)
          set_status(a.status, FP8MOE_ERR_CONCURRENT);
        atomicExch(wk, 0ull);
        atomicExch(dn, 0ull);
        atomicExch(pu, 0ull);
      }
    }
    return;
  }

  // ======================= consumers =======================
  // Two groups of CJ_GW warps take alternate units, so that one group's
  // maxima pass (its boxes landing) overlaps the other group's cast.
  const int grp = warp / CJ_GW, gw = warp % CJ_GW, gt_ = tid % (32 * CJ_GW);
  const int cc = gt_ & 7, rp = gt_ >> 3;    // maxima: 16-byte column chunk, row phase (0 .. 31)
  const int cl = lane & 7, rq = lane >> 3;  // cast: 8 columns x 8 rows per lane in a 32-row quarter
  auto group_sync = [&]() {
    if (grp == 0)
      asm volatile("bar.sync 1, %0;" ::"n"(32 * CJ_GW) : "memory");
    else
      asm volatile("bar.sync 2, %0;" ::"n"(32 * CJ_GW) : "memory");
  };
  // Fill fb of slot s completes phase fb / CJ_NS of full[s].  The barrier
  // knows phases only by their parity, and the two groups consume fills out
  // of step, so a group first waits until the producer has issued fill fb:
  // it did so after the release of fill fb - CJ_NS, so the barrier is then
  // at phase fb / CJ_NS or at the one before it, never two behind (which
  // would show the wanted parity already).
  auto wait_fill = [&](uint32_t fb) -> bool {
    const volatile uint32_t* iss = &issued_s;
    if (*iss <= fb) {
      const uint64_t t0 = globaltimer();
      while (*iss <= fb) {
        if (abort_s || globaltimer() - t0 > WAIT_LIMIT_NS) return false;
      }
    }
    __threadfence_block();
    return mbar_wait(&full[fb % CJ_NS], (fb / CJ_NS) & 1u, &abort_s);
  };
  // the group's elected thread takes queue entry n and hands it to the
  // group (one decision for all its warps, so that they meet the same
  // barriers)
  auto take = [&](int n) -> CjEntry {
    if (gw == 0 && lane == 0) {
      CjEntry e;
      e.u = -2;
      e.f0 = 0;
      const volatile int* nq = &nq_s;
      const uint64_t t0 = globaltimer();
      bool got = true;
      while (*nq <= n) {
        if (abort_s) {
          got = false;
          break;
        }
        if (globaltimer() - t0 > WAIT_LIMIT_NS) {
          set_status(a.status, FP8MOE_ERR_TIMEOUT);
          abort_s = 1;
          got = false;
          break;
        }
      }
      if (got) {
        __threadfence_block();
        const volatile CjEntry* q = &uq[n % CJ_UQ];
        e.u = q->u;
        e.f0 = q->f0;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&read_s[grp]) = n + 1;
      }
      ubc[grp] = e;
    }
    group_sync();
    return ubc[grp];
  };
  bool ok = true;   // false after a wait ran out: the warps keep meeting their barriers, no more work
  // entries alternate between the groups: group grp takes grp, grp + 2, ...
  for (int n = grp;; n += 2) {
    const CjEntry e = take(n);
    if (e.u < 0) break;
    U u;
    unit_of(e.u, u);
    const bool res = u.nbox <= CJ_NS;
    const uint32_t f0 = e.f0;
    ok = ok && !abort_s;
    // ---- 1. column maxima, box by box as they land
    uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    for (int b = 0; b < u.nbox && ok; ++b) {
      const uint32_t fb = f0 + b, s = fb % CJ_NS;
      if (!wait_fill(fb)) {
        if (!abort_s) set_status(a.status, FP8MOE_ERR_TIMEOUT);
        abort_s = 1;
        ok = false;
        break;
      }
      const uint8_t* box = ring + s * CJ_BOX_BYTES;
      const int64_t left = u.rg - (int64_t)b * CJ_BOXR;
      const int n = left < CJ_BOXR ? (int)left : CJ_BOXR;
#pragma unroll
      for (int h = 0; h < CJ_BOXR / (4 * CJ_GW); ++h) {
        const int r = rp + 4 * CJ_GW * h;
        if (r < n) {
          const uint4 v = *reinterpret_cast<const uint4*>(box + r * 128 + ((cc ^ (r & 7)) << 4));
          m0 = umax16x2(m0, v.x & 0x7FFF7FFFu);
          m1 = umax16x2(m1, v.y & 0x7FFF7FFFu);
          m2 = umax16x2(m2, v.z & 0x7FFF7FFFu);
          m3 = umax16x2(m3, v.w & 0x7FFF7FFFu);
        }
      }
      if (!res) {
        // a long unit: its box is loaded again for the cast
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
    }
    // lanes cc, cc + 8, cc + 16, cc + 24 hold the same columns
#pragma unroll
    for (int o = 8; o < 32; o <<= 1) {
      m0 = umax16x2(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = umax16x2(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      m2 = umax16x2(m2, __shfl_xor_sync(0xffffffffu, m2, o));
      m3 = umax16x2(m3, __shfl_xor_sync(0xffffffffu, m3, o));
    }
    if (lane < 8) wmax[grp][gw][lane] = make_uint4(m0, m1, m2, m3);
    group_sync();
    // ---- 2. the 64 scales
    if (gt_ < CJ_COLS) {
      uint32_t mc = 0;
#pragma unroll
      for (int w = 0; w < CJ_GW; ++w) {
        const uint32_t pair = reinterpret_cast<const uint32_t*>(&wmax[grp][w][gt_ >> 3])[(gt_ & 7) >> 1];
        mc = max(mc, (gt_ & 1) ? pair >> 16 : pair & 0xFFFFu);
      }
      float sc, iv;
      rowwise_scale<FNUZ>(bf16bits_to_float(mc), sc, iv);
      scol[grp][gt_] = sc;
      if (ok && u.col0 + gt_ < a.C) a.inv[u.g * a.C + u.col0 + gt_] = iv;
    }
    group_sync();
    ok = ok && !abort_s;
    // ---- 3. cast and transposed store: the unit's 32-row quarters of its
    // boxes over the group's warps (a box's four quarters on four warps,
    // which then release its slot together)
    uint64_t mul2[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) mul2[t] = pair_f32(enc_mul<FNUZ>(scol[grp][cl * 8 + t]));
    const int64_t col = u.col0 + cl * 8;
    for (int i = gw; i < 4 * u.nbox && ok; i += CJ_GW) {
      const int b = i >> 2;
      const uint32_t fb = res ? f0 + b : f0 + u.nbox + b, s = fb % CJ_NS;
      if (!res && !wait_fill(fb)) {
        if (!abort_s) set_status(a.status, FP8MOE_ERR_TIMEOUT);
        abort_s = 1;
        ok = false;
        break;
      }
      const uint8_t* box = ring + s * CJ_BOX_BYTES;
      const int64_t lr0 = (int64_t)b * CJ_BOXR + (i & 3) * 32 + rq * 8;   // this lane's first row in the group
      if (lr0 < u.rpad && col < a.C) {
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = (int)((lr0 + k) & 127);
          v[k] = *reinterpret_cast<const uint4*>(box + r * 128 + ((cl ^ (r & 7)) << 4));
        }
        uint2 cw[8];
        cast8x8_cols<FNUZ>(v, mul2, cw);
        // the group's padding rows (from rg to the next multiple of 32) get zero codes
        const int64_t nv = u.rg - lr0;
        if (nv < 8) {
          const uint64_t keep = nv <= 0 ? 0ull : (1ull << (8 * nv)) - 1;
#pragma unroll
          for (int t = 0; t < 8; ++t) cw[t] = make_uint2(cw[t].x & (uint32_t)keep, cw[t].y & (uint32_t)(keep >> 32));
        }
        // q[col + t][group column + row] for the 8 columns t
        uint8_t* base = a.q + col * a.ldt + u.qcol0 + lr0;
#pragma unroll
        for (int t = 0; t < 8; ++t) *reinterpret_cast<uint2*>(base + (int64_t)t * a.ldt) = cw[t];
      }
      // the box's slot: four warps x (CJ_GW / 4) arrivals
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&empty[s], CJ_GW / 4);
    }
  }
  // the slack of q after the last group: columns [32 * sub-tiles, ldt)
  {
    const int64_t E = a.E, last = gt.end[E - 1] - (E > 1 ? gt.end[E - 2] : 0);
    const int64_t from = 32 * (gt.pad[E - 1] + (last + 31) / 32);
    const int64_t chunks = (a.ldt - from) / 16;
    if (chunks > 0)
      for (int64_t i = (int64_t)blockIdx.x * (32 * CJ_CONS) + tid; i < a.C * chunks;
           i += (int64_t)gridDim.x * (32 * CJ_CONS)) {
        const int64_t row = i / chunks, ch = i - row * chunks;
        *reinterpret_cast<uint4*>(a.q + row * a.ldt + from + ch * 16) = make_uint4(0, 0, 0, 0);
      }
  }
}

}  // namespace

cudaError_t launch_colwise_jagged_ws(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs, int kind,
                                     int64_t ldt, void* q, float* inv, int* status, int num_sms, cudaStream_t st) {
  CjArgs a;
  a.E = E;
  a.R = R;
  a.C = C;
  a.n_ct = (C + CJ_COLS - 1) / CJ_COLS;
  a.units = E * a.n_ct;
  a.ldt = ldt;
  a.offs = offs;
  a.q = (uint8_t*)q;
  a.inv = inv;
  a.status = status;
  a.stall_test = take_ring_stall_hook();
  // units + one end-of-work take per CTA must fit the counter's 32 bits
  if (a.units + num_sms >= ((int64_t)1 << 32)) return cudaErrorInvalidValue;
  static std::atomic<uint32_t> gen{0};
  uint32_t g = gen.fetch_add(1, std::memory_order_relaxed) + 1;
  while (g == 0) g = gen.fetch_add(1, std::memory_order_relaxed) + 1;
  a.gen = g;
  CUtensorMap tm;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(R > 0 ? R : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)(C * 2)};
  cuuint32_t box[2] = {CJ_COLS, CJ_BOXR};
  if (!make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 2, dims, strides, box)) return cudaErrorInvalidValue;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(k_cw_jag_ws<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CJ_SMEM);
    cudaFuncSetAttribute(k_cw_jag_ws<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CJ_SMEM);
  });
  const unsigned grid = (unsigned)num_sms;
  if (kind == FP8MOE_E4M3FNUZ)
    k_cw_jag_ws<true><<<grid, CJ_THREADS, CJ_SMEM, st>>>(tm, a);
  else
    k_cw_jag_ws<false><<<grid, CJ_THREADS, CJ_SMEM, st>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace fp8moe
