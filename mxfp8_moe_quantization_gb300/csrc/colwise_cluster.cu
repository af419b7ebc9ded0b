// Colwise FP8 quantization with transposed output, in one pass over HBM, of
// dense 3D expert weights and of routed rows grouped by offsets
// ("FP8-обучение на AMD", sections "MoE: почему DeepSeek-V3 ломал пайплайн"
// (a column scale per expert) and "Три уровня оптимизации Triton-ядер" (the
// backward colwise-scales kernel: the columns staged on chip, a single pass,
// the transposed output written without a separate copy)).
//
// Dense: x [E, R, C] bf16 -> q [E, C, R] codes, scale_inv [E, C].  Jagged:
// x [R, C] in E groups -> q [C, ldt] (group-padded columns), scale_inv
// [E, C].  A unit is one expert's (group's) 64-column strip (128 bytes of
// every row).  A thread-block cluster
// of CL CTAs owns a unit at a time, each CTA a slice of S rows (a multiple of
// 32):
//   1. the CTA's slice lands in shared memory by TMA (boxes of 128 rows x 64
//      columns, 128-byte swizzle) and its column maxima are taken there;
//   2. the cluster combines the CTAs' maxima through distributed shared
//      memory, and every CTA derives the 64 scales;
//   3. each CTA casts its slice from shared memory and writes the codes
//      transposed: a lane turns 8 rows x 8 columns into 8-byte runs of its
//      columns (each conversion pairs one column's values from two
//      neighbouring rows, so the codes come out in column order), four
//      lanes complete a 32-byte sector of an output row.
// The boxes stream through a ring of NB slots: a slice of more boxes than
// that keeps its last NB boxes for the cast and loads the earlier ones again
// (read moments before, they come back from L2), so HBM still sees every
// input byte once; the cast then runs in a pipeline over two groups of four
// warps, each reload going into the slot its group has just freed.
#include <cuda.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "scales.cuh"
#include "tma.cuh"

namespace fp8moe {
namespace {

constexpr int CC_COLS = 64;                          // columns of a unit: 128 bytes of a bf16 row
constexpr int CC_BOXR = 128;                         // rows of one TMA box
constexpr int CC_BOX_BYTES = CC_BOXR * CC_COLS * 2;  // 16 KB
constexpr int CC_NB_MAX = 6;                         // box slots of the larger ring: 96 KB, two CTAs per SM
constexpr int CC_STREAM_SLACK = 2;                    // boxes of a slice past the ring worth a smaller cluster
constexpr int CC_THREADS = 256;

struct CcArgs {
  int64_t E, R, C;  // jagged: E groups of routed rows, R rows in all
  int64_t S;       // dense: rows of a unit per CTA (a multiple of 32)
  int64_t n_ct;    // 64-column tiles
  int64_t units;   // E * n_ct
  uint8_t* q;      // dense [E, C, R]; jagged [C, ldt]
  float* inv;      // [E, C]
  const int32_t* offs;  // jagged: group ends
  int64_t ldt;     // jagged: row length of q (group g at column 32 * its 32-row blocks before it)
  int* status;
};

FP8MOE_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
FP8MOE_DEV uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
FP8MOE_DEV uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
FP8MOE_DEV void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
FP8MOE_DEV uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
// a 32-bit store into CTA `rank`'s shared memory that completes 4 bytes of
// the transaction count of the mbarrier at `bar` there (no fence: the peer
// observes the data through its own barrier wait)
FP8MOE_DEV void st_async_peer(const void* dst, const void* bar, uint32_t rank, uint32_t v) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(peer_addr(dst, rank)),
               "r"(v), "r"(peer_addr(bar, rank))
               : "memory");
}

// NB box slots.  PRE: a slice takes at most half of them, so the boxes of
// the CTA's next units load while it casts the current one (a ring over the
// sequence of its units' boxes); otherwise each unit's slice streams through
// the ring on its own.
// JAG: routed rows [R, C] in E groups (offsets), codes in the group-padded
// transposed layout [C, ldt] (group g's rows at columns 32 * pad[g] ..., its
// padding up to the next multiple of 32 and the slack after the last group
// zero).  A unit is a group's 64-column strip; the CTAs of a cluster split
// the group's rows.  Units go to clusters largest group first, in a snake
// order (round k forward for even k, backward for odd), so the clusters'
// loads even out although group sizes vary widely.
template <int CL, int NB, bool PRE, bool FNUZ, bool JAG>
__global__ void __launch_bounds__(CC_THREADS, 2) k_cw_cluster(const __grid_constant__ CUtensorMap tmX, CcArgs a) {
  static_assert(!(JAG && PRE), "jagged units stream on their own");
  // jagged: the group table and the group order (largest first)
  __shared__ std::conditional_t<JAG, GroupTable, char> gt_s;
  __shared__ std::conditional_t<JAG, int[QG_MAX], char> order_s;
  constexpr int CC_NB = NB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sx = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);  // CC_NB box slots
  __shared__ uint64_t bars[NB];
  // the cluster's column maxima (bf16 bits) by unit parity and source CTA,
  // delivered by st.async; xbar[parity] completes when all CL x 64 landed
  __shared__ uint32_t xmax[2][CL][CC_COLS];
  __shared__ uint64_t xbar[2];
  __shared__ uint4 wmax[8][8];           // per warp and 16-byte column chunk: 8 maxima as bf16 pairs
  __shared__ float scol[CC_COLS];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
  const int64_t cid = CL > 1 ? (int64_t)cluster_id_x() : (int64_t)blockIdx.x;
  const int64_t ncl = CL > 1 ? (int64_t)num_clusters_x() : (int64_t)gridDim.x;
  if (tid == 0) {
    for (int i = 0; i < CC_NB; ++i) mbar_init(&bars[i], 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if constexpr (JAG) {
    // every CTA builds the same table, so a bad offsets vector sends every
    // CTA home here (before any cluster barrier)
    build_group_table(gt_s, a.offs, (int)a.E, a.R, GT_SUB32, a.status);
    if (gt_s.bad) return;
    for (int g = tid; g < (int)a.E; g += CC_THREADS) {
      const int64_t sg = gt_s.end[g] - (g ? gt_s.end[g - 1] : 0);
      int rk = 0;
      for (int h = 0; h < (int)a.E; ++h) {
        const int64_t sh = gt_s.end[h] - (h ? gt_s.end[h - 1] : 0);
        rk += (sh > sg || (sh == sg && h < g)) ? 1 : 0;
      }
      order_s[rk] = g;
    }
    __syncthreads();
  }
  // every CTA's barriers are initialised before a peer's st.async reaches them
  if constexpr (CL > 1) cluster_barrier();
  uint32_t xph = 0;  // phase bit of each exchange barrier
  uint32_t phases = 0;     // phase bit of each slot's next completion
  uint32_t pending = 0;    // slots with a load in flight (thread 0's view, for the exit path)
  bool ok = true;          // false after a load that never completed: the CTA keeps
                           // meeting its barriers but does no more work
  int ub = 0;
  const int cc = tid & 7, rp = tid >> 3;  // maxima pass: 16-byte column chunk, row phase (32)
  const int cl = lane & 7, rq = lane >> 3;  // cast: 8 columns x 8 rows per lane in a 32-row sub-tile

  // dense: this CTA's first row within each expert, its rows and boxes (the
  // same for every unit); jagged: set per unit
  int64_t r0 = (int64_t)rank * a.S;
  int nr = (int)(r0 < a.R ? (a.R - r0 < a.S ? a.R - r0 : a.S) : 0);
  int nbox = (nr + CC_BOXR - 1) / CC_BOXR;
  int npad = nr;          // rows whose codes this CTA writes (jagged: padding included)
  int64_t xrow0 = 0;      // row of x where this CTA's slice of the unit starts
  int64_t qcol0 = 0;      // jagged: column of q where the unit's group starts
  // PRE: global box j (unit k = j / nbox of this CTA, box j % nbox) sits in
  // slot j % NB; `issued` boxes have been requested so far
  const int64_t my_units = cid < a.units ? (a.units - 1 - cid) / ncl + 1 : 0;
  const int64_t total_boxes = my_units * nbox;
  int64_t issued = 0;
  auto unit_geom = [&](int64_t k, int64_t& g, int& col0) {
    const int64_t u = cid + k * ncl;
    g = u / a.n_ct;
    col0 = (int)((u - g * a.n_ct) * CC_COLS);
  };
  // thread 0: global box j into its slot (PRE) / box `box` of the unit at
  // (g, col0) into slot box % NB
  auto issue_at = [&](int slot, int64_t g, int col0, int box) {
    mbar_expect_tx(&bars[slot], CC_BOX_BYTES);
    const int64_t row = JAG ? xrow0 + (int64_t)box * CC_BOXR : g * a.R + r0 + (int64_t)box * CC_BOXR;
    tma_load_2d(sx + slot * CC_BOX_BYTES, &tmX, &bars[slot], col0, (int)row);
    pending |= 1u << slot;
  };
  auto issue_global = [&](int64_t j) {
    int64_t g;
    int col0;
    unit_geom(j / nbox, g, col0);
    issue_at((int)(j % NB), g, col0, (int)(j % nbox));
  };
  // (a wait that runs out leaves the slot pending with its phase, for the
  // exit path)
  auto wait_slot = [&](int slot) {
    if (!mbar_wait(&bars[slot], (phases >> slot) & 1u, nullptr)) {
      ok = false;
      return;
    }
    phases ^= 1u << slot;
    if (tid == 0 || tid == 128) pending &= ~(1u << slot);
  };
  // every thread is done with the slots before the ring refills them
  auto refill_barrier = [&]() {
    fence_proxy_async_smem();
    ok = __syncthreads_and(ok) != 0;
  };

  // Jagged: this CTA's part of the unit at snake position kk (false: no
  // unit there).  Its boxes are numbered on across the CTA's units; box j
  // sits in slot j % NB.  A unit whose boxes fit the ring has them loaded
  // ahead by a cursor that runs over the following units' boxes while slots
  // are free (it stops before a unit that does not fit: that one streams
  // through the ring on its own, as the dense kernel does).
  struct UG {
    int64_t g, r0, xrow0, qcol0;
    int col0, nr, nbox, npad;
  };
  auto jgeom = [&](int64_t kk, UG& o) -> bool {
    if constexpr (!JAG) {
      return false;
    } else {
    const int64_t u = kk * ncl + ((kk & 1) ? ncl - 1 - cid : cid);
    if (u >= a.units) return false;
    const int64_t gi = u / a.n_ct;
    o.col0 = (int)((u - gi * a.n_ct) * CC_COLS);
    o.g = order_s[gi];
    const int64_t gs = o.g ? gt_s.end[o.g - 1] : 0, rg = gt_s.end[o.g] - gs;
    const int64_t S = ((rg + CL - 1) / CL + 31) / 32 * 32;
    o.r0 = (int64_t)rank * S;
    o.nr = (int)(o.r0 < rg ? (rg - o.r0 < S ? rg - o.r0 : S) : 0);
    o.nbox = (o.nr + CC_BOXR - 1) / CC_BOXR;
    const int64_t rpad = (rg + 31) / 32 * 32;   // the group's rows with its padding
    o.npad = (int)(o.r0 < rpad ? (rpad - o.r0 < S ? rpad - o.r0 : S) : 0);
    o.xrow0 = gs + o.r0;
    o.qcol0 = 32 * gt_s.pad[o.g];
    return true;
    }
  };
  int64_t base = 0;      // jagged: number of this unit's first box
  // the cursor (thread 0): the next box to load is box pb of the unit at pkk
  int64_t pkk = 0;
  int pb = 0;
  UG pu{};
  bool pvalid = false;
  auto seek = [&](int64_t from) {
    pb = 0;
    for (pkk = from; pkk * ncl < a.units; ++pkk)
      if (jgeom(pkk, pu) && pu.nbox > 0) return true;
    return false;
  };
  if (JAG && tid == 0) pvalid = seek(0);
  auto issue_row = [&](int slot, int col0, int64_t row) {
    mbar_expect_tx(&bars[slot], CC_BOX_BYTES);
    tma_load_2d(sx + slot * CC_BOX_BYTES, &tmX, &bars[slot], col0, (int)row);
    pending |= 1u << slot;
  };

  int64_t k = 0;
  int preloaded = 0;   // boxes of this unit already loading (issued during the last unit's cast)
  for (int64_t kk = 0; JAG ? kk * ncl < a.units : cid + kk * ncl < a.units; ++kk) {
    int64_t u = cid + kk * ncl;
    int64_t g = u / a.n_ct;
    int col0 = (int)((u - g * a.n_ct) * CC_COLS);
    if constexpr (JAG) {
      UG c;
      if (!jgeom(kk, c)) continue;
      g = c.g;
      col0 = c.col0;
      r0 = c.r0;
      nr = c.nr;
      nbox = c.nbox;
      npad = c.npad;
      xrow0 = c.xrow0;
      qcol0 = c.qcol0;
    }
    const bool fits = nbox <= NB;
    // slot of box bx of this unit
    auto slot_of = [&](int bx) {
      return JAG ? (int)((base + bx) % NB) : (PRE ? (int)((k * nbox + bx) % NB) : bx % NB);
    };
    auto issue = [&](int box) {
      if constexpr (JAG) {
        issue_row(slot_of(box), col0, xrow0 + (int64_t)box * CC_BOXR);
      } else {
        issue_at(box % NB, g, col0, box);
      }
    };

    // ---- 1. column maxima: the slice streams through the ring once
    refill_barrier();
    if (PRE) {
      // the boxes whose slots are free: every box before this unit's has been cast
      if (ok && tid == 0) {
        const int64_t limit = k * nbox + NB < total_boxes ? k * nbox + NB : total_boxes;
        for (; issued < limit; ++issued) issue_global(issued);
      }
    } else if (JAG && fits) {
      // this unit's boxes not yet loaded and the following units' while
      // slots are free (every box before this unit's has been cast)
      if (ok && tid == 0)
        while (pvalid && issued < base + NB && pu.nbox <= NB) {
          issue_row((int)(issued % NB), pu.col0, pu.xrow0 + (int64_t)pb * CC_BOXR);
          ++issued;
          if (++pb == pu.nbox) pvalid = seek(pkk + 1);
        }
    } else if (ok && tid == 0) {
      for (int bx = preloaded; bx < nbox && bx < CC_NB; ++bx) issue(bx);
    }
    preloaded = 0;
    uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    for (int bx = 0; bx < nbox && ok; ++bx) {
      wait_slot(slot_of(bx));
      const uint8_t* box = sx + slot_of(bx) * CC_BOX_BYTES;
      const int n = nr - bx * CC_BOXR < CC_BOXR ? nr - bx * CC_BOXR : CC_BOXR;
#pragma unroll 4
      for (int r = rp; r < n; r += 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(box + (r & 127) * 128 + ((cc ^ (r & 7)) << 4));
        m0 = umax16x2(m0, v.x & 0x7FFF7FFFu);
        m1 = umax16x2(m1, v.y & 0x7FFF7FFFu);
        m2 = umax16x2(m2, v.z & 0x7FFF7FFFu);
        m3 = umax16x2(m3, v.w & 0x7FFF7FFFu);
      }
      if (!PRE && bx + CC_NB < nbox) {
        refill_barrier();
        if (ok && tid == 0) issue(bx + CC_NB);
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
    if (lane < 8) wmax[warp][lane] = make_uint4(m0, m1, m2, m3);
    ok = __syncthreads_and(ok) != 0;
    // ---- 2. the cluster's maxima -> scales
    if (tid < CC_COLS) {
      uint32_t mc = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const uint32_t pair = reinterpret_cast<const uint32_t*>(&wmax[w][tid >> 3])[(tid & 7) >> 1];
        mc = max(mc, (tid & 1) ? pair >> 16 : pair & 0xFFFFu);
      }
      if constexpr (CL > 1) {
        // to every CTA of the cluster (this one included), then wait for all
        if (tid == 0) mbar_expect_tx(&xbar[ub], CL * CC_COLS * 4);
#pragma unroll
        for (int r = 0; r < CL; ++r) st_async_peer(&xmax[ub][rank][tid], &xbar[ub], (uint32_t)r, mc);
        if (!mbar_wait(&xbar[ub], (xph >> ub) & 1u, nullptr)) ok = false;
#pragma unroll
        for (int r = 0; r < CL; ++r) mc = max(mc, xmax[ub][r][tid]);
      }
      float s, iv;
      rowwise_scale<FNUZ>(bf16bits_to_float(mc), s, iv);
      scol[tid] = s;
      if (ok && rank == 0 && col0 + tid < a.C) a.inv[g * a.C + col0 + tid] = iv;
    }
    xph ^= 1u << ub;
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
      ub ^= 1;
      ++k;
      base += nbox;
      continue;
    }
    // ---- 3. cast and transposed store
    uint64_t mul2[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) mul2[t] = pair_f32(enc_mul<FNUZ>(scol[cl * 8 + t]));
    const int64_t col = col0 + cl * 8;
    // one 32-row x 64-column sub-tile: local row lr0 (a multiple of 8) of
    // this lane, held in the slot at `box`
    auto cast_sub = [&](const uint8_t* box, int lr0) {
      // dense: R % 8 == 0, so a lane's 8 rows are all in or all out; jagged:
      // rows from nr to npad are the group's padding (zero codes)
      if (lr0 >= npad || col >= a.C) return;
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int r = (lr0 + k) & 127;
        v[k] = *reinterpret_cast<const uint4*>(box + r * 128 + ((cl ^ (r & 7)) << 4));
      }
      uint2 cw[8];
      cast8x8_cols<FNUZ>(v, mul2, cw);
      if (JAG && nr - lr0 < 8) {
        const int nv = nr - lr0;
        const uint64_t keep = nv <= 0 ? 0ull : (1ull << (8 * nv)) - 1;
#pragma unroll
        for (int t = 0; t < 8; ++t) cw[t] = make_uint2(cw[t].x & (uint32_t)keep, cw[t].y & (uint32_t)(keep >> 32));
      }
      // q[g][col + t][row .. row + 7] (jagged: q[col + t][group column + row])
      // for the 8 columns t
      const int64_t pitch = JAG ? a.ldt : a.R;
      uint8_t* base = JAG ? a.q + col * a.ldt + qcol0 + r0 + lr0 : a.q + (g * a.C + col) * a.R + r0 + lr0;
#pragma unroll
      for (int t = 0; t < 8; ++t) *reinterpret_cast<uint2*>(base + (int64_t)t * pitch) = cw[t];
    };
    // the boxes still resident after the maxima pass (the last CC_NB)
    const int first = nbox > CC_NB ? nbox - CC_NB : 0;
    bool piped = false;
    if constexpr (!JAG && !PRE && (NB % 2) == 0) piped = first > 0;
    if (!piped) {
      // by all warps: sub-tile i of them is box first + i / 4, quarter i % 4
      for (int i = warp; i < (nbox - first) * 4; i += 8) {
        const int bx = first + (i >> 2);
        cast_sub(sx + slot_of(bx) * CC_BOX_BYTES, bx * CC_BOXR + (i & 3) * 32 + rq * 8);
      }
      // the earlier boxes come back through the ring (from L2: read moments ago)
      if (first > 0) {
        refill_barrier();
        if (ok && tid == 0)
          for (int bx = 0; bx < first && bx < CC_NB; ++bx) issue(bx);
        for (int bx = 0; bx < first && ok; ++bx) {
          wait_slot(slot_of(bx));
          if (warp < 4) cast_sub(sx + slot_of(bx) * CC_BOX_BYTES, bx * CC_BOXR + warp * 32 + rq * 8);
          if (bx + CC_NB < first) {
            refill_barrier();
            if (ok && tid == 0) issue(bx + CC_NB);
          }
        }
      }
    } else {
      // A slice longer than the ring: two groups of four warps cast every
      // other box of the sequence [the CC_NB resident boxes, then boxes
      // 0 .. first - 1 again], a box's four 32-row quarters one per warp.
      // The box at position p + CC_NB of the sequence reloads into the slot
      // that position p frees (CC_NB is even: the same group), as soon as
      // the group is done with it, so the reloads (from L2: read moments
      // ago) overlap the casts of the resident boxes and both groups work
      // throughout.
      const int h = warp >> 2, wq = warp & 3;
      const int itid = h * 128;   // the group's issuing thread
      // the CTA's next unit, whose first CC_NB boxes load into the slots as
      // they are freed for the last time here (box b into slot b, where its
      // maxima pass expects it)
      int64_t gn = 0;
      int coln = 0;
      const bool more = cid + (k + 1) * ncl < a.units;
      if (more) unit_geom(k + 1, gn, coln);
      for (int p = h; p < nbox; p += 2) {
        const int bx = p < CC_NB ? first + p : p - CC_NB;
        const int slot = (int)((first + p) % CC_NB);
        if (p >= CC_NB && ok) {
          if (mbar_wait(&bars[slot], (phases >> slot) & 1u, nullptr)) {
            phases ^= 1u << slot;
            if (tid == itid) pending &= ~(1u << slot);
          } else {
            ok = false;   // the load stays pending: the exit path waits for it
          }
        }
        if (ok) cast_sub(sx + slot * CC_BOX_BYTES, bx * CC_BOXR + wq * 32 + rq * 8);
        if (p + CC_NB < nbox || more) {
          // the slot is free once the group's four warps are done with it
          fence_proxy_async_smem();
          if (h == 0) {
            asm volatile("bar.sync 1, 128;" ::: "memory");
          } else {
            asm volatile("bar.sync 2, 128;" ::: "memory");
          }
          if (tid == itid && ok) {
            if (p + CC_NB < nbox) {
              issue_at(slot, g, col0, p);
            } else {
              issue_at(slot, gn, coln, slot);
            }
          }
        }
      }
      preloaded = more ? CC_NB : 0;
      // every thread follows every slot's phase: the other group's reloads
      // (a slot serves one group here: positions p and p + CC_NB share it)
      for (int p = CC_NB + (h ^ 1); p < nbox; p += 2) phases ^= 1u << ((first + p) % CC_NB);
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok && tid == 0) set_status(a.status, FP8MOE_ERR_TIMEOUT);
    if (JAG && !fits && tid == 0) {
      // a unit that streamed on its own: the cursor resumes after it
      issued = base + nbox;
      pvalid = seek(kk + 1);
    }
    ub ^= 1;
    ++k;
    base += nbox;
  }
  if constexpr (JAG) {
    // the slack of q after the last group: columns [32 * sub-tiles, ldt)
    const int64_t E = a.E, last = gt_s.end[E - 1] - (E > 1 ? gt_s.end[E - 2] : 0);
    const int64_t from = 32 * (gt_s.pad[E - 1] + (last + 31) / 32);
    const int64_t chunks = (a.ldt - from) / 16;
    if (chunks > 0)
      for (int64_t i = (int64_t)blockIdx.x * CC_THREADS + tid; i < a.C * chunks; i += (int64_t)gridDim.x * CC_THREADS) {
        const int64_t row = i / chunks, ch = i - row * chunks;
        *reinterpret_cast<uint4*>(a.q + row * a.ldt + from + ch * 16) = make_uint4(0, 0, 0, 0);
      }
  }
  // after a load that timed out, wait (bounded) for the loads still in flight
  // (threads 0 and 128 issue loads)
  if (tid == 0 || tid == 128)
    for (int sl = 0; sl < CC_NB; ++sl)
      if (pending & (1u << sl)) (void)mbar_wait(&bars[sl], (phases >> sl) & 1u, nullptr);
  // no CTA leaves while its st.async to a peer may be in flight
  if constexpr (CL > 1) cluster_barrier();
}

template <int CL, int NB, bool PRE, bool FNUZ, bool JAG = false>
cudaError_t launch_cc(const CUtensorMap& tm, const CcArgs& a, int smem, int num_sms, cudaStream_t st) {
  auto kern = k_cw_cluster<CL, NB, PRE, FNUZ, JAG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(CC_THREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)CL);
  // persistent clusters: as many as are resident at once (per device and
  // shared-memory size: this cache holds the size it was computed for)
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  constexpr int kMaxDev = 64;
  static std::atomic<long long> cache[kMaxDev] = {};
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  long long c = cache[dev].load(std::memory_order_relaxed);
  int ncl = (int)(c & 0xFFFFFFFF);
  if ((int)(c >> 32) != smem || ncl <= 0) {
    if (cudaOccupancyMaxActiveClusters(&ncl, (void*)kern, &cfg) != cudaSuccess || ncl <= 0) {
      (void)cudaGetLastError();
      ncl = num_sms / CL;
    }
    if (ncl < 1) ncl = 1;
    cache[dev].store(((long long)smem << 32) | (unsigned)ncl, std::memory_order_relaxed);
  }
  // jagged: every resident cluster (the CTAs also zero the slack of q)
  const int64_t nc = JAG ? ncl : (a.units < ncl ? a.units : ncl);
  cfg.gridDim = dim3((unsigned)(CL * (nc < 1 ? 1 : nc)));
  return cudaLaunchKernelEx(&cfg, kern, tm, a);
}

template <bool PRE, bool FNUZ>
cudaError_t launch_cc_k(int CL, const CUtensorMap& tm, const CcArgs& a, int smem, int num_sms, cudaStream_t st) {
  switch (CL) {
    case 1: return launch_cc<1, CC_NB_MAX, PRE, FNUZ>(tm, a, smem, num_sms, st);
    case 2: return launch_cc<2, CC_NB_MAX, PRE, FNUZ>(tm, a, smem, num_sms, st);
    case 4: return launch_cc<4, CC_NB_MAX, PRE, FNUZ>(tm, a, smem, num_sms, st);
    default: return launch_cc<8, CC_NB_MAX, PRE, FNUZ>(tm, a, smem, num_sms, st);
  }
}

}  // namespace

// Jagged: clusters of two, a five-slot ring (the group table takes the room
// of the sixth at two CTAs per SM).
constexpr int CCJ_CL = 2, CCJ_NB = 5;

bool colwise_cluster_jagged_supported(int64_t E, int64_t R, int64_t C) {
  return E > 0 && E <= QG_MAX && R >= 0 && C > 0 && C % 16 == 0 && R < ((int64_t)1 << 31) - CC_BOXR &&
         C < ((int64_t)1 << 31);
}

cudaError_t launch_colwise_cluster_jagged(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                                          int kind, int64_t ldt, void* q, float* inv, int* status, int num_sms,
                                          cudaStream_t st) {
  CcArgs a;
  a.E = E;
  a.R = R;
  a.C = C;
  a.S = 0;
  a.n_ct = (C + CC_COLS - 1) / CC_COLS;
  a.units = E * a.n_ct;
  a.q = (uint8_t*)q;
  a.inv = inv;
  a.offs = offs;
  a.ldt = ldt;
  a.status = status;
  const int smem = CCJ_NB * CC_BOX_BYTES + 1024;
  CUtensorMap tm;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(R > 0 ? R : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)(C * 2)};
  cuuint32_t box[2] = {CC_COLS, CC_BOXR};
  if (!make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 2, dims, strides, box)) return cudaErrorInvalidValue;
  return kind == FP8MOE_E4M3FNUZ ? launch_cc<CCJ_CL, CCJ_NB, false, true, true>(tm, a, smem, num_sms, st)
                                 : launch_cc<CCJ_CL, CCJ_NB, false, false, true>(tm, a, smem, num_sms, st);
}

bool colwise_cluster_supported(int64_t E, int64_t R, int64_t C) {
  return E > 0 && R > 0 && C > 0 && R % 8 == 0 && C % 16 == 0 && E * R < ((int64_t)1 << 31) &&
         C < ((int64_t)1 << 31);
}

cudaError_t launch_colwise_cluster(const void* x, int64_t E, int64_t R, int64_t C, int kind, void* q, float* inv,
                                   int* status, int num_sms, cudaStream_t st) {
  // the smallest cluster whose CTAs' slices hold at most CC_STREAM_SLACK
  // boxes more than the ring (those few come back through it from L2),
  // the largest one when none does (its CTAs then stream their slices
  // through the ring); with room for two slices, the next unit's boxes load
  // during the cast.  Measured over eleven expert-weight shapes: every
  // doubling of the cluster costs more in per-unit waiting for the slowest
  // CTA than it saves, except where it takes a slice from more than
  // CC_STREAM_SLACK boxes over the ring down to that or fewer
  auto rows_per_cta = [&](int cl) { return (((R + cl - 1) / cl) + 31) / 32 * 32; };
  auto boxes_of = [&](int cl) { return (rows_per_cta(cl) + CC_BOXR - 1) / CC_BOXR; };
  int CL = 0;
  for (int cl = 1; cl <= 8 && !CL; cl *= 2)
    if (boxes_of(cl) <= CC_NB_MAX + CC_STREAM_SLACK) CL = cl;
  if (!CL) CL = 8;
  const bool pre = 2 * boxes_of(CL) <= CC_NB_MAX;
  CcArgs a;
  a.E = E;
  a.R = R;
  a.C = C;
  a.offs = nullptr;
  a.ldt = 0;
  a.S = rows_per_cta(CL);
  a.n_ct = (C + CC_COLS - 1) / CC_COLS;
  a.units = E * a.n_ct;
  a.q = (uint8_t*)q;
  a.inv = inv;
  a.status = status;
  const int smem = CC_NB_MAX * CC_BOX_BYTES + 1024;
  CUtensorMap tm;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)(E * R)};
  cuuint64_t strides[1] = {(cuuint64_t)(C * 2)};
  cuuint32_t box[2] = {CC_COLS, CC_BOXR};
  if (!make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, 2, dims, strides, box)) return cudaErrorInvalidValue;
  const bool fnuz = kind == FP8MOE_E4M3FNUZ;
  if (pre) return fnuz ? launch_cc_k<true, true>(CL, tm, a, smem, num_sms, st)
                       : launch_cc_k<true, false>(CL, tm, a, smem, num_sms, st);
  return fnuz ? launch_cc_k<false, true>(CL, tm, a, smem, num_sms, st)
              : launch_cc_k<false, false>(CL, tm, a, smem, num_sms, st);
}

}  // namespace fp8moe
