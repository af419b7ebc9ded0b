// Blockwise-scaled grouped GEMM on tcgen05 (sm_103a): forward, dgrad and
// wgrad of an MoE expert layer whose FP8 operands carry one fp32 scale per
// tile ("FP8-обучение на AMD", section "Скейлы: от тензора до микроблока":
// blockwise scaling, a scale per tile of fixed size; 1 x 128 tiles along the
// contracting dimension for the row operand, 128 x 128 tiles for the
// weights, 128-token tiles per group for both wgrad operands).
//
// The scales change every 128 elements of the contraction, so the tensor
// core cannot accumulate across k-blocks: each k-block's product goes to its
// own TMEM partial and is promoted into an fp32 accumulator held in
// registers, scaled by (row scale x column scale) of that k-block.
//  * persistent kernel, one CTA per SM; warp 0: TMA producer (A 128 x 128
//    and B BN x 128 byte tiles, 128-byte swizzle, 4-stage ring); warp 1:
//    TMEM allocator and MMA issuer (kind::f8f6f4, M = 128, N = BN, four
//    K = 32 steps per k-block); the group offsets and per-group tile counts
//    are copied to shared memory once;
//  * two TMEM partials (columns 0 and 256): the MMAs of k-block i + 1 run
//    while the epilogue promotes k-block i;
//  * the other warps: epilogue; warp w reads TMEM lanes 32 (w % 4) .. +31
//    and one column slice of the tile, holds its fp32 accumulators (part of
//    one output row per thread) and writes bf16 at the end through 2 KB
//    staging tiles (32 rows x 32 columns, 64-byte swizzle) handed to TMA
//    stores, so the LSU is not the bottleneck;
//  * forward / dgrad (tiles of K / 128 k-blocks, one scalar scale per
//    k-block and warp): BN = 256, eight epilogue warps of 128 columns, ten
//    warps in all, so 168 registers a thread (each SM sub-partition holds
//    16K registers and three of the warps).  Here the operand feed is the
//    bound: a 192-column tile moves more bytes per flop and ran 12% slower;
//  * wgrad (tiles of ~8 k-blocks, a scale per row and per column of every
//    k-block, so twice the promotion arithmetic): BN = 192, twelve epilogue
//    warps of 64 columns, three per sub-partition, so that one warp's TMEM
//    load latency hides behind the others' arithmetic; fourteen warps allow
//    128 registers a thread.  The N = 192 MMA takes as long as an N = 256
//    one (75% of the per-clock tensor peak at most); with 256 columns the
//    promotion was the bound, 15% slower;
//  * wgrad's row and column scales change with every k-block: the producer
//    bulk-copies each k-block's 128 + 192 of them into a ring slot that the
//    epilogue warps release, so the promotion loop makes no global loads;
//  * every wait is bounded; a timeout sets the device status word.
#include <cuda.h>

#include "common.cuh"
#include "gemm.h"
#include "launch.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace fp8moe {
namespace {

constexpr int BM = 128, BK = 128;
constexpr int PSTRIDE = 256;   // TMEM columns between the two partials
constexpr int A_BYTES = BM * BK;
constexpr int MAXG = 1024;
constexpr uint32_t TMEM_COLS = 512;

// Tile shape, warp roles and shared-memory layout of one mode.  Wgrad keeps
// two staging tiles per warp, so that a slice is written while the previous
// one's TMA store still reads (its stores recur 5x as often as forward's).
template <int MODE>
struct Cfg {
  static constexpr bool WG = MODE == GEMM_WGRAD;
  static constexpr int BN = WG ? 192 : 256;
  static constexpr int EPI_WARPS = WG ? 12 : 8;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // columns per epilogue thread
  static constexpr int LDW = WG ? 32 : 16;              // TMEM columns per load
  static constexpr int STAGES = 4;
  static constexpr int NSTG = WG ? 2 : 1;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // full, empty, cs_full, cs_empty per stage; pfull[2], pempty[2], drain
  static constexpr int bars = STAGES * STAGE_BYTES;
  static constexpr int misc = bars + (4 * STAGES + 6) * 8;  // tmem base, abort flag, total tiles
  static constexpr int colsc = misc + 16;                   // wgrad column scales [STAGES][BN]
  static constexpr int rowsc = colsc + STAGES * BN * 4;     // wgrad row scales [STAGES][BM]
  static constexpr int offs = rowsc + (WG ? STAGES * BM * 4 : 0);  // group ends [MAXG]
  static constexpr int tiles_prefix = offs + MAXG * 4;
  static constexpr int blk_prefix = tiles_prefix + (MAXG + 1) * 4;
  static constexpr int stg = (blk_prefix + (MAXG + 1) * 4 + 1023) / 1024 * 1024;  // [warps][NSTG][2 KB]
  static constexpr int total = stg + EPI_WARPS * 2048 * NSTG;
  static constexpr int SMEM_BYTES = total + 1024;
  static_assert(EPI_COLS % LDW == 0 && EPI_COLS % 64 == 0, "epilogue column split");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct BwParams {
  GemmArgs g;
  int n_tiles;    // output column tiles
  int m_tiles_w;  // wgrad: output row tiles per group
  int tma_out;    // output stored by TMA (tmOut valid)
};

struct BwTile {
  int e;
  int64_t row0, rows;    // output rows
  int64_t col0, ncols;   // output columns
  int64_t x0, kvalid;    // contraction start and length
  int nk;                // k-blocks
  int64_t blk0;          // wgrad: first token block of the group
};

template <int MODE>
FP8MOE_DEV BwTile bw_tile(const BwParams& p, const int* offs, const int* tiles_prefix, const int* blk_prefix, int t) {
  constexpr bool WGRAD = MODE == GEMM_WGRAD;
  constexpr int BN = Cfg<MODE>::BN;
  const GemmArgs& g = p.g;
  int lo = 0, hi = g.E - 1, e = 0;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (tiles_prefix[mid] <= t) {
      e = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  const int local = t - tiles_prefix[e];
  const int64_t gs = e == 0 ? 0 : offs[e - 1];
  const int64_t ge = offs[e];
  BwTile tl;
  tl.e = e;
  if (!WGRAD) {
    // m-tiles of the group fastest: CTAs running together share the B tile
    const int mt = (int)((ge - gs + BM - 1) / BM);
    const int ni = local / mt, mi = local % mt;
    tl.row0 = gs + (int64_t)mi * BM;
    tl.rows = min((int64_t)BM, ge - tl.row0);
    tl.col0 = (int64_t)ni * BN;
    tl.x0 = 0;
    tl.kvalid = g.kk;
    tl.blk0 = 0;
  } else {
    const int ni = local / p.m_tiles_w, mi = local % p.m_tiles_w;
    tl.row0 = (int64_t)mi * BM;
    tl.rows = min((int64_t)BM, g.rows - tl.row0);
    tl.col0 = (int64_t)ni * BN;
    tl.x0 = gs;
    tl.kvalid = ge - gs;
    tl.blk0 = blk_prefix[e];
  }
  tl.ncols = min((int64_t)BN, g.cols - tl.col0);
  tl.nk = (int)((tl.kvalid + BK - 1) / BK);
  return tl;
}

template <int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::THREADS, 1)
    k_blockwise_mm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmOut, BwParams p) {
  using C = Cfg<MODE>;
  constexpr bool WGRAD = C::WG;
  constexpr int STAGES = C::STAGES, NSTG = C::NSTG, BN = C::BN, THREADS = C::THREADS;
  constexpr int EPI_WARPS = C::EPI_WARPS, EPI_COLS = C::EPI_COLS, LDW = C::LDW;
  constexpr int STAGE_BYTES = C::STAGE_BYTES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* full = (uint64_t*)(smem + C::bars);
  uint64_t* empty = full + STAGES;
  uint64_t* cs_full = empty + STAGES;
  uint64_t* cs_empty = cs_full + STAGES;
  uint64_t* pfull = cs_empty + STAGES;
  uint64_t* pempty = pfull + 2;
  uint64_t* drain = pempty + 2;  // the MMA thread's own work, awaited before TMEM is released
  uint32_t* tmem_holder = (uint32_t*)(smem + C::misc);
  volatile int* abort_flag = (volatile int*)(smem + C::misc + 4);
  int* total_s = (int*)(smem + C::misc + 8);
  float* colsc = (float*)(smem + C::colsc);
  float* rowsc = (float*)(smem + C::rowsc);
  int* offs_s = (int*)(smem + C::offs);
  int* tiles_prefix = (int*)(smem + C::tiles_prefix);
  int* blk_prefix = (int*)(smem + C::blk_prefix);
  const GemmArgs& g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&cs_full[s], 1);
      mbar_init(&cs_empty[s], EPI_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    tc_fence_before();
  }
  // per-group tile and token-block counts, then one warp scans them and
  // validates the offsets
  for (int e = threadIdx.x; e < g.E; e += THREADS) {
    const int32_t end = g.offs[e];
    offs_s[e] = end;
    const int64_t sz = (int64_t)end - (e == 0 ? 0 : g.offs[e - 1]);
    int nt, nb = 0;
    if (!WGRAD) {
      nt = (int)((sz + BM - 1) / BM) * p.n_tiles;
    } else {
      nt = p.m_tiles_w * p.n_tiles;
      nb = (int)((sz + 127) / 128);
    }
    tiles_prefix[e + 1] = sz < 0 ? 0 : nt;
    blk_prefix[e + 1] = sz < 0 ? 0 : nb;
  }
  __syncthreads();
  if (warp == 0) {
    int bad = 0, carry_t = 0, carry_b = 0;
    for (int base = 0; base < g.E; base += 32) {
      const int e = base + lane;
      int vt = 0, vb = 0;
      if (e < g.E) {
        const int64_t gs = e == 0 ? 0 : g.offs[e - 1];
        const int64_t ge = g.offs[e];
        if (ge < gs || ge > g.M || (e == g.E - 1 && ge != g.M)) bad = 1;
        if (WGRAD && (ge % 32)) bad = 1;
        vt = tiles_prefix[e + 1];
        vb = blk_prefix[e + 1];
      }
      for (int o = 1; o < 32; o <<= 1) {
        const int ut = __shfl_up_sync(0xffffffffu, vt, o);
        const int ub = __shfl_up_sync(0xffffffffu, vb, o);
        if (lane >= o) {
          vt += ut;
          vb += ub;
        }
      }
      if (e < g.E) {
        tiles_prefix[e + 1] = carry_t + vt;
        blk_prefix[e + 1] = carry_b + vb;
      }
      carry_t += __shfl_sync(0xffffffffu, vt, 31);
      carry_b += __shfl_sync(0xffffffffu, vb, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      tiles_prefix[0] = 0;
      blk_prefix[0] = 0;
      *total_s = bad ? 0 : carry_t;
      if (bad && blockIdx.x == 0) set_status(g.status, FP8MOE_ERR_DEVICE_OFFSETS);
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = *total_s;

  if (warp == 0 && lane == 0) {
    // ======================= TMA producer =======================
    int stage = 0;
    uint32_t phase = 0;
    int filled[STAGES], cs_filled[STAGES];  // phase of each slot's last fill, -1: never
    for (int s2 = 0; s2 < STAGES; ++s2) filled[s2] = cs_filled[s2] = -1;
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
      const BwTile tl = bw_tile<MODE>(p, offs_s, tiles_prefix, blk_prefix, t);
      for (int ks = 0; ks < tl.nk; ++ks) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
          set_status(g.status, FP8MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        filled[stage] = (int)phase;
        uint8_t* sa = smem + stage * STAGE_BYTES;
        mbar_expect_tx(&full[stage], STAGE_BYTES);
        const int x = (int)(tl.x0 + (int64_t)ks * BK);
        tma_load_2d(sa, &tmA, &full[stage], x, (int)tl.row0);
        if (WGRAD) {
          tma_load_2d(sa + A_BYTES, &tmB, &full[stage], x, (int)tl.col0);
          // this k-block's column and row scales (the epilogue released the
          // slot); rows and columns are multiples of 128, the scale arrays
          // 16-byte aligned
          if (!mbar_wait(&cs_empty[stage], phase ^ 1, abort_flag)) {
            set_status(g.status, FP8MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          const uint32_t cbytes = (uint32_t)(tl.ncols * 4), rbytes = (uint32_t)(tl.rows * 4);
          cs_filled[stage] = (int)phase;
          mbar_expect_tx(&cs_full[stage], cbytes + rbytes);
          bulk_load(colsc + stage * BN, (const float*)g.b_scale + (tl.blk0 + ks) * g.cols + tl.col0, cbytes,
                    &cs_full[stage]);
          bulk_load(rowsc + stage * BM, (const float*)g.a_scale + (tl.blk0 + ks) * g.rows + tl.row0, rbytes,
                    &cs_full[stage]);
        } else {
          tma_load_3d(sa + A_BYTES, &tmB, &full[stage], x, (int)tl.col0, tl.e);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // every stage's MMAs have completed (their loads landed), and the
    // epilogue has read every column-scale slot, before exit
    for (int i = 0; i < STAGES && !*abort_flag; ++i) {
      if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag) ||
          (WGRAD && !mbar_wait(&cs_empty[stage], phase ^ 1, abort_flag))) {
        set_status(g.status, FP8MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }
    // after a timeout: wait (bounded) until the copies in flight have landed
    if (*abort_flag) {
      for (int s2 = 0; s2 < STAGES; ++s2) {
        if (filled[s2] >= 0) (void)mbar_wait(&full[s2], (uint32_t)filled[s2], nullptr);
        if (WGRAD && cs_filled[s2] >= 0) (void)mbar_wait(&cs_full[s2], (uint32_t)cs_filled[s2], nullptr);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ======================= MMA issuer =======================
    int stage = 0;
    uint32_t phase = 0;
    uint32_t np = 0;  // partials issued
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
      const BwTile tl = bw_tile<MODE>(p, offs_s, tiles_prefix, blk_prefix, t);
      bool ok = true;
      for (int ks = 0; ks < tl.nk; ++ks) {
        const uint32_t buf = np & 1, use = np >> 1;
        if (!mbar_wait(&full[stage], phase, abort_flag) || !mbar_wait(&pempty[buf], (use & 1) ^ 1, abort_flag)) {
          set_status(g.status, FP8MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
        const uint64_t adesc = sdesc_sw128(a_addr), bdesc = sdesc_sw128(a_addr + A_BYTES);
        const uint32_t d = tmem_base + buf * PSTRIDE;
        const int64_t rem = tl.kvalid - (int64_t)ks * BK;
        if (rem >= BK) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8<false>(d, adesc + (uint64_t)(k * 2), bdesc + (uint64_t)(k * 2), idesc_f8n<BM, BN>(), k > 0);
        } else {
          const int nsub = (int)((rem + 31) / 32);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k < nsub)
              mma_f8<false>(d, adesc + (uint64_t)(k * 2), bdesc + (uint64_t)(k * 2), idesc_f8n<BM, BN>(), k > 0);
        }
        tc_commit(&empty[stage]);
        tc_commit(&pfull[buf]);
        ++np;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    // every MMA this thread issued has completed before TMEM is released
    tc_commit(drain);
    if (!mbar_wait(drain, 0, nullptr)) set_status(g.status, FP8MOE_ERR_TIMEOUT);
  } else if (warp >= 2) {
    // ======================= epilogue: promotion and stores =======================
    const int quarter = warp & 3;
    const int part = (warp - 2) >> 2;  // column slice of the tile
    const int lrow = quarter * 32 + lane;
    const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + part * EPI_COLS;
    uint8_t* stg0 = smem + C::stg + (warp - 2) * 2048 * NSTG;
    int slice = 0;  // slices staged by this warp (alternating tiles when NSTG == 2)
    const float* sa_p = (const float*)g.a_scale;
    const float* sb_p = (const float*)g.b_scale;
    uint32_t np = 0;
    for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
      const int64_t c0 = part * EPI_COLS;  // first column of this thread inside the tile
      // only the scale pointers and the k-block count live through the
      // promotion loop; the tile's geometry is recomputed for the stores
      int nk;
      const float* rsp;  // row scale of k-block 0 (nullptr: row past the tile)
      const float* csp;  // forward / dgrad: column scale of k-block 0 (nullptr: columns past the output)
      {
        const BwTile tl = bw_tile<MODE>(p, offs_s, tiles_prefix, blk_prefix, t);
        nk = tl.nk;
        if (nk == 0) {
          // an empty group in wgrad: dW[e] = 0
          if (lrow < tl.rows) {
            uint16_t* orow = g.out + ((int64_t)tl.e * g.rows + tl.row0 + lrow) * g.cols + tl.col0;
            for (int c = (int)c0; c < c0 + EPI_COLS && c < tl.ncols; c += 8)
              *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          }
          continue;
        }
        rsp = lrow >= tl.rows ? nullptr
                              : WGRAD ? sa_p + tl.blk0 * g.rows + tl.row0 + lrow : sa_p + tl.row0 + lrow;
        const int64_t cb = (tl.col0 + c0) / 128;
        csp = WGRAD || cb * 128 >= g.cols ? nullptr
              : MODE == GEMM_FWD          ? sb_p + ((int64_t)tl.e * (g.cols / 128) + cb) * (g.kk / 128)
                                          : sb_p + (int64_t)tl.e * (g.kk / 128) * (g.cols / 128) + cb;
      }
      // scale of k-block ks: row part (per thread) and column part (one per
      // warp's columns for forward / dgrad, per column for wgrad)
      auto row_scale = [&](int ks) -> float {
        if (WGRAD || rsp == nullptr) return 0.0f;  // wgrad: from the ring
        return rsp[(int64_t)ks * (WGRAD ? g.rows : g.M)];
      };
      auto col_scale = [&](int ks) -> float {
        if (WGRAD) return 1.0f;  // per column, from the ring
        if (csp == nullptr) return 0.0f;
        return csp[MODE == GEMM_FWD ? (int64_t)ks : (int64_t)ks * (g.cols / 128)];   // dgrad: W^T tiles
      };
      // column pairs: the promotion runs on packed fp32x2 multiplies / FMAs
      float2 acc[EPI_COLS / 2];
#pragma unroll
      for (int j = 0; j < EPI_COLS / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
      float rs_next = row_scale(0), cs_next = col_scale(0);
      bool ok = true;
      for (int ks = 0; ks < nk; ++ks) {
        const float rs = rs_next, cs = cs_next;
        if (ks + 1 < nk) {
          rs_next = row_scale(ks + 1);
          cs_next = col_scale(ks + 1);
        }
        const float* csv = nullptr;
        const int slot = (int)(np % STAGES);
        if (WGRAD) {
          if (!mbar_wait(&cs_full[slot], (np / STAGES) & 1, abort_flag)) {
            set_status(g.status, FP8MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
          }
          csv = colsc + slot * BN + c0;
        }
        const uint32_t pb = np & 1, use = np >> 1;
        if (!mbar_wait(&pfull[pb], use & 1, abort_flag)) {
          set_status(g.status, FP8MOE_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = WGRAD ? rowsc[slot * BM + lrow] : rs * cs;
#pragma unroll
        for (int c = 0; c < EPI_COLS; c += LDW) {
          uint32_t r[LDW];
          if constexpr (LDW == 32) {
            tmem_ld32(taddr + pb * PSTRIDE + c, r);
          } else {
            tmem_ld16(taddr + pb * PSTRIDE + c, r);
          }
          tmem_ld_wait();
          const float2 f2 = make_float2(f, f);
          if constexpr (WGRAD) {
            // the product times its column scale, then times the row scale
#pragma unroll
            for (int j = 0; j < LDW; j += 2) {
              const float2 cv = *reinterpret_cast<const float2*>(csv + c + j);
              const float2 pr = __fmul2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), cv);
              acc[(c + j) / 2] = __ffma2_rn(pr, f2, acc[(c + j) / 2]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < LDW; j += 2)
              acc[(c + j) / 2] =
                  __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), f2, acc[(c + j) / 2]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&pempty[pb]);
          if (WGRAD) mbar_arrive(&cs_empty[slot]);
        }
        ++np;
      }
      if (!ok) break;
      const BwTile tl = bw_tile<MODE>(p, offs_s, tiles_prefix, blk_prefix, t);
      // 32-column slices through the warp's staging tile: 16-byte chunk ch
      // of row r at r * 64 + ((ch ^ ((r >> 1) & 3)) << 4) (the 64-byte
      // swizzle of the output map; conflict-free for the row-per-lane writes
      // and the 2-rows-per-8-lanes reads).  A warp whose 32 rows all belong
      // to the tile hands the slice to a TMA store (wgrad's 3-D map clips
      // rows past N); otherwise the lanes store with bounds checks.
      const bool tma = p.tma_out && (WGRAD ? quarter * 32 < tl.rows : (quarter + 1) * 32 <= tl.rows);
      if (!tma && quarter * 32 >= tl.rows) continue;
#pragma unroll
      for (int j = 0; j < EPI_COLS / 32; ++j) {
        const int64_t cc = c0 + j * 32;  // tile column of the slice
        if (cc < tl.ncols) {
          uint8_t* stg = stg0 + (slice % NSTG) * 2048;
          ++slice;
          // the store that last read this staging tile is done with it
          if (lane == 0) {
            if (tma && NSTG == 2) {
              bulk_wait_read<1>();
            } else {
              bulk_wait_read<0>();
            }
          }
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int a0 = j * 32 + c * 8;
            *reinterpret_cast<uint4*>(stg + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(pack_bf16(acc[a0 / 2].x, acc[a0 / 2].y), pack_bf16(acc[a0 / 2 + 1].x, acc[a0 / 2 + 1].y),
                           pack_bf16(acc[a0 / 2 + 2].x, acc[a0 / 2 + 2].y),
                           pack_bf16(acc[a0 / 2 + 3].x, acc[a0 / 2 + 3].y));
          }
          if (tma) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (WGRAD) {
                tma_store_3d(&tmOut, stg, (int)(tl.col0 + cc), (int)(tl.row0 + quarter * 32), tl.e);
              } else {
                tma_store_2d(&tmOut, stg, (int)(tl.col0 + cc), (int)(tl.row0 + quarter * 32));
              }
              bulk_commit();
            }
          } else {
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = i * 8 + (lane >> 2), ch = lane & 3;
              const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
              const int64_t trow = quarter * 32 + r, col = cc + ch * 8;
              if (trow < tl.rows && col < tl.ncols) {
                uint16_t* o = WGRAD ? g.out + ((int64_t)tl.e * g.rows + tl.row0 + trow) * g.cols + tl.col0 + col
                                    : g.out + (tl.row0 + trow) * g.cols + tl.col0 + col;
                *reinterpret_cast<uint4*>(o) = v;
              }
            }
            __syncwarp();
          }
        }
      }
    }
    // the staged stores have left shared memory before the CTA exits
    if (lane == 0) bulk_wait_all();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
  }
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to, const BwParams& p,
                        int64_t tiles, cudaStream_t st) {
  auto kern = k_blockwise_mm<MODE>;
  constexpr int SMEM_BYTES = Cfg<MODE>::SMEM_BYTES, THREADS = Cfg<MODE>::THREADS;
  if (SMEM_BYTES > p.g.max_smem) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t grid = tiles < p.g.num_sms ? tiles : p.g.num_sms;
  kern<<<(unsigned)(grid > 0 ? grid : 1), THREADS, SMEM_BYTES, st>>>(ta, tb, to, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_blockwise_mm(const GemmArgs& g, cudaStream_t st) {
  if (g.E > MAXG) return cudaErrorNotSupported;
  if (g.kk > INT32_MAX || g.rows > INT32_MAX || g.cols > INT32_MAX || g.M > INT32_MAX) return cudaErrorInvalidValue;
  const bool wgrad = g.mode == GEMM_WGRAD;
  const int bn = wgrad ? Cfg<GEMM_WGRAD>::BN : Cfg<GEMM_FWD>::BN;
  BwParams p;
  p.g = g;
  p.n_tiles = (int)((g.cols + bn - 1) / bn);
  p.m_tiles_w = (int)((g.rows + BM - 1) / BM);
  CUtensorMap ta, tb;
  {
    const int64_t arows = wgrad ? g.rows : g.M;
    cuuint64_t dims[2] = {(cuuint64_t)g.kk, (cuuint64_t)(arows > 0 ? arows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)g.kk};
    cuuint32_t box[2] = {BK, BM};
    if (!make_tmap(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.a, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  if (wgrad) {
    cuuint64_t dims[2] = {(cuuint64_t)g.kk, (cuuint64_t)g.cols};
    cuuint64_t strides[1] = {(cuuint64_t)g.kk};
    cuuint32_t box[2] = {BK, (cuuint32_t)bn};
    if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.b, 2, dims, strides, box)) return cudaErrorInvalidValue;
  } else {
    cuuint64_t dims[3] = {(cuuint64_t)g.kk, (cuuint64_t)g.cols, (cuuint64_t)g.E};
    cuuint64_t strides[2] = {(cuuint64_t)g.kk, (cuuint64_t)(g.kk * g.cols)};
    cuuint32_t box[3] = {BK, (cuuint32_t)bn, 1};
    if (!make_tmap(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.b, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  // bf16 output slices of 32 columns x 32 rows, 64-byte swizzle; wgrad as
  // [E, rows, cols] so that rows past an expert are clipped
  CUtensorMap to = ta;
  p.tma_out = 0;
  if (((uintptr_t)g.out % 16) == 0) {
    bool ok;
    if (wgrad) {
      cuuint64_t dims[3] = {(cuuint64_t)g.cols, (cuuint64_t)g.rows, (cuuint64_t)g.E};
      cuuint64_t strides[2] = {(cuuint64_t)(g.cols * 2), (cuuint64_t)(g.rows * g.cols * 2)};
      cuuint32_t box[3] = {32, 32, 1};
      ok = make_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_UINT16, g.out, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
    } else {
      cuuint64_t dims[2] = {(cuuint64_t)g.cols, (cuuint64_t)(g.M > 0 ? g.M : 1)};
      cuuint64_t strides[1] = {(cuuint64_t)(g.cols * 2)};
      cuuint32_t box[2] = {32, 32};
      ok = make_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_UINT16, g.out, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
    }
    p.tma_out = ok ? 1 : 0;
  }
  // an upper bound on the tiles (the exact count needs the offsets)
  const int64_t tiles = wgrad ? (int64_t)g.E * p.m_tiles_w * p.n_tiles
                              : ((g.M + BM - 1) / BM + g.E) * (int64_t)p.n_tiles;
  if (g.mode == GEMM_FWD) return launch_mode<GEMM_FWD>(ta, tb, to, p, tiles, st);
  if (g.mode == GEMM_DGRAD) return launch_mode<GEMM_DGRAD>(ta, tb, to, p, tiles, st);
  return launch_mode<GEMM_WGRAD>(ta, tb, to, p, tiles, st);
}

}  // namespace fp8moe
