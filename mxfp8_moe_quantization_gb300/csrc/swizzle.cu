// 128x4 tiled layout of e8m0 scale factors for tcgen05 block-scaled MMA.
//
// "Accelerating Llama4 Scout training with TorchAO MXFP8 MoE primitives",
// section details and the caption of its 128x4 tile layout table: a dedicated
// kernel rearranges row-major scale factors into 128x4 tiles.  The byte order
// inside a tile is the one tcgen05 consumes: 512 bytes per tile, element
// (r, c) at (r % 32) * 16 + (r / 32) * 4 + c, i.e. 32 rows of 16 bytes, each
// holding rows r, r+32, r+64, r+96 -- one 16-byte row per TMEM lane.
//
// A 128-row block of the tiled output is one contiguous region, and its
// source rows are contiguous too (groups are padded to whole tiles), so each
// CTA stages the block's source rows (a chunk of up to 128 scale columns) in
// shared memory with coalesced loads and writes the tiles with contiguous
// 16-byte stores; every output byte, padding included, is written once.
// Group boundaries come from device offsets: each group starts a new 128-row
// block (rows) or 4-column block (columns).
#include "common.cuh"
#include "launch.h"
#include "scales.cuh"
#include "tma.cuh"

#include <type_traits>

namespace fp8moe {

SwizzleGeom swizzle_geom(int64_t R, int64_t Cs, int64_t E, int group_axis) {
  int64_t rb = (R + 127) / 128, cb = (Cs + 3) / 4;
  if (group_axis == FP8MOE_GROUP_ROWS) rb += E;
  if (group_axis == FP8MOE_GROUP_COLS) cb += E;
  return SwizzleGeom{rb * 128, cb * 4};
}

constexpr int SW_CC = 128;             // padded scale columns per chunk
constexpr int SW_PITCH = SW_CC + 4;    // staged row: 33 words, so the 32 rows a warp reads hit 32 banks

struct SwizzleArgs {
  const uint8_t* s;
  int64_t B, R, Cs;
  const int32_t* offs;
  int E;
  int group_axis;
  int64_t Rp, Cp;
  uint8_t* out;
  int* status;
};

// Source column of padded column pc in GROUP_COLS mode (-1 in a padding
// column), and the source position the chunk boundary pc maps to.
FP8MOE_DEV int find_last_le(const int64_t* pad, int E, int64_t key) {
  int lo = 0, hi = E - 1, g = 0;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if (pad[mid] <= key) {
      g = mid;
      lo = mid + 1;
    } else {
      hi = mid - 1;
    }
  }
  return g;
}

__global__ void __launch_bounds__(256) k_swizzle(SwizzleArgs a) {
  __shared__ GroupTable gt;
  __shared__ __align__(16) uint8_t tile[128 * SW_PITCH];
  const bool grouped = a.group_axis != FP8MOE_NO_GROUPS;
  const bool gcols = a.group_axis == FP8MOE_GROUP_COLS, grows = a.group_axis == FP8MOE_GROUP_ROWS;
  if (grouped) build_group_table(gt, a.offs, a.E, grows ? a.R : a.Cs * 32, grows ? GT_ROWS128 : GT_COLS, a.status);
  const bool bad = grouped && gt.bad;
  // source column position of padded column pc (GROUP_COLS): inside group g,
  // or the end of g's source columns when pc lies in g's padding
  auto src_pos = [&](int64_t pc, bool& valid) -> int64_t {
    if (!gcols) {
      valid = pc < a.Cs;
      return pc < a.Cs ? pc : a.Cs;
    }
    const int g = find_last_le(gt.pad, a.E, pc);
    const int64_t st = (g == 0 ? 0 : gt.end[g - 1]) / 32, sz = gt.end[g] / 32 - st, w = pc - gt.pad[g];
    valid = w < sz;
    return st + (w < sz ? w : sz);
  };
  const int64_t nrb = a.Rp / 128, ncc = (a.Cp + SW_CC - 1) / SW_CC;
  const bool words = !gcols && (a.Cs % 4) == 0;  // 4-byte loads: rows and chunk starts are word-aligned
  for (int64_t u = blockIdx.x; u < a.B * nrb * ncc; u += gridDim.x) {
    const int64_t b = u / (nrb * ncc), rbk = (u / ncc) % nrb, cc = u % ncc;
    const int64_t pc0 = cc * SW_CC;
    const int pcn = (int)min((int64_t)SW_CC, a.Cp - pc0);
    // source rows of this padded row block
    int64_t r0 = rbk * 128, rn;
    if (grows) {
      const int g = find_last_le(gt.pad, a.E, rbk * 128);
      const int64_t st = g == 0 ? 0 : gt.end[g - 1], w = rbk * 128 - gt.pad[g];
      r0 = st + w;
      rn = gt.end[g] - r0;
    } else {
      rn = a.R - r0;
    }
    rn = bad ? 0 : (rn < 0 ? 0 : (rn > 128 ? 128 : rn));
    bool v_unused;
    const int64_t s_lo = src_pos(pc0, v_unused), s_hi = src_pos(pc0 + pcn, v_unused);
    const int span = bad ? 0 : (int)(s_hi - s_lo);
    __syncthreads();  // the previous unit's reads of the staged rows are done
    const uint8_t* src = a.s + (b * a.R + r0) * a.Cs + s_lo;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (words) {
      // warp w stages rows w, w + 8, ...; lane j their word j (spans are at
      // most 32 words), 16 loads in flight per lane
      const int spw = span / 4;
      uint32_t wv[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int i = warp + 8 * t;
        wv[t] = i < rn && lane < spw ? __ldg(reinterpret_cast<const uint32_t*>(src + (int64_t)i * a.Cs) + lane) : 0u;
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int i = warp + 8 * t;
        if (i < rn && lane < spw) *reinterpret_cast<uint32_t*>(tile + i * SW_PITCH + lane * 4) = wv[t];
      }
    } else {
      for (int i = warp; i < rn; i += 8)
        for (int j = lane; j < span; j += 32) tile[i * SW_PITCH + j] = __ldg(src + (int64_t)i * a.Cs + j);
    }
    __syncthreads();
    // tiles (rbk, pc0/4 ...) are consecutive 512-byte blocks of the output
    uint4* dst = reinterpret_cast<uint4*>(a.out + b * a.Rp * a.Cp + (rbk * (a.Cp / 4) + pc0 / 4) * 512);
    for (int k = threadIdx.x; k < (pcn / 4) * 32; k += 256) {
      const int t = k >> 5, r32 = k & 31;
      // the tile's 4 padded columns: first staged column and how many hold data
      bool v0;
      const int64_t sp = src_pos(pc0 + 4 * t, v0);
      int nvalid = 0;
      if (!bad) {
        if (gcols) {
          bool vv;
          const int64_t e4 = src_pos(pc0 + 4 * t + 3, vv);
          nvalid = v0 ? (int)(e4 - sp) + (vv ? 1 : 0) : 0;
        } else {
          nvalid = (int)min((int64_t)4, a.Cs - (pc0 + 4 * t));
          nvalid = nvalid < 0 ? 0 : nvalid;
        }
      }
      const int lc = (int)(sp - s_lo);
      uint32_t w[4];
      if (nvalid == 4 && (lc & 3) == 0) {
        // a whole aligned word of each of the four rows
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = r32 + 32 * q;
          w[q] = i < rn ? *reinterpret_cast<const uint32_t*>(tile + i * SW_PITCH + lc) : 0u;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = r32 + 32 * q;
          uint32_t word = 0;
          if (i < rn) {
            const uint8_t* row = tile + i * SW_PITCH + lc;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
              if (c4 < nvalid) word |= (uint32_t)row[c4] << (8 * c4);
          }
          w[q] = word;
        }
      }
      dst[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Rows of whole 16-byte chunks (Cs % 16 == 0), without column groups: the
// source rows of a padded 128-row block are contiguous (groups are padded to
// whole blocks), so one bulk copy brings the block into shared memory, and
// every CTA has its block's load in flight at once (a 21 MB tiling is one
// round of loads, where the staged kernel above takes two or three rounds of
// load, then store).  A thread then takes the 16-byte chunk j of rows r32,
// r32 + 32, r32 + 64 and r32 + 96: word s of each holds that row's columns
// of tile 4j + s, so the four words make the tile's 16 output bytes at row
// r32; a warp's stores cover a whole 512-byte tile.
constexpr int SWR_THREADS = 128;
constexpr int64_t SWR_MAX_CS = 384;   // a block of at most 48 KB

template <bool GROWS>
__global__ void __launch_bounds__(SWR_THREADS) k_swizzle_rows(SwizzleArgs a) {
  extern __shared__ __align__(128) uint8_t rows[];
  __shared__ uint64_t bar;
  __shared__ std::conditional_t<GROWS, GroupTable, char> gt_s;
  bool bad = false;
  if constexpr (GROWS) {
    build_group_table(gt_s, a.offs, a.E, a.R, GT_ROWS128, a.status);
    bad = gt_s.bad;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  const int64_t nrb = a.Rp / 128;
  const int nch = (int)(a.Cs / 16);
  uint32_t phase = 0;
  bool ok = true;
  int lost = -1;   // thread 0: the phase of a load whose wait ran out
  for (int64_t u = blockIdx.x; u < a.B * nrb; u += gridDim.x) {
    const int64_t b = u / nrb, rbk = u - b * nrb;
    int64_t r0 = rbk * 128, rn;
    if constexpr (GROWS) {
      const int g = find_last_le(gt_s.pad, a.E, rbk * 128);
      const int64_t st = g == 0 ? 0 : gt_s.end[g - 1];
      r0 = st + (rbk * 128 - gt_s.pad[g]);
      rn = gt_s.end[g] - r0;
    } else {
      rn = a.R - r0;
    }
    rn = bad ? 0 : (rn < 0 ? 0 : (rn > 128 ? 128 : rn));
    const uint32_t bytes = (uint32_t)(rn * a.Cs);
    // the previous block's reads (generic proxy) come before the copy's writes
    fence_proxy_async_smem();
    ok = __syncthreads_and(ok) != 0;
    if (bytes > 0) {
      if (threadIdx.x == 0 && ok) {
        mbar_expect_tx(&bar, bytes);
        bulk_load(rows, a.s + (b * a.R + r0) * a.Cs, bytes, &bar);
      }
      if (ok && !mbar_wait(&bar, phase, nullptr)) {
        ok = false;
        if (threadIdx.x == 0) {
          set_status(a.status, FP8MOE_ERR_TIMEOUT);
          lost = (int)phase;
        }
      }
      phase ^= 1;
    }
    uint4* dst = reinterpret_cast<uint4*>(a.out + b * a.Rp * a.Cp + rbk * (a.Cp / 4) * 512);
    for (int e = threadIdx.x; e < 32 * nch; e += SWR_THREADS) {
      const int j = e >> 5, r32 = e & 31;
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = r32 + 32 * q;
        v[q] = i < rn && ok ? *reinterpret_cast<const uint4*>(rows + (int64_t)i * a.Cs + 16 * j)
                            : make_uint4(0, 0, 0, 0);
      }
      dst[(4 * j + 0) * 32 + r32] = make_uint4(v[0].x, v[1].x, v[2].x, v[3].x);
      dst[(4 * j + 1) * 32 + r32] = make_uint4(v[0].y, v[1].y, v[2].y, v[3].y);
      dst[(4 * j + 2) * 32 + r32] = make_uint4(v[0].z, v[1].z, v[2].z, v[3].z);
      dst[(4 * j + 3) * 32 + r32] = make_uint4(v[0].w, v[1].w, v[2].w, v[3].w);
    }
  }
  // a load whose wait ran out may still land: wait for it (bounded) before
  // the shared memory goes away
  if (lost >= 0) (void)mbar_wait(&bar, (uint32_t)lost, nullptr);
}

cudaError_t launch_swizzle(const uint8_t* s, int64_t B, int64_t R, int64_t Cs, const int32_t* offs,
                           int64_t E, int group_axis, uint8_t* out, int* status, int num_sms,
                           cudaStream_t st) {
  SwizzleArgs a;
  const SwizzleGeom g = swizzle_geom(R, Cs, group_axis == FP8MOE_NO_GROUPS ? 0 : E, group_axis);
  a.s = s;
  a.B = B;
  a.R = R;
  a.Cs = Cs;
  a.offs = offs;
  a.E = (int)E;
  a.group_axis = group_axis;
  a.Rp = g.Rp;
  a.Cp = g.Cp;
  a.out = out;
  a.status = status;
  if (group_axis != FP8MOE_GROUP_COLS && Cs % 16 == 0 && Cs <= SWR_MAX_CS &&
      (reinterpret_cast<uintptr_t>(s) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const int64_t blocks_all = B * (g.Rp / 128);
    if (blocks_all == 0) return cudaSuccess;
    const size_t smem = (size_t)(128 * Cs);
    const bool grows = group_axis == FP8MOE_GROUP_ROWS;
    // resident CTAs per SM at this block size (cached per variant and size)
    static std::atomic<long long> occ[2];
    long long c = occ[grows].load(std::memory_order_relaxed);
    int per = (int)(c & 0xFFFFFFFF);
    if ((size_t)(c >> 32) != smem || per <= 0) {
      auto kern = grows ? k_swizzle_rows<true> : k_swizzle_rows<false>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, SWR_THREADS, smem) != cudaSuccess || per < 1) {
        (void)cudaGetLastError();
        per = 2;
      }
      occ[grows].store(((long long)smem << 32) | (unsigned)per, std::memory_order_relaxed);
    }
    const int64_t cap = (int64_t)num_sms * per;
    const int64_t blocks = blocks_all < cap ? blocks_all : cap;
    if (grows)
      k_swizzle_rows<true><<<(unsigned)blocks, SWR_THREADS, smem, st>>>(a);
    else
      k_swizzle_rows<false><<<(unsigned)blocks, SWR_THREADS, smem, st>>>(a);
    return cudaGetLastError();
  }
  const int64_t units = B * (g.Rp / 128) * ((g.Cp + SW_CC - 1) / SW_CC);
  if (units == 0) return cudaSuccess;
  // as many CTAs as fit on the GPU at once (each unit is a load-then-store
  // round trip, so more units in flight hide more DRAM latency)
  static std::atomic<int> per_sm{0};
  const int64_t cap = (int64_t)num_sms * blocks_per_sm(per_sm, k_swizzle, 256, 0, 4);
  const int64_t blocks = units < cap ? units : cap;
  k_swizzle<<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fp8moe
