// Shared device helpers for the fp8moe kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/fp8moe.h"

#define FP8MOE_DEV __device__ __forceinline__

namespace fp8moe {

// Sticky device error word: the first error wins.
FP8MOE_DEV void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// lane-wise unsigned max of two pairs of 16-bit values, as __vmaxu2 gives it,
// in one PTX instruction (applied to bf16 bit patterns with the sign bits
// cleared it is the maximum magnitude, NaN patterns above every number)
FP8MOE_DEV uint32_t umax16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

FP8MOE_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
FP8MOE_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two e4m3fn codes, round to nearest even, saturating to
// +-448 (the hardware conversion).  Byte 0 of the result holds `lo`.
FP8MOE_DEV uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// e4m3fnuz code of an fp32 value v (|v| may exceed 240: saturates).
// fnuz (bias 8) has exactly half the value of the fn code with the same bits
// for every finite code, so enc_fnuz(v) = enc_fn'(2v), where fn' extends
// e4m3fn by the code 0x7F = 480: |2v| above the 448/480 midpoint 464 maps to
// 0x7F; the tie at 464 goes to the even code 0x7E, as the hardware
// conversion already does.  Zero is unsigned in fnuz.
FP8MOE_DEV uint32_t enc_fnuz(float v) {
  float v2 = 2.0f * v;  // exact
  uint32_t c = cvt_e4m3x2(v2, 0.0f) & 0xFFu;
  if (fabsf(v2) > 464.0f) c = 0x7Fu | (v2 < 0.0f ? 0x80u : 0u);
  if ((c & 0x7Fu) == 0u) c = 0u;
  return c;
}

template <bool FNUZ>
FP8MOE_DEV uint32_t enc2(float lo, float hi) {
  if constexpr (FNUZ) {
    return enc_fnuz(lo) | (enc_fnuz(hi) << 8);
  } else {
    return cvt_e4m3x2(lo, hi);
  }
}

// Four doubled values (2v) -> four fnuz codes packed little-endian: the
// packed fn conversion of 2v, then two byte-wise fix-ups on the word (plain
// bit arithmetic, exact per byte: no carry crosses a byte).  A byte can need
// the 0x7F (= 240) code only where the fn conversion gave +-448 (0x7E /
// 0xFE: |v| >= 216, within 10% of the fnuz maximum), so the per-value check
// runs only when such a byte is present; -0 (0x80) becomes the unsigned zero.
FP8MOE_DEV uint32_t enc4_fnuz_x2(float a, float b, float c, float d) {
  uint32_t w = cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
  const uint32_t y = (w & 0x7F7F7F7Fu) ^ 0x7E7E7E7Eu;   // a zero byte where the code is +-448
  if ((y - 0x01010101u) & ~y & 0x80808080u) {            // some byte of y is zero
    const float v2[4] = {a, b, c, d};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (fabsf(v2[i]) > 464.0f)
        w = (w & ~(0xFFu << (8 * i))) | ((0x7Fu | (v2[i] < 0.0f ? 0x80u : 0u)) << (8 * i));
  }
  // bytes equal to 0x80: t = w ^ 0x80808080 has a zero byte there; nz has
  // bit 7 set in every byte of t that is not zero
  const uint32_t t = w ^ 0x80808080u;
  const uint32_t z = ((((t & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | t) & 0x80808080u) ^ 0x80808080u;
  return w & ~(z | (z - (z >> 7)));
}

// Four fp32 -> four codes packed little-endian into a 32-bit word (fnuz:
// through the doubled values, see enc4_fnuz_x2).
template <bool FNUZ>
FP8MOE_DEV uint32_t enc4(float a, float b, float c, float d) {
  if constexpr (FNUZ) {
    return enc4_fnuz_x2(2.0f * a, 2.0f * b, 2.0f * c, 2.0f * d);
  } else {
    return enc2<false>(a, b) | (enc2<false>(c, d) << 16);
  }
}

// The multiplier that enc4_pre takes: s itself, or 2s for fnuz (whose codes
// come from the doubled values, see enc4_fnuz_x2 and enc8_bf16)
template <bool FNUZ>
FP8MOE_DEV float enc_mul(float s) {
  return FNUZ ? 2.0f * s : s;
}
// Four products x * enc_mul(s) -> four codes
template <bool FNUZ>
FP8MOE_DEV uint32_t enc4_pre(float a, float b, float c, float d) {
  if constexpr (FNUZ) {
    return enc4_fnuz_x2(a, b, c, d);
  } else {
    return enc2<false>(a, b) | (enc2<false>(c, d) << 16);
  }
}

// Encode 8 bf16 values (a uint4 of packed bf16 pairs) scaled by s.  fnuz
// multiplies by 2s instead of doubling each product: x * 2s = 2 * (x * s)
// exactly wherever the code can be non-zero (the two can differ only where
// x * s is a subnormal fp32, far below the smallest fnuz code).
template <bool FNUZ>
FP8MOE_DEV uint2 enc8_bf16(uint4 v, float s) {
  uint2 r;
  if constexpr (FNUZ) {
    const float s2 = 2.0f * s;
    r.x = enc4_fnuz_x2(__fmul_rn(bf16_lo(v.x), s2), __fmul_rn(bf16_hi(v.x), s2), __fmul_rn(bf16_lo(v.y), s2),
                       __fmul_rn(bf16_hi(v.y), s2));
    r.y = enc4_fnuz_x2(__fmul_rn(bf16_lo(v.z), s2), __fmul_rn(bf16_hi(v.z), s2), __fmul_rn(bf16_lo(v.w), s2),
                       __fmul_rn(bf16_hi(v.w), s2));
  } else {
    r.x = enc4<false>(__fmul_rn(bf16_lo(v.x), s), __fmul_rn(bf16_hi(v.x), s), __fmul_rn(bf16_lo(v.y), s),
                      __fmul_rn(bf16_hi(v.y), s));
    r.y = enc4<false>(__fmul_rn(bf16_lo(v.z), s), __fmul_rn(bf16_hi(v.z), s), __fmul_rn(bf16_lo(v.w), s),
                      __fmul_rn(bf16_hi(v.w), s));
  }
  return r;
}

// max |x| over 8 bf16 values: works on the bit patterns (|x| is the pattern
// with the sign bit cleared, and for non-negative IEEE values integer order
// is value order), exact.
FP8MOE_DEV uint32_t absmax8_bits(uint4 v) {
  uint32_t m = 0;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = max(m, w[i] & 0x7FFFu);
    m = max(m, (w[i] >> 16) & 0x7FFFu);
  }
  return m;  // a bf16 bit pattern without sign
}

FP8MOE_DEV float bf16bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// 16-byte read-only load that does not allocate in L1 (streamed inputs).
FP8MOE_DEV uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// (m, m) in one 64-bit register pair: the second operand of fmul2_rn
FP8MOE_DEV uint64_t pair_f32(float m) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(m));
  return r;
}

// x = a * m, y = b * m with (m, m) = m2: the packed fp32 multiply of sm_100
// and later (two IEEE products, round to nearest even, subnormals kept:
// bit-identical to two __fmul_rn)
FP8MOE_DEV void fmul2_rn(float a, float b, uint64_t m2, float& x, float& y) {
  asm("{\n .reg .b64 p, r;\n mov.b64 p, {%2, %3};\n mul.rn.f32x2 r, p, %4;\n mov.b64 {%0, %1}, r;\n}"
      : "=f"(x), "=f"(y)
      : "f"(a), "f"(b), "l"(m2));
}

// The codes of an 8-row x 8-column bf16 block scaled per column, column by
// column: v[k] holds row k (columns 0..7 as bf16 pairs), m2[c] the pair
// (enc_mul(s_c), enc_mul(s_c)), and col[c] receives column c's eight codes
// with row k in byte k.  Each product pair and each packed conversion takes
// one column from neighbouring rows, so the codes come out already in
// column order: no byte transposes.
template <bool FNUZ>
FP8MOE_DEV void cast8x8_cols(const uint4 (&v)[8], const uint64_t (&m2)[8], uint2 (&col)[8]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = w == 0 ? v[k].x : w == 1 ? v[k].y : w == 2 ? v[k].z : v[k].w;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float p[8];
#pragma unroll
      for (int k = 0; k < 8; k += 2)
        fmul2_rn(h ? bf16_hi(x[k]) : bf16_lo(x[k]), h ? bf16_hi(x[k + 1]) : bf16_lo(x[k + 1]), m2[2 * w + h], p[k],
                 p[k + 1]);
      col[2 * w + h] = make_uint2(enc4_pre<FNUZ>(p[0], p[1], p[2], p[3]), enc4_pre<FNUZ>(p[4], p[5], p[6], p[7]));
    }
  }
}

// Column t (0..3) of four row words (byte t of each) as one word, rows in
// byte order: a 4x4 byte transpose.
FP8MOE_DEV void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3, uint32_t (&col)[4]) {
  const uint32_t a01 = __byte_perm(r0, r1, 0x5140);  // c0 r0, c0 r1, c1 r0, c1 r1
  const uint32_t a23 = __byte_perm(r2, r3, 0x5140);
  const uint32_t b01 = __byte_perm(r0, r1, 0x7362);  // c2 r0, c2 r1, c3 r0, c3 r1
  const uint32_t b23 = __byte_perm(r2, r3, 0x7362);
  col[0] = __byte_perm(a01, a23, 0x5410);
  col[1] = __byte_perm(a01, a23, 0x7632);
  col[2] = __byte_perm(b01, b23, 0x5410);
  col[3] = __byte_perm(b01, b23, 0x7632);
}

// Rowwise / colwise scale from an absolute maximum (all IEEE fp32, RN).
template <bool FNUZ>
FP8MOE_DEV void rowwise_scale(float amax, float& s, float& inv) {
  const float fmax = FNUZ ? 240.0f : 448.0f;
  s = __fdiv_rn(fmax, fmaxf(amax, 1e-12f));
  inv = __fdiv_rn(1.0f, s);
}

// e8m0 block exponent from the bf16 bit pattern (sign cleared) of the block
// absolute maximum: e = clamp(floor(log2(amax)) - 8, -127, 127).
// floor(log2) of a normal bf16 is its exponent field - 127; a subnormal
// (exponent field 0, 7-bit mantissa m) has floor(log2) = msb(m) - 133.
FP8MOE_DEV int e8m0_exponent(uint32_t amax_bits) {
  if (amax_bits == 0) return -127;
  int ef = (int)(amax_bits >> 7);
  int E;
  if (ef != 0) {
    E = ef - 127;
  } else {
    E = (31 - __clz((int)(amax_bits & 0x7F))) - 133;
  }
  int e = E - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as an fp32 (e in [-127, 127]): built from the exponent field; for
// e = 127 (2^-127) the value is a subnormal.
FP8MOE_DEV float exp2_neg(int e) {
  int be = 127 - e;  // biased exponent of 2^-e
  if (be >= 1) return __uint_as_float((uint32_t)be << 23);
  return __uint_as_float(1u << (22 + be));  // subnormal: 2^(be-127) = 2^-149 * 2^(be+22)
}

}  // namespace fp8moe
