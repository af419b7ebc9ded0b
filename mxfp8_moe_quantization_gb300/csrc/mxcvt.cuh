// Exact MXFP8 block arithmetic on packed bf16 pairs, shared by the
// quantizers and the grouped GEMM's fused A-quantization prologue
// ("Accelerating Llama4 Scout training with TorchAO MXFP8 MoE primitives",
// MXFP8 layout diagram: 1x32 blocks of e4m3 with one e8m0 scale each; the
// scale exponent is floor(log2(amax)) - 8, clamped to [-127, 127]).
#pragma once
#include <stdint.h>

#include "common.cuh"

namespace fp8moe {

// lane-wise max of two pairs of non-negative bf16 values (sign bits cleared):
// the result is one of the inputs, so the maximum is exact.  Only an all-zero
// or all-subnormal block could see a subnormal flushed, and its scale byte is
// 0 either way (its exponent field is 0).
FP8MOE_DEV uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// lane-wise max of the magnitudes of two bf16 pairs, in one instruction:
// each half of the result has magnitude max(|a|, |b|) (NaN ignored unless
// both are NaN, as in max_u16x2) and a sign bit that is the XOR of the
// inputs' signs, which callers must not use (the exponent field, bits 7-14
// of a half, is exact).
FP8MOE_DEV uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// The e8m0 byte of a block, clamp(floor(log2 amax) - 8, -127, 127) + 127, is
// max(ef, 8) - 8 for the bf16 exponent field ef of the block maximum (a zero
// or subnormal maximum has ef = 0 and gets byte 0, as the clamp gives); 2^-e
// is then the bf16 with exponent field 262 - max(ef, 8), a normal number.
// x * 2^-e on two bf16 values: exact (an 8-bit significand times a power of
// two, below 2^9 in magnitude; only values far under the e4m3 range can
// round, and they encode to a signed zero either way)
FP8MOE_DEV uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// four fp32 values -> four e4m3fn codes (RNE, saturating), byte i from the
// i-th argument, packed in one word
FP8MOE_DEV uint32_t cvt4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n .reg .b16 l, h;\n cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n"
      " mov.b32 %0, {l, h};\n}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}
FP8MOE_DEV float lo_f32(uint32_t y) { return __uint_as_float(y << 16); }
FP8MOE_DEV float hi_f32(uint32_t y) { return __uint_as_float(y & 0xFFFF0000u); }
// 8 codes of one row chunk (4 bf16 pairs) scaled by the pair p2
FP8MOE_DEV uint2 enc_row8(const uint4& v, uint32_t p2) {
  const uint32_t y0 = mul_bf16x2(v.x, p2), y1 = mul_bf16x2(v.y, p2);
  const uint32_t y2 = mul_bf16x2(v.z, p2), y3 = mul_bf16x2(v.w, p2);
  return make_uint2(cvt4(lo_f32(y0), hi_f32(y0), lo_f32(y1), hi_f32(y1)),
                    cvt4(lo_f32(y2), hi_f32(y2), lo_f32(y3), hi_f32(y3)));
}

// e8m0 byte of a block and the packed bf16 pair 2^-e by which its values are
// scaled, from the exponent field ef of the block's absolute maximum (see
// mul_bf16x2): byte = max(ef, 8) - 8, 2^-e = bf16 with exponent field
// 262 - max(ef, 8).
FP8MOE_DEV uint32_t mx_block_scale(uint32_t amax_bits, uint32_t& p2) {
  const uint32_t ef = max((amax_bits >> 7) & 0xFFu, 8u);
  p2 = ((262u - ef) << 7) | ((262u - ef) << 23);
  return ef - 8u;
}

}  // namespace fp8moe
