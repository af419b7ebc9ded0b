// Arguments of the grouped GEMM kernels (internal).
//
// Every mode computes C[rows, cols] = A[rows, kk] . B[cols, kk]^T with both
// operands K-major (the contracting dimension contiguous), e4m3 codes, and
// bf16 output:
//   GEMM_FWD / GEMM_DGRAD  groups split the rows; B is one [cols, kk] matrix
//                          per expert; out is [M, cols].
//   GEMM_WGRAD             groups split the contracting dimension; out is
//                          [E, rows, cols].
#pragma once
#include <stdint.h>

namespace fp8moe {

enum GemmMode { GEMM_FWD = 0, GEMM_DGRAD = 1, GEMM_WGRAD = 2 };

struct GemmArgs {
  int recipe;            // FP8MOE_ROWWISE / _MXFP8 / _TENSORWISE / _BLOCKWISE
  int mode;              // GemmMode
  const uint8_t* a;      // [rows or M, kk]
  const void* a_scale;
  const uint8_t* b;      // fwd/dgrad: [E, cols, kk]; wgrad: [cols, kk]
  const void* b_scale;
  const int32_t* offs;   // [E] cumulative exclusive ends
  int E;
  int64_t M;             // routed rows (fwd/dgrad: = rows of A; wgrad: tokens)
  int64_t rows, cols, kk;
  uint16_t* out;         // bf16
  // MXFP8 forward / dgrad with the A operand given as bf16 [M, kk] and
  // quantized in the kernel's prologue (a_scale unused); qa_out / sa_out:
  // optional copies of its codes [M, kk] and row-major e8m0 scales [M, kk/32]
  int quant_a;
  uint8_t* qa_out;
  uint8_t* sa_out;
  int* status;
  int num_sms;
  int max_smem;
};

}  // namespace fp8moe
