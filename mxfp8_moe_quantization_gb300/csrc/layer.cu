// MXFP8 MoE expert layer composites: the forward quantizes A and W in both
// directions (one read of each) and runs the grouped GEMM forward, keeping
// the dim1 operands of the backward GEMMs; the backward quantizes dY in both
// directions and runs dgrad and wgrad on the kept operands.  Host code only:
// every step is one of the library's own launches.
#include <stdint.h>

#include "../../include/fp8moe.h"

namespace {

constexpr int64_t kAlign = 256;

int64_t up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Byte offsets inside the workspace.  The kept part (A^T and W^T codes and
// scales) comes first; the forward-only operands (A, W dim0) and the
// backward-only ones (dY in both directions) share the rest.
struct Ws {
  int64_t qat, sat, qwt, swt;  // kept from forward to backward
  int64_t qa, sa, qw, sw;      // forward only
  int64_t qdy, sdy, qdyt, sdyt;  // backward only
  int64_t total;
};

Ws layout(int64_t E, int64_t M, int64_t N, int64_t K) {
  Ws w;
  int64_t o = 0;
  auto take = [&](int64_t bytes) {
    const int64_t at = o;
    o += up(bytes);
    return at;
  };
  w.qat = take(K * M);
  w.sat = take(fp8moe_swizzled_scales_bytes(1, K, M / 32, E, FP8MOE_GROUP_COLS));
  w.qwt = take(E * K * N);
  w.swt = take(fp8moe_swizzled_scales_bytes(E, K, N / 32, 0, FP8MOE_NO_GROUPS));
  const int64_t shared = o;
  w.qa = take(M * K);
  w.sa = take(fp8moe_swizzled_scales_bytes(1, M, K / 32, E, FP8MOE_GROUP_ROWS));
  w.qw = take(E * N * K);
  w.sw = take(fp8moe_swizzled_scales_bytes(E, N, K / 32, 0, FP8MOE_NO_GROUPS));
  const int64_t fwd_end = o;
  o = shared;
  w.qdy = take(M * N);
  w.sdy = take(fp8moe_swizzled_scales_bytes(1, M, N / 32, E, FP8MOE_GROUP_ROWS));
  w.qdyt = take(N * M);
  w.sdyt = take(fp8moe_swizzled_scales_bytes(1, N, M / 32, E, FP8MOE_GROUP_COLS));
  w.total = o > fwd_end ? o : fwd_end;
  return w;
}

bool sizes_ok(int64_t E, int64_t M, int64_t N, int64_t K) {
  return E >= 1 && E <= FP8MOE_MAX_GROUPS && M >= 0 && N > 0 && K > 0;
}

bool mult32(int64_t M, int64_t N, int64_t K) { return M % 32 == 0 && N % 32 == 0 && K % 32 == 0; }

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

int64_t fp8moe_mxfp8_moe_workspace_bytes(int64_t E, int64_t M, int64_t N, int64_t K) {
  if (!sizes_ok(E, M, N, K) || !mult32(M, N, K)) return -1;
  return layout(E, M, N, K).total;
}

fp8moe_status fp8moe_mxfp8_moe_fwd(const void* a, const void* w, const int32_t* offs, int64_t E, int64_t M,
                                   int64_t N, int64_t K, void* out, void* workspace, int64_t workspace_bytes,
                                   fp8moe_stream_t stream) {
  if (!sizes_ok(E, M, N, K)) return FP8MOE_ERR_INVALID_ARG;
  if (!mult32(M, N, K)) return FP8MOE_ERR_ALIGNMENT;
  if (!w || !offs || !workspace || (M > 0 && (!a || !out))) return FP8MOE_ERR_INVALID_ARG;
  const Ws L = layout(E, M, N, K);
  if (workspace_bytes < L.total) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(workspace)) return FP8MOE_ERR_ALIGNMENT;
  uint8_t* ws = (uint8_t*)workspace;
  // A: dim0 with row-grouped scales (forward operand) + dim1 with
  // column-grouped scales (kept for wgrad)
  fp8moe_status st = fp8moe_mxfp8_quantize_dual(a, 1, M, K, offs, E, ws + L.qa, ws + L.sa, FP8MOE_GROUP_ROWS,
                                                ws + L.qat, ws + L.sat, FP8MOE_GROUP_COLS, stream);
  if (st) return st;
  // W: per-expert 128x4 tiles in both directions (dim1 kept for dgrad)
  st = fp8moe_mxfp8_quantize_dual(w, E, N, K, nullptr, 0, ws + L.qw, ws + L.sw, FP8MOE_NO_GROUPS, ws + L.qwt,
                                  ws + L.swt, FP8MOE_NO_GROUPS, stream);
  if (st) return st;
  if (M == 0) return FP8MOE_OK;
  return fp8moe_scaled_grouped_mm_fwd(FP8MOE_MXFP8, ws + L.qa, ws + L.sa, ws + L.qw, ws + L.sw, offs, E, M, N, K,
                                      out, stream);
}

fp8moe_status fp8moe_mxfp8_moe_bwd(const void* dy, const int32_t* offs, int64_t E, int64_t M, int64_t N,
                                   int64_t K, void* workspace, int64_t workspace_bytes, void* da, void* dw,
                                   fp8moe_stream_t stream) {
  if (!sizes_ok(E, M, N, K)) return FP8MOE_ERR_INVALID_ARG;
  if (!mult32(M, N, K)) return FP8MOE_ERR_ALIGNMENT;
  if (!offs || !workspace || (M > 0 && !dy)) return FP8MOE_ERR_INVALID_ARG;
  const Ws L = layout(E, M, N, K);
  if (workspace_bytes < L.total) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(workspace)) return FP8MOE_ERR_ALIGNMENT;
  if (!da && !dw) return FP8MOE_OK;
  uint8_t* ws = (uint8_t*)workspace;
  // dY: dim0 (dgrad operand) and dim1 (wgrad operand), each only if used
  fp8moe_status st = fp8moe_mxfp8_quantize_dual(dy, 1, M, N, offs, E, da ? ws + L.qdy : nullptr, ws + L.sdy,
                                                FP8MOE_GROUP_ROWS, dw ? ws + L.qdyt : nullptr, ws + L.sdyt,
                                                FP8MOE_GROUP_COLS, stream);
  if (st) return st;
  if (da && M > 0) {
    st = fp8moe_scaled_grouped_mm_dgrad(FP8MOE_MXFP8, ws + L.qdy, ws + L.sdy, ws + L.qwt, ws + L.swt, offs, E, M,
                                        N, K, da, stream);
    if (st) return st;
  }
  if (dw) {
    st = fp8moe_scaled_grouped_mm_wgrad(FP8MOE_MXFP8, ws + L.qdyt, ws + L.sdyt, ws + L.qat, ws + L.sat, offs, E, M,
                                        N, K, dw, stream);
  }
  return st;
}

}  // extern "C"
