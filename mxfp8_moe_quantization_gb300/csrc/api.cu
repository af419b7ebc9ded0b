// C-ABI entry points of libfp8moe: argument checks on the host, then launches
// on the caller's stream.  See include/fp8moe.h for the contract of each call.
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "launch.h"

// Sticky device status word (static device memory: the library allocates
// nothing).  Kernels receive its address; fp8moe_get_device_status takes it
// (reads and clears it in one atomic exchange) into the take slot.
static __device__ int g_fp8moe_status;
static __device__ int g_fp8moe_status_take;

static __global__ void k_take_status(int* status, int* take) { *take = atomicExch(status, 0); }

namespace {

struct DevInfo {
  bool init = false;
  int* status = nullptr;
  int* take = nullptr;
  int num_sms = 0;
  int max_smem = 0;
};

constexpr int kMaxDevices = 128;
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;
std::mutex g_take_mu;

fp8moe_status device_info(DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaGetSymbolAddress((void**)&d.status, g_fp8moe_status) != cudaSuccess) return FP8MOE_ERR_CUDA;
    if (cudaGetSymbolAddress((void**)&d.take, g_fp8moe_status_take) != cudaSuccess) return FP8MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FP8MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return FP8MOE_ERR_CUDA;
    d.init = true;
  }
  *out = &d;
  return FP8MOE_OK;
}

inline bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline fp8moe_status cuda_result(cudaError_t e) { return e == cudaSuccess ? FP8MOE_OK : FP8MOE_ERR_CUDA; }

inline bool valid_kind(int kind) { return kind == FP8MOE_E4M3FN || kind == FP8MOE_E4M3FNUZ; }

}  // namespace

extern "C" {

const char* fp8moe_status_string(int s) {
  switch (s) {
    case FP8MOE_OK: return "ok";
    case FP8MOE_ERR_INVALID_ARG: return "invalid argument";
    case FP8MOE_ERR_ALIGNMENT: return "misaligned pointer or size";
    case FP8MOE_ERR_UNSUPPORTED: return "unsupported combination";
    case FP8MOE_ERR_CUDA: return "CUDA error";
    case FP8MOE_ERR_DEVICE_OFFSETS: return "invalid routing offsets (device)";
    case FP8MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case FP8MOE_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the library's static array holds";
    case FP8MOE_ERR_CONCURRENT: return "launches in flight at once shared a device work counter";
    default: return "unknown status";
  }
}

int fp8moe_version(void) { return (1 << 16) | 0; }

int64_t fp8moe_jagged_t_cols(int64_t M, int64_t E) { return (M + 31 * E + 15) / 16 * 16; }

fp8moe_status fp8moe_quantize_rowwise(const void* x, int64_t R, int64_t C, int64_t ldx, int kind, void* q,
                                      float* scale_inv, fp8moe_stream_t stream) {
  if (R < 0 || C < 0 || ldx < C || !valid_kind(kind)) return FP8MOE_ERR_INVALID_ARG;
  if (R == 0 || C == 0) return FP8MOE_OK;
  if (!x || !q || !scale_inv) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(q) || C % 16 || ldx % 8 || ((uintptr_t)scale_inv & 3)) return FP8MOE_ERR_ALIGNMENT;
  if (C > (int64_t)1 << 30) return FP8MOE_ERR_INVALID_ARG;
  return cuda_result(fp8moe::launch_quant_rowwise(x, R, C, ldx, kind, q, scale_inv, (cudaStream_t)stream));
}

fp8moe_status fp8moe_quantize_colwise_3d(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                                         int transpose_out, int kind, void* q, float* scale_inv,
                                         fp8moe_stream_t stream) {
  if (E < 0 || R < 0 || C < 0 || !valid_kind(kind)) return FP8MOE_ERR_INVALID_ARG;
  if (offs && E == 0) return FP8MOE_ERR_INVALID_ARG;
  if (offs && E > FP8MOE_MAX_GROUPS) return FP8MOE_ERR_INVALID_ARG;
  if (E == 0 || C == 0) return FP8MOE_OK;
  if (!x || !q || !scale_inv) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(q) || C % 16 || ((uintptr_t)scale_inv & 3)) return FP8MOE_ERR_ALIGNMENT;
  if (!offs && transpose_out && R % 16) return FP8MOE_ERR_ALIGNMENT;
  if (offs && ((uintptr_t)offs & 3)) return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  const int64_t ldt = offs ? fp8moe_jagged_t_cols(R, E) : 0;
  return cuda_result(fp8moe::launch_colwise(x, E, R, C, offs, transpose_out, kind, ldt, q, scale_inv, d->status,
                                            d->num_sms, (cudaStream_t)stream));
}

fp8moe_status fp8moe_mxfp8_quantize_dim0(const void* x, int64_t B, int64_t R, int64_t C, void* q, uint8_t* scale,
                                         fp8moe_stream_t stream) {
  if (B < 0 || R < 0 || C < 0) return FP8MOE_ERR_INVALID_ARG;
  if (C % 32) return FP8MOE_ERR_ALIGNMENT;
  if (B == 0 || R == 0 || C == 0) return FP8MOE_OK;
  if (!x || !q || !scale) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(q)) return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  return cuda_result(fp8moe::launch_mx_dim0(x, B, R, C, q, scale, FP8MOE_SCALES_ROWMAJOR, nullptr, 0, d->num_sms,
                                            d->status, (cudaStream_t)stream));
}

fp8moe_status fp8moe_mxfp8_quantize_dim1(const void* x, int64_t B, int64_t R, int64_t C, void* qt,
                                         uint8_t* scale, fp8moe_stream_t stream) {
  if (B < 0 || R < 0 || C < 0) return FP8MOE_ERR_INVALID_ARG;
  if (R % 32 || C % 16) return FP8MOE_ERR_ALIGNMENT;
  if (B == 0 || R == 0 || C == 0) return FP8MOE_OK;
  if (!x || !qt || !scale) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(qt)) return FP8MOE_ERR_ALIGNMENT;
  if (C > ((int64_t)1 << 31) || R > ((int64_t)1 << 31) || B > 65535) return FP8MOE_ERR_INVALID_ARG;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  return cuda_result(fp8moe::launch_mx_dual(x, B, R, C, nullptr, nullptr, FP8MOE_SCALES_ROWMAJOR, qt, scale,
                                            FP8MOE_SCALES_ROWMAJOR, nullptr, 0, d->num_sms, d->status,
                                            (cudaStream_t)stream));
}

fp8moe_status fp8moe_mxfp8_quantize_dual(const void* x, int64_t B, int64_t R, int64_t C, const int32_t* offs,
                                         int64_t E, void* q0, uint8_t* s0, int s0_layout, void* q1, uint8_t* s1,
                                         int s1_layout, fp8moe_stream_t stream) {
  if (B < 0 || R < 0 || C < 0 || E < 0) return FP8MOE_ERR_INVALID_ARG;
  if (!q0 && !q1) return FP8MOE_ERR_INVALID_ARG;
  if (C % 32 || (q1 && R % 32)) return FP8MOE_ERR_ALIGNMENT;
  if ((q0 && !s0) || (q1 && !s1)) return FP8MOE_ERR_INVALID_ARG;
  const bool ok0 = !q0 || s0_layout == FP8MOE_SCALES_ROWMAJOR || s0_layout == FP8MOE_NO_GROUPS ||
                   s0_layout == FP8MOE_GROUP_ROWS;
  const bool ok1 = !q1 || s1_layout == FP8MOE_SCALES_ROWMAJOR || s1_layout == FP8MOE_NO_GROUPS ||
                   s1_layout == FP8MOE_GROUP_COLS;
  if (!ok0 || !ok1) return FP8MOE_ERR_INVALID_ARG;
  const bool grouped = (q0 && s0_layout == FP8MOE_GROUP_ROWS) || (q1 && s1_layout == FP8MOE_GROUP_COLS);
  if (grouped && (B != 1 || E < 1 || E > 1024 || !offs)) return FP8MOE_ERR_INVALID_ARG;
  if (grouped && ((uintptr_t)offs & 3)) return FP8MOE_ERR_ALIGNMENT;
  if (B == 0 || R == 0 || C == 0) return FP8MOE_OK;
  if (!x || !al16(x) || (q0 && !al16(q0)) || (q1 && !al16(q1))) return x ? FP8MOE_ERR_ALIGNMENT : FP8MOE_ERR_INVALID_ARG;
  if (B > 65535 || R > ((int64_t)1 << 31) || C > ((int64_t)1 << 31)) return FP8MOE_ERR_INVALID_ARG;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  // both directions: one fused launch reading x once (4 bytes moved per
  // element instead of 6); dim1 alone: the same kernel without dim0; dim0
  // alone: its own kernel.  Scales go straight to their final layout.
  const int64_t Eg = grouped ? E : 0;
  cudaError_t e = cudaSuccess;
  if (q1) {
    e = fp8moe::launch_mx_dual(x, B, R, C, q0, s0, q0 ? s0_layout : FP8MOE_SCALES_ROWMAJOR, q1, s1, s1_layout, offs,
                               Eg, d->num_sms, d->status, (cudaStream_t)stream);
  } else {
    e = fp8moe::launch_mx_dim0(x, B, R, C, q0, s0, s0_layout, offs, Eg, d->num_sms, d->status,
                               (cudaStream_t)stream);
  }
  return e == cudaSuccess ? FP8MOE_OK : FP8MOE_ERR_CUDA;
}

int64_t fp8moe_swizzled_scales_bytes(int64_t B, int64_t R, int64_t Cs, int64_t E, int group_axis) {
  if (B < 0 || R < 0 || Cs < 0 || E < 0) return -1;
  if (group_axis != FP8MOE_NO_GROUPS && group_axis != FP8MOE_GROUP_ROWS && group_axis != FP8MOE_GROUP_COLS)
    return -1;
  const fp8moe::SwizzleGeom g = fp8moe::swizzle_geom(R, Cs, group_axis == FP8MOE_NO_GROUPS ? 0 : E, group_axis);
  return B * g.Rp * g.Cp;
}

fp8moe_status fp8moe_swizzle_scales_128x4(const uint8_t* s, int64_t B, int64_t R, int64_t Cs, const int32_t* offs,
                                          int64_t E, int group_axis, uint8_t* out, fp8moe_stream_t stream) {
  if (B < 0 || R < 0 || Cs < 0 || E < 0) return FP8MOE_ERR_INVALID_ARG;
  if (group_axis != FP8MOE_NO_GROUPS && group_axis != FP8MOE_GROUP_ROWS && group_axis != FP8MOE_GROUP_COLS)
    return FP8MOE_ERR_INVALID_ARG;
  if (group_axis != FP8MOE_NO_GROUPS) {
    if (B != 1 || E < 1 || E > 1024 || !offs) return FP8MOE_ERR_INVALID_ARG;
    if ((uintptr_t)offs & 3) return FP8MOE_ERR_ALIGNMENT;
  }
  if (fp8moe_swizzled_scales_bytes(B, R, Cs, E, group_axis) == 0) return FP8MOE_OK;
  if (!out || (!s && R * Cs > 0)) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(out)) return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  return cuda_result(fp8moe::launch_swizzle(s, B, R, Cs, offs, E, group_axis, out, d->status, d->num_sms,
                                            (cudaStream_t)stream));
}

fp8moe_status fp8moe_quantize_tensorwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                                         int transpose_out, int kind, void* q, float* scale_inv,
                                         fp8moe_stream_t stream) {
  if (E < 0 || R < 0 || C < 0 || !valid_kind(kind)) return FP8MOE_ERR_INVALID_ARG;
  if (offs && E == 0) return FP8MOE_ERR_INVALID_ARG;
  if (offs && transpose_out && E > FP8MOE_MAX_GROUPS) return FP8MOE_ERR_INVALID_ARG;
  if (!scale_inv) return FP8MOE_ERR_INVALID_ARG;
  if ((uintptr_t)scale_inv & 3) return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  if (E == 0 || C == 0 || (R == 0 && !(offs && transpose_out))) {
    // nothing to cast (the jagged transposed layout still gets its zero
    // padding below); the scale is that of an all-zero tensor
    return cuda_result(fp8moe::launch_tensorwise(nullptr, 0, 0, 0, nullptr, 0, kind, nullptr, scale_inv,
                                                 d->num_sms, d->status, (cudaStream_t)stream));
  }
  if (!q || (!x && R > 0)) return FP8MOE_ERR_INVALID_ARG;
  if ((x && !al16(x)) || !al16(q)) return FP8MOE_ERR_ALIGNMENT;
  if (transpose_out && (C % 16 || (!offs && R % 16))) return FP8MOE_ERR_ALIGNMENT;
  if (offs && ((uintptr_t)offs & 3)) return FP8MOE_ERR_ALIGNMENT;
  return cuda_result(fp8moe::launch_tensorwise(x, E, R, C, offs, transpose_out, kind, q, scale_inv, d->num_sms,
                                               d->status, (cudaStream_t)stream));
}

fp8moe_status fp8moe_quantize_blockwise_rows(const void* x, int64_t R, int64_t C, int kind, void* q,
                                             float* scale_inv, fp8moe_stream_t stream) {
  if (R < 0 || C < 0 || !valid_kind(kind)) return FP8MOE_ERR_INVALID_ARG;
  if (C % 128) return FP8MOE_ERR_ALIGNMENT;
  if (R == 0 || C == 0) return FP8MOE_OK;
  if (!x || !q || !scale_inv) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(q) || ((uintptr_t)scale_inv & 3)) return FP8MOE_ERR_ALIGNMENT;
  if (R > ((int64_t)1 << 35)) return FP8MOE_ERR_INVALID_ARG;
  return cuda_result(fp8moe::launch_bw_rows(x, R, C, kind, q, scale_inv, (cudaStream_t)stream));
}

fp8moe_status fp8moe_quantize_blockwise_weight(const void* w, int64_t E, int64_t N, int64_t K, int kind, void* q,
                                               void* qt, float* scale_inv, fp8moe_stream_t stream) {
  if (E < 0 || N < 0 || K < 0 || !valid_kind(kind) || (!q && !qt)) return FP8MOE_ERR_INVALID_ARG;
  if (N % 128 || K % 128) return FP8MOE_ERR_ALIGNMENT;
  if (E == 0 || N == 0 || K == 0) return FP8MOE_OK;
  if (!w || !scale_inv) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(w) || (q && !al16(q)) || (qt && !al16(qt)) || ((uintptr_t)scale_inv & 3)) return FP8MOE_ERR_ALIGNMENT;
  if (E * (N / 128) * (K / 128) >= ((int64_t)1 << 31)) return FP8MOE_ERR_INVALID_ARG;
  return cuda_result(fp8moe::launch_bw_weight(w, E, N, K, kind, q, qt, scale_inv, (cudaStream_t)stream));
}

int64_t fp8moe_blockwise_token_blocks(int64_t M, int64_t E) {
  if (M < 0 || E < 1) return -1;
  return (M + 127) / 128 + E;
}

fp8moe_status fp8moe_quantize_blockwise_tokens(const void* x, int64_t M, int64_t C, const int32_t* offs, int64_t E,
                                               int kind, void* qt, float* scale_inv, fp8moe_stream_t stream) {
  if (M < 0 || C < 0 || E < 1 || E > FP8MOE_MAX_GROUPS || !valid_kind(kind) || !offs) return FP8MOE_ERR_INVALID_ARG;
  if (M % 32 || C % 16) return FP8MOE_ERR_ALIGNMENT;
  if (((uintptr_t)offs & 3)) return FP8MOE_ERR_ALIGNMENT;
  if (M == 0 || C == 0) return FP8MOE_OK;
  if (!x || !qt || !scale_inv) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(qt) || !al16(scale_inv)) return FP8MOE_ERR_ALIGNMENT;
  if (fp8moe_blockwise_token_blocks(M, E) * ((C + 127) / 128) >= ((int64_t)1 << 31)) return FP8MOE_ERR_INVALID_ARG;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  return cuda_result(fp8moe::launch_bw_tokens(x, M, C, offs, E, kind, qt, scale_inv, d->num_sms, d->status,
                                              (cudaStream_t)stream));
}

static fp8moe_status grouped_mm(int mode, int recipe, const void* a, const void* a_scale, const void* b,
                                const void* b_scale, const int32_t* offs, int64_t E, int64_t M, int64_t N,
                                int64_t K, void* out, fp8moe_stream_t stream) {
  if (recipe != FP8MOE_ROWWISE && recipe != FP8MOE_MXFP8 && recipe != FP8MOE_TENSORWISE &&
      recipe != FP8MOE_BLOCKWISE)
    return FP8MOE_ERR_INVALID_ARG;
  if (E < 1 || M < 0 || N < 0 || K < 0 || E > 4096) return FP8MOE_ERR_INVALID_ARG;
  if (!offs || ((uintptr_t)offs & 3)) return FP8MOE_ERR_INVALID_ARG;
  if (N % 16 || K % 16) return FP8MOE_ERR_ALIGNMENT;
  if (recipe == FP8MOE_MXFP8) {
    // the contracting dimension must hold whole 32-element scale blocks
    if (mode == fp8moe::GEMM_FWD && K % 32) return FP8MOE_ERR_ALIGNMENT;
    if (mode == fp8moe::GEMM_DGRAD && N % 32) return FP8MOE_ERR_ALIGNMENT;
    if (mode == fp8moe::GEMM_WGRAD && M % 32) return FP8MOE_ERR_ALIGNMENT;
  }
  if (recipe == FP8MOE_BLOCKWISE) {
    // weight tiles are 128 x 128; wgrad's token tiles are cut at 32-multiple
    // group boundaries
    if (N % 128 || K % 128 || (mode == fp8moe::GEMM_WGRAD && M % 32)) return FP8MOE_ERR_ALIGNMENT;
  }
  if (!a || !b || !out || !a_scale || !b_scale) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(a) || !al16(b) || !al16(out)) return FP8MOE_ERR_ALIGNMENT;
  if (recipe == FP8MOE_TENSORWISE || (recipe == FP8MOE_BLOCKWISE && mode != fp8moe::GEMM_WGRAD)
          ? (((uintptr_t)a_scale | (uintptr_t)b_scale) & 3)
          : (!al16(a_scale) || !al16(b_scale)))
    return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  fp8moe::GemmArgs g{};
  g.recipe = recipe;
  g.mode = mode;
  g.E = (int)E;
  g.offs = offs;
  g.out = (uint16_t*)out;
  g.status = d->status;
  g.num_sms = d->num_sms;
  g.max_smem = d->max_smem;
  g.M = M;
  g.a = (const uint8_t*)a;
  g.b = (const uint8_t*)b;
  g.a_scale = a_scale;
  g.b_scale = b_scale;
  if (mode == fp8moe::GEMM_FWD) {          // [M,K] x [E,N,K] -> [M,N]
    g.rows = M, g.cols = N, g.kk = K;
  } else if (mode == fp8moe::GEMM_DGRAD) { // [M,N] x [E,K,N] -> [M,K]
    g.rows = M, g.cols = K, g.kk = N;
  } else {                                 // [N,Mt] x [K,Mt] -> [E,N,K]
    g.rows = N, g.cols = K;
    g.kk = recipe == FP8MOE_MXFP8 || recipe == FP8MOE_BLOCKWISE ? M : fp8moe_jagged_t_cols(M, E);
  }
  if (g.rows == 0 || g.cols == 0) return FP8MOE_OK;
  if (g.kk == 0) {
    // nothing to contract (e.g. wgrad of a batch without routed tokens):
    // every output element is an empty sum
    const int64_t n = (mode == fp8moe::GEMM_WGRAD ? E : 1) * g.rows * g.cols;
    return cuda_result(cudaMemsetAsync(out, 0, (size_t)n * 2, (cudaStream_t)stream));
  }
  cudaError_t e = recipe == FP8MOE_BLOCKWISE ? fp8moe::launch_blockwise_mm(g, (cudaStream_t)stream)
                                             : fp8moe::launch_grouped_mm(g, (cudaStream_t)stream);
  if (e == cudaErrorNotSupported) return FP8MOE_ERR_UNSUPPORTED;
  return cuda_result(e);
}

fp8moe_status fp8moe_scaled_grouped_mm_fwd(int recipe, const void* a, const void* a_scale, const void* w,
                                           const void* w_scale, const int32_t* offs, int64_t E, int64_t M,
                                           int64_t N, int64_t K, void* out, fp8moe_stream_t stream) {
  return grouped_mm(fp8moe::GEMM_FWD, recipe, a, a_scale, w, w_scale, offs, E, M, N, K, out, stream);
}

fp8moe_status fp8moe_scaled_grouped_mm_dgrad(int recipe, const void* dy, const void* dy_scale, const void* wt,
                                             const void* wt_scale, const int32_t* offs, int64_t E, int64_t M,
                                             int64_t N, int64_t K, void* out, fp8moe_stream_t stream) {
  return grouped_mm(fp8moe::GEMM_DGRAD, recipe, dy, dy_scale, wt, wt_scale, offs, E, M, N, K, out, stream);
}

fp8moe_status fp8moe_scaled_grouped_mm_wgrad(int recipe, const void* dyt, const void* dyt_scale, const void* at,
                                             const void* at_scale, const int32_t* offs, int64_t E, int64_t M,
                                             int64_t N, int64_t K, void* out, fp8moe_stream_t stream) {
  return grouped_mm(fp8moe::GEMM_WGRAD, recipe, dyt, dyt_scale, at, at_scale, offs, E, M, N, K, out, stream);
}

static fp8moe_status grouped_mm_quant_a(int mode, const void* a_bf16, const void* b, const void* b_scale,
                                        const int32_t* offs, int64_t E, int64_t M, int64_t N, int64_t K, void* out,
                                        void* a_q, uint8_t* a_s, fp8moe_stream_t stream) {
  if (E < 1 || E > FP8MOE_MAX_GROUPS || M < 0 || N < 0 || K < 0) return FP8MOE_ERR_INVALID_ARG;
  if (!offs || ((uintptr_t)offs & 3)) return FP8MOE_ERR_INVALID_ARG;
  if ((a_q == nullptr) != (a_s == nullptr)) return FP8MOE_ERR_INVALID_ARG;
  const int64_t kk = mode == fp8moe::GEMM_FWD ? K : N;      // the contracting dimension
  const int64_t cols = mode == fp8moe::GEMM_FWD ? N : K;
  if (N % 16 || K % 16 || kk % 32) return FP8MOE_ERR_ALIGNMENT;
  if (!a_bf16 || !b || !b_scale || !out) return FP8MOE_ERR_INVALID_ARG;
  if (!al16(a_bf16) || !al16(b) || !al16(b_scale) || !al16(out) || (a_q && !al16(a_q))) return FP8MOE_ERR_ALIGNMENT;
  if (M == 0 || cols == 0) return FP8MOE_OK;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  fp8moe::GemmArgs g{};
  g.recipe = FP8MOE_MXFP8;
  g.mode = mode;
  g.E = (int)E;
  g.offs = offs;
  g.out = (uint16_t*)out;
  g.status = d->status;
  g.num_sms = d->num_sms;
  g.max_smem = d->max_smem;
  g.M = M;
  g.a = (const uint8_t*)a_bf16;
  g.b = (const uint8_t*)b;
  g.a_scale = nullptr;
  g.b_scale = b_scale;
  g.rows = M, g.cols = cols, g.kk = kk;
  g.quant_a = 1;
  g.qa_out = (uint8_t*)a_q;
  g.sa_out = a_s;
  cudaError_t e = fp8moe::launch_grouped_mm(g, (cudaStream_t)stream);
  if (e == cudaErrorNotSupported) return FP8MOE_ERR_UNSUPPORTED;
  return cuda_result(e);
}

fp8moe_status fp8moe_mxfp8_grouped_mm_fwd_quant_a(const void* a, const void* w, const void* w_scale,
                                                  const int32_t* offs, int64_t E, int64_t M, int64_t N, int64_t K,
                                                  void* out, void* a_q, uint8_t* a_s, fp8moe_stream_t stream) {
  return grouped_mm_quant_a(fp8moe::GEMM_FWD, a, w, w_scale, offs, E, M, N, K, out, a_q, a_s, stream);
}

fp8moe_status fp8moe_mxfp8_grouped_mm_dgrad_quant_a(const void* dy, const void* wt, const void* wt_scale,
                                                    const int32_t* offs, int64_t E, int64_t M, int64_t N, int64_t K,
                                                    void* out, void* dy_q, uint8_t* dy_s, fp8moe_stream_t stream) {
  return grouped_mm_quant_a(fp8moe::GEMM_DGRAD, dy, wt, wt_scale, offs, E, M, N, K, out, dy_q, dy_s, stream);
}

int64_t fp8moe_route_rows(int64_t T, int64_t k, int64_t E) {
  if (T < 0 || k < 1 || E < 1) return -1;
  return (T * k + 31 * E + 31) / 32 * 32;
}

int64_t fp8moe_route_workspace_bytes(int64_t T, int64_t k, int64_t E) {
  if (T < 0 || k < 1 || E < 1) return -1;
  return fp8moe::route_workspace_bytes(T, k, E);
}

fp8moe_status fp8moe_route_permute(const void* x, int64_t T, int64_t H, const int32_t* topk_idx,
                                   const float* topk_w, int64_t k, int64_t E, void* a, int32_t* offs,
                                   int32_t* row_of, void* workspace, int64_t workspace_bytes,
                                   fp8moe_stream_t stream) {
  if (T < 0 || H < 0 || k < 1 || E < 1 || E > 1024) return FP8MOE_ERR_INVALID_ARG;
  if (T * k > ((int64_t)1 << 30)) return FP8MOE_ERR_INVALID_ARG;
  if (!a || !offs || !workspace || (T > 0 && (!x || !topk_idx || !row_of))) return FP8MOE_ERR_INVALID_ARG;
  if (workspace_bytes < fp8moe::route_workspace_bytes(T, k, E)) return FP8MOE_ERR_INVALID_ARG;
  if (H % 8 || (x && !al16(x)) || !al16(a)) return FP8MOE_ERR_ALIGNMENT;
  if (((uintptr_t)topk_idx | (uintptr_t)offs | (uintptr_t)row_of | (uintptr_t)topk_w | (uintptr_t)workspace) & 3)
    return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  return cuda_result(fp8moe::launch_route_permute(x, T, H, topk_idx, topk_w, k, E, fp8moe_route_rows(T, k, E), a,
                                                  offs, row_of, workspace, d->num_sms, d->status,
                                                  (cudaStream_t)stream));
}

fp8moe_status fp8moe_route_permute_noalloc(const void* x, int64_t T, int64_t H, const int32_t* topk_idx,
                                           const float* topk_w, int64_t k, int64_t E, void* a, int32_t* offs,
                                           int32_t* row_of, fp8moe_stream_t stream) {
  if (T < 0 || H < 0 || k < 1 || E < 1 || E > 1024) return FP8MOE_ERR_INVALID_ARG;
  if (T * k > ((int64_t)1 << 30)) return FP8MOE_ERR_INVALID_ARG;
  // the scratch this problem needs must fit the library's static array
  if (fp8moe::route_workspace_bytes(T, k, E) > fp8moe::route_static_scratch_bytes()) return FP8MOE_ERR_SCRATCH_LIMIT;
  if (!a || !offs || (T > 0 && (!x || !topk_idx || !row_of))) return FP8MOE_ERR_INVALID_ARG;
  if (H % 8 || (x && !al16(x)) || !al16(a)) return FP8MOE_ERR_ALIGNMENT;
  if (((uintptr_t)topk_idx | (uintptr_t)offs | (uintptr_t)row_of | (uintptr_t)topk_w) & 3)
    return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  void* scratch = nullptr;
  if (fp8moe::route_static_scratch(&scratch) != cudaSuccess) return FP8MOE_ERR_CUDA;
  return cuda_result(fp8moe::launch_route_permute(x, T, H, topk_idx, topk_w, k, E, fp8moe_route_rows(T, k, E), a,
                                                  offs, row_of, scratch, d->num_sms, d->status,
                                                  (cudaStream_t)stream));
}

fp8moe_status fp8moe_route_unpermute(const void* y, int64_t T, int64_t N, const int32_t* row_of,
                                     const float* topk_w, int64_t k, void* out, fp8moe_stream_t stream) {
  if (T < 0 || N < 0 || k < 1) return FP8MOE_ERR_INVALID_ARG;
  if (T == 0 || N == 0) return FP8MOE_OK;
  if (!y || !row_of || !out) return FP8MOE_ERR_INVALID_ARG;
  if (N % 8 || !al16(y) || !al16(out) || (((uintptr_t)row_of | (uintptr_t)topk_w) & 3)) return FP8MOE_ERR_ALIGNMENT;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  return cuda_result(fp8moe::launch_route_unpermute(y, N, row_of, topk_w, T, k, out, (cudaStream_t)stream));
}

fp8moe_status fp8moe_get_device_status(fp8moe_stream_t stream, int32_t* out_code) {
  if (!out_code) return FP8MOE_ERR_INVALID_ARG;
  DevInfo* d;
  fp8moe_status st = device_info(&d);
  if (st) return st;
  // The read and the clear are one atomic exchange on the device, ordered
  // after the stream's work: a status that a kernel on another stream sets
  // meanwhile is either taken here or stays for the next call.  The mutex
  // keeps concurrent callers from sharing the take slot.
  std::lock_guard<std::mutex> lk(g_take_mu);
  k_take_status<<<1, 1, 0, (cudaStream_t)stream>>>(d->status, d->take);
  if (cudaGetLastError() != cudaSuccess) return FP8MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, d->take, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return FP8MOE_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FP8MOE_ERR_CUDA;
  *out_code = v;
  return FP8MOE_OK;
}

fp8moe_status fp8moe_testing_stall_next_gemm(void) {
  fp8moe::arm_gemm_stall_hook();
  return FP8MOE_OK;
}

fp8moe_status fp8moe_testing_stall_next_tensorwise(void) {
  fp8moe::arm_tensorwise_stall_hook();
  return FP8MOE_OK;
}

fp8moe_status fp8moe_testing_stall_next_quant_ring(void) {
  fp8moe::arm_ring_stall_hook();
  return FP8MOE_OK;
}

}  // extern "C"
