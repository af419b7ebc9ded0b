// Internal launchers shared between the kernel files and the C-ABI layer.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace fp8moe {

// Resident CTAs per SM of `kern` at `threads` threads and `smem` bytes of
// dynamic shared memory, queried on the first call and kept in `slot`.  The
// figure depends only on the kernel's resources and the SM architecture (one
// per build), so one value serves every device; the relaxed atomic keeps
// concurrent first calls from several host threads well defined.  A failed
// query yields `fallback`.
template <typename K>
inline int blocks_per_sm(std::atomic<int>& slot, K kern, int threads, size_t smem, int fallback) {
  int v = slot.load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, smem) != cudaSuccess || v < 1) {
    (void)cudaGetLastError();
    v = fallback;
  }
  slot.store(v, std::memory_order_relaxed);
  return v;
}

// Padded geometry of one swizzled scale matrix.
struct SwizzleGeom {
  int64_t Rp, Cp;  // padded rows / columns
};
SwizzleGeom swizzle_geom(int64_t R, int64_t Cs, int64_t E, int group_axis);

cudaError_t launch_quant_rowwise(const void* x, int64_t R, int64_t C, int64_t ldx, int kind, void* q,
                                 float* inv, cudaStream_t st);
// MXFP8 quantization; scales written in `layout` (FP8MOE_SCALES_ROWMAJOR,
// FP8MOE_NO_GROUPS = 128x4 per batch, FP8MOE_GROUP_ROWS / _COLS with offs).
cudaError_t launch_mx_dim0(const void* x, int64_t B, int64_t R, int64_t C, void* q, uint8_t* s, int layout,
                           const int32_t* offs, int64_t E, int num_sms, int* status, cudaStream_t st);
// MXFP8 along both dims from one read of x (R % 32 == 0, C % 32 == 0), or
// dim1 alone (q0 == NULL; C % 8 == 0); scales written in their layouts.
cudaError_t launch_mx_dual(const void* x, int64_t B, int64_t R, int64_t C, void* q0, uint8_t* s0, int s0_layout,
                           void* q1, uint8_t* s1, int s1_layout, const int32_t* offs, int64_t E, int num_sms,
                           int* status, cudaStream_t st);
// colwise FP8 (colwise.cu); jagged (offs != NULL) needs E <= 1024
cudaError_t launch_colwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                           int transpose_out, int kind, int64_t ldt, void* q, float* inv, int* status,
                           int num_sms, cudaStream_t st);

// colwise FP8 of dense [E, R, C] with transposed output in one HBM pass
// (colwise_cluster.cu), for the sizes colwise_cluster_supported accepts
bool colwise_cluster_jagged_supported(int64_t E, int64_t R, int64_t C);
// the same operation on one persistent CTA per SM (no cluster exchange);
// takes the same arguments and the same supported shapes
cudaError_t launch_colwise_jagged_ws(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs, int kind,
                                     int64_t ldt, void* q, float* inv, int* status, int num_sms, cudaStream_t st);
cudaError_t launch_colwise_cluster_jagged(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                                          int kind, int64_t ldt, void* q, float* inv, int* status, int num_sms,
                                          cudaStream_t st);
bool colwise_cluster_supported(int64_t E, int64_t R, int64_t C);
cudaError_t launch_colwise_cluster(const void* x, int64_t E, int64_t R, int64_t C, int kind, void* q, float* inv,
                                   int* status, int num_sms, cudaStream_t st);
// colwise transposed cast with one scale from the tensor's maximum (bf16
// bits at amax_bits); no per-column scales
cudaError_t launch_colwise_fixed(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs, int kind,
                                 int64_t ldt, void* q, const uint32_t* amax_bits, int* status, int num_sms,
                                 cudaStream_t st);
// tensorwise FP8: plain layout, or transposed (dense [E, C, R] / jagged
// [C, fp8moe_jagged_t_cols(R, E)]); scale_inv: one float
cudaError_t launch_tensorwise(const void* x, int64_t E, int64_t R, int64_t C, const int32_t* offs,
                              int transpose_out, int kind, void* q, float* scale_inv, int num_sms, int* status,
                              cudaStream_t st);
// blockwise FP8 (blockwise.cu): 1 x 128 row tiles, 128 x 128 weight tiles,
// per-group 128-token tiles (transposed codes)
cudaError_t launch_bw_rows(const void* x, int64_t R, int64_t C, int kind, void* q, float* inv, cudaStream_t st);
cudaError_t launch_bw_weight(const void* w, int64_t E, int64_t N, int64_t K, int kind, void* q, void* qt,
                             float* inv, cudaStream_t st);
cudaError_t launch_bw_tokens(const void* x, int64_t M, int64_t C, const int32_t* offs, int64_t E, int kind,
                             void* qt, float* inv, int num_sms, int* status, cudaStream_t st);
// token routing (routing.cu)
int64_t route_workspace_bytes(int64_t T, int64_t k, int64_t E);
cudaError_t launch_route_permute(const void* x, int64_t T, int64_t H, const int32_t* idx, const float* w, int64_t k,
                                 int64_t E, int64_t rows, void* a, int32_t* offs, int32_t* row_of, void* workspace,
                                 int num_sms, int* status, cudaStream_t st);
// the static scratch of the no-allocation permute: its size, and its device
// address on the current device (looked up on the first call per device)
int64_t route_static_scratch_bytes();
cudaError_t route_static_scratch(void** out);
cudaError_t launch_route_unpermute(const void* y, int64_t N, const int32_t* row_of, const float* w, int64_t T,
                                   int64_t k, void* out, cudaStream_t st);
cudaError_t launch_swizzle(const uint8_t* s, int64_t B, int64_t R, int64_t Cs, const int32_t* offs,
                           int64_t E, int group_axis, uint8_t* out, int* status, int num_sms,
                           cudaStream_t st);

struct GemmArgs;
cudaError_t launch_grouped_mm(const GemmArgs& g, cudaStream_t st);
// arms the one-shot stall of the next grouped GEMM launch (timeout-path test)
void arm_gemm_stall_hook();
// arms the one-shot stall of the next one-launch tensorwise kernel (its
// grid-wide meeting; timeout-path test)
void arm_tensorwise_stall_hook();
// arms the one-shot stall of the next warp-specialised quantization launch
// (dual-direction MXFP8 or jagged colwise: its first CTA never loads its
// first tile); take_ring_stall_hook reads and clears it at launch
void arm_ring_stall_hook();
int take_ring_stall_hook();
// blockwise-scaled grouped GEMM (blockwise_mm.cu)
cudaError_t launch_blockwise_mm(const GemmArgs& g, cudaStream_t st);

}  // namespace fp8moe
