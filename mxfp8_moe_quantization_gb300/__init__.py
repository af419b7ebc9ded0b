"""Python binding of libfp8moe (FP8 / MXFP8 MoE quantization + grouped GEMM).

Argument marshalling only: every function below passes device pointers,
sizes and the current CUDA stream of PyTorch to the C ABI declared in
``include/fp8moe.h`` and raises ``Fp8MoeError`` on any non-OK status.  PyTorch
provides device memory and streams; all arithmetic runs in the library's CUDA
kernels.  There is no CPU path: importing works without a GPU (so the host
logic can be tested), but every call needs the built library and a CUDA
device.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

__all__ = [
    "E4M3FN", "E4M3FNUZ", "ROWWISE", "MXFP8", "SCALES_ROWMAJOR", "NO_GROUPS", "GROUP_ROWS", "GROUP_COLS",
    "Fp8MoeError", "lib", "library_path", "SYMBOLS",
    "fp8moe_quantize_rowwise", "fp8moe_quantize_colwise_3d", "fp8moe_quantize_tensorwise",
    "fp8moe_jagged_t_cols", "fp8moe_route_rows", "fp8moe_route_workspace_bytes",
    "fp8moe_route_permute", "fp8moe_route_unpermute", "fp8moe_route_permute_noalloc",
    "ROUTE_STATIC_SCRATCH_BYTES",
    "fp8moe_mxfp8_quantize_dim0", "fp8moe_mxfp8_quantize_dim1", "fp8moe_mxfp8_quantize_dual",
    "fp8moe_swizzled_scales_bytes", "fp8moe_swizzle_scales_128x4",
    "fp8moe_scaled_grouped_mm_fwd", "fp8moe_scaled_grouped_mm_dgrad",
    "fp8moe_scaled_grouped_mm_wgrad", "fp8moe_get_device_status", "fp8moe_status_string",
    "fp8moe_mxfp8_grouped_mm_fwd_quant_a", "fp8moe_mxfp8_grouped_mm_dgrad_quant_a",
    "fp8moe_testing_stall_next_gemm",
    "fp8moe_testing_stall_next_tensorwise",
    "fp8moe_testing_stall_next_quant_ring",
    "fp8moe_mxfp8_moe_workspace_bytes", "fp8moe_mxfp8_moe_fwd", "fp8moe_mxfp8_moe_bwd",
    "fp8moe_quantize_blockwise_rows", "fp8moe_quantize_blockwise_weight", "fp8moe_blockwise_token_blocks",
    "fp8moe_quantize_blockwise_tokens",
]

E4M3FN, E4M3FNUZ = 0, 1
ROWWISE, MXFP8, TENSORWISE, BLOCKWISE = 0, 1, 2, 3
SCALES_ROWMAJOR, NO_GROUPS, GROUP_ROWS, GROUP_COLS = -2, -1, 0, 1
ROUTE_STATIC_SCRATCH_BYTES = 1 << 20   # the static scratch of fp8moe_route_permute_noalloc

HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(HERE, "libfp8moe.so")

_i64, _i32, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p

# name -> (restype, argtypes), mirroring include/fp8moe.h
SYMBOLS = {
    "fp8moe_quantize_rowwise": (_i32, [_vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp]),
    "fp8moe_quantize_colwise_3d": (_i32, [_vp, _i64, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp]),
    "fp8moe_quantize_tensorwise": (_i32, [_vp, _i64, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp]),
    "fp8moe_jagged_t_cols": (_i64, [_i64, _i64]),
    "fp8moe_route_rows": (_i64, [_i64, _i64, _i64]),
    "fp8moe_route_workspace_bytes": (_i64, [_i64, _i64, _i64]),
    "fp8moe_route_permute": (_i32, [_vp, _i64, _i64, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _vp]),
    "fp8moe_route_unpermute": (_i32, [_vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp]),
    "fp8moe_route_permute_noalloc": (_i32, [_vp, _i64, _i64, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp]),
    "fp8moe_mxfp8_quantize_dim0": (_i32, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "fp8moe_mxfp8_quantize_dim1": (_i32, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "fp8moe_mxfp8_quantize_dual": (_i32, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _i32, _vp, _vp, _i32, _vp]),
    "fp8moe_swizzled_scales_bytes": (_i64, [_i64, _i64, _i64, _i64, _i32]),
    "fp8moe_swizzle_scales_128x4": (_i32, [_vp, _i64, _i64, _i64, _vp, _i64, _i32, _vp, _vp]),
    "fp8moe_scaled_grouped_mm_fwd": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "fp8moe_scaled_grouped_mm_dgrad": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "fp8moe_scaled_grouped_mm_wgrad": (_i32, [_i32, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "fp8moe_mxfp8_grouped_mm_fwd_quant_a": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "fp8moe_mxfp8_grouped_mm_dgrad_quant_a": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                                                     _vp]),
    "fp8moe_quantize_blockwise_rows": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "fp8moe_quantize_blockwise_weight": (_i32, [_vp, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _vp]),
    "fp8moe_blockwise_token_blocks": (_i64, [_i64, _i64]),
    "fp8moe_quantize_blockwise_tokens": (_i32, [_vp, _i64, _i64, _vp, _i64, _i32, _vp, _vp, _vp]),
    "fp8moe_mxfp8_moe_workspace_bytes": (_i64, [_i64, _i64, _i64, _i64]),
    "fp8moe_mxfp8_moe_fwd": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _i64, _vp]),
    "fp8moe_mxfp8_moe_bwd": (_i32, [_vp, _vp, _i64, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp]),
    "fp8moe_get_device_status": (_i32, [_vp, ctypes.POINTER(ctypes.c_int32)]),
    "fp8moe_testing_stall_next_gemm": (_i32, []),
    "fp8moe_testing_stall_next_tensorwise": (_i32, []),
    "fp8moe_testing_stall_next_quant_ring": (_i32, []),
    "fp8moe_status_string": (ctypes.c_char_p, [_i32]),
    "fp8moe_version": (_i32, []),
}


class Fp8MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        msg = _lib_raw().fp8moe_status_string(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{fn}: status {code} ({msg})")


_LIB: Optional[ctypes.CDLL] = None


def _lib_raw() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(library_path):
            raise ImportError(
                f"libfp8moe.so is not built ({library_path}); run "
                "`python -m mxfp8_moe_quantization_gb300.build`")
        l = ctypes.CDLL(library_path)
        for name, (res, args) in SYMBOLS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _LIB = l
    return _LIB


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it is not built)."""
    return _lib_raw()


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(fn: str, code: int):
    if code != 0:
        raise Fp8MoeError(fn, code)


def _empty(shape, dtype, like):
    return _torch().empty(shape, dtype=dtype, device=like.device)


def _u8(t):
    torch = _torch()
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


# ----------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ----------------------------------------------------------------------------

def fp8moe_jagged_t_cols(M: int, E: int) -> int:
    return int(_lib_raw().fp8moe_jagged_t_cols(M, E))


def fp8moe_swizzled_scales_bytes(B: int, R: int, Cs: int, E: int = 0, group_axis: int = NO_GROUPS) -> int:
    return int(_lib_raw().fp8moe_swizzled_scales_bytes(B, R, Cs, E, group_axis))


def fp8moe_quantize_rowwise(x, kind: int = E4M3FN, q=None, scale_inv=None, stream=None):
    """x [R, C] bf16 (row stride may exceed C) -> (q uint8 [R, C], scale_inv fp32 [R])."""
    torch = _torch()
    R, C = x.shape
    q = _empty((R, C), torch.uint8, x) if q is None else q
    scale_inv = _empty((R,), torch.float32, x) if scale_inv is None else scale_inv
    _check("fp8moe_quantize_rowwise", _lib_raw().fp8moe_quantize_rowwise(
        _ptr(x), R, C, x.stride(0), kind, _ptr(q), _ptr(scale_inv), _stream(stream)))
    return q, scale_inv


def fp8moe_quantize_colwise_3d(x, offs=None, transpose_out: bool = True, kind: int = E4M3FN,
                               E: Optional[int] = None, q=None, scale_inv=None, stream=None):
    """Dense x [E, R, C] (offs None) or jagged x [R, C] with offs [E] int32 (device).

    Returns (q, scale_inv [E, C]); q is [E, C, R] / [E, R, C] (dense) or
    [C, fp8moe_jagged_t_cols(R, E)] / [R, C] (jagged).
    """
    torch = _torch()
    if offs is None:
        E_, R, C = x.shape
        qshape = (E_, C, R) if transpose_out else (E_, R, C)
    else:
        R, C = x.shape
        E_ = offs.numel() if E is None else E
        qshape = (C, fp8moe_jagged_t_cols(R, E_)) if transpose_out else (R, C)
    q = _empty(qshape, torch.uint8, x) if q is None else q
    scale_inv = _empty((E_, C), torch.float32, x) if scale_inv is None else scale_inv
    _check("fp8moe_quantize_colwise_3d", _lib_raw().fp8moe_quantize_colwise_3d(
        _ptr(x), E_, R, C, _ptr(offs), int(bool(transpose_out)), kind, _ptr(q), _ptr(scale_inv),
        _stream(stream)))
    return q, scale_inv


def fp8moe_quantize_tensorwise(x, offs=None, transpose_out: bool = False, kind: int = E4M3FN,
                               E: Optional[int] = None, q=None, scale_inv=None, stream=None):
    """One FP8 scale for the whole tensor.  Layouts as fp8moe_quantize_colwise_3d:
    dense x [E, R, C] (or any 2-D x as E = 1 when not transposed) or jagged
    x [R, C] with offs.  Returns (q, scale_inv float32 [1])."""
    torch = _torch()
    if offs is None:
        E_, R, C = x.shape if x.dim() == 3 else (1,) + tuple(x.shape)
        qshape = ((E_, C, R) if x.dim() == 3 else (C, R)) if transpose_out else tuple(x.shape)
    else:
        R, C = x.shape
        E_ = offs.numel() if E is None else E
        qshape = (C, fp8moe_jagged_t_cols(R, E_)) if transpose_out else (R, C)
    q = _empty(qshape, torch.uint8, x) if q is None else q
    scale_inv = _empty((1,), torch.float32, x) if scale_inv is None else scale_inv
    _check("fp8moe_quantize_tensorwise", _lib_raw().fp8moe_quantize_tensorwise(
        _ptr(x), E_, R, C, _ptr(offs), int(bool(transpose_out)), kind, _ptr(q), _ptr(scale_inv),
        _stream(stream)))
    return q, scale_inv


def fp8moe_route_rows(T: int, k: int, E: int) -> int:
    return int(_lib_raw().fp8moe_route_rows(T, k, E))


def fp8moe_route_workspace_bytes(T: int, k: int, E: int) -> int:
    return int(_lib_raw().fp8moe_route_workspace_bytes(T, k, E))


def fp8moe_route_permute(x, topk_idx, E: int, topk_w=None, a=None, offs=None, row_of=None, workspace=None,
                         stream=None):
    """x [T, H] bf16, topk_idx [T, k] int32 -> (a [rows, H] bf16, offs [E] int32,
    row_of [T, k] int32), every expert's group padded to 32 rows."""
    torch = _torch()
    T, H = x.shape
    k = topk_idx.shape[1]
    rows = fp8moe_route_rows(T, k, E)
    a = _empty((rows, H), torch.bfloat16, x) if a is None else a
    offs = _empty((E,), torch.int32, x) if offs is None else offs
    row_of = _empty((T, k), torch.int32, x) if row_of is None else row_of
    nbytes = fp8moe_route_workspace_bytes(T, k, E)
    workspace = _empty((max(nbytes, 4),), torch.uint8, x) if workspace is None else workspace
    _check("fp8moe_route_permute", _lib_raw().fp8moe_route_permute(
        _ptr(x), T, H, _ptr(topk_idx), _ptr(topk_w), k, E, _ptr(a), _ptr(offs), _ptr(row_of),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return a, offs, row_of


def fp8moe_route_permute_noalloc(x, topk_idx, E: int, topk_w=None, a=None, offs=None, row_of=None,
                                 stream=None):
    """fp8moe_route_permute without a workspace: the library routes through
    its own static 1 MiB device scratch, so the C call allocates nothing.
    For callers that cannot allocate device memory at routing time, pass
    preallocated ``a``, ``offs`` and ``row_of`` as well.  Calls that overlap
    on the GPU share the scratch and race."""
    torch = _torch()
    T, H = x.shape
    k = topk_idx.shape[1]
    rows = fp8moe_route_rows(T, k, E)
    a = _empty((rows, H), torch.bfloat16, x) if a is None else a
    offs = _empty((E,), torch.int32, x) if offs is None else offs
    row_of = _empty((T, k), torch.int32, x) if row_of is None else row_of
    _check("fp8moe_route_permute_noalloc", _lib_raw().fp8moe_route_permute_noalloc(
        _ptr(x), T, H, _ptr(topk_idx), _ptr(topk_w), k, E, _ptr(a), _ptr(offs), _ptr(row_of), _stream(stream)))
    return a, offs, row_of


def fp8moe_route_unpermute(y, row_of, topk_w=None, out=None, stream=None):
    """y [rows, N] bf16, row_of [T, k] -> out [T, N] bf16 (sum over k, weighted)."""
    torch = _torch()
    T, k = row_of.shape
    N = y.shape[1]
    out = _empty((T, N), torch.bfloat16, y) if out is None else out
    _check("fp8moe_route_unpermute", _lib_raw().fp8moe_route_unpermute(
        _ptr(y), T, N, _ptr(row_of), _ptr(topk_w), k, _ptr(out), _stream(stream)))
    return out


def fp8moe_mxfp8_quantize_dim0(x, q=None, scale=None, stream=None):
    """x [..., C] bf16 contiguous -> (q uint8 [..., C], scale uint8 [..., C/32])."""
    torch = _torch()
    C = x.shape[-1]
    rows = x.numel() // C if C else 0
    q = _empty(x.shape, torch.uint8, x) if q is None else q
    scale = _empty(tuple(x.shape[:-1]) + (C // 32,), torch.uint8, x) if scale is None else scale
    _check("fp8moe_mxfp8_quantize_dim0", _lib_raw().fp8moe_mxfp8_quantize_dim0(
        _ptr(x), 1, rows, C, _ptr(q), _ptr(scale), _stream(stream)))
    return q, scale


def fp8moe_mxfp8_quantize_dim1(x, qt=None, scale=None, stream=None):
    """x [B, R, C] or [R, C] bf16 -> (qt uint8 [B, C, R], scale uint8 [B, C, R/32])."""
    torch = _torch()
    squeeze = x.dim() == 2
    B, R, C = (1,) + tuple(x.shape) if squeeze else tuple(x.shape)
    qshape, sshape = (B, C, R), (B, C, R // 32)
    if squeeze:
        qshape, sshape = qshape[1:], sshape[1:]
    qt = _empty(qshape, torch.uint8, x) if qt is None else qt
    scale = _empty(sshape, torch.uint8, x) if scale is None else scale
    _check("fp8moe_mxfp8_quantize_dim1", _lib_raw().fp8moe_mxfp8_quantize_dim1(
        _ptr(x), B, R, C, _ptr(qt), _ptr(scale), _stream(stream)))
    return qt, scale


def _scale_buffer(layout, B, R, Cs, E, like):
    torch = _torch()
    if layout == SCALES_ROWMAJOR:
        return _empty((B, R, Cs) if B > 1 else (R, Cs), torch.uint8, like)
    return _torch().zeros(fp8moe_swizzled_scales_bytes(B, R, Cs, E, layout), dtype=torch.uint8, device=like.device)


def fp8moe_mxfp8_quantize_dual(x, offs=None, s0_layout: int = NO_GROUPS, s1_layout: int = NO_GROUPS,
                               dim0: bool = True, dim1: bool = True, q0=None, s0=None, q1=None, s1=None,
                               stream=None):
    """MXFP8 of x [B, R, C] (or [R, C]) along both dims from one read.

    Returns (q0 [.., R, C], s0, q1 [.., C, R], s1); scales are allocated
    zero-filled in the requested layouts when not given.  A direction with
    ``dim0=False`` / ``dim1=False`` returns None for its outputs.
    """
    torch = _torch()
    squeeze = x.dim() == 2
    B, R, C = (1,) + tuple(x.shape) if squeeze else tuple(x.shape)
    E = offs.numel() if offs is not None else 0
    if dim0:
        q0 = _empty(x.shape, torch.uint8, x) if q0 is None else q0
        s0 = _scale_buffer(s0_layout, B, R, C // 32, E, x) if s0 is None else s0
    else:
        q0 = s0 = None
    if dim1:
        q1 = _empty((C, R) if squeeze else (B, C, R), torch.uint8, x) if q1 is None else q1
        s1 = _scale_buffer(s1_layout, B, C, R // 32, E, x) if s1 is None else s1
    else:
        q1 = s1 = None
    _check("fp8moe_mxfp8_quantize_dual", _lib_raw().fp8moe_mxfp8_quantize_dual(
        _ptr(x), B, R, C, _ptr(offs), E, _ptr(q0), _ptr(s0), s0_layout, _ptr(q1), _ptr(s1), s1_layout,
        _stream(stream)))
    return q0, s0, q1, s1


def fp8moe_swizzle_scales_128x4(s, offs=None, group_axis: int = NO_GROUPS, E: Optional[int] = None,
                                out=None, stream=None):
    """s [R, Cs] or [B, R, Cs] uint8 -> flat uint8 swizzled buffer."""
    torch = _torch()
    B, R, Cs = (1,) + tuple(s.shape) if s.dim() == 2 else tuple(s.shape)
    E_ = (offs.numel() if offs is not None else 0) if E is None else E
    n = fp8moe_swizzled_scales_bytes(B, R, Cs, E_, group_axis)
    out = _empty((n,), torch.uint8, s) if out is None else out
    _check("fp8moe_swizzle_scales_128x4", _lib_raw().fp8moe_swizzle_scales_128x4(
        _ptr(s), B, R, Cs, _ptr(offs), E_, group_axis, _ptr(out), _stream(stream)))
    return out


def _gemm(name, recipe, a, a_scale, b, b_scale, offs, E, M, N, K, out, out_shape, stream):
    torch = _torch()
    out = _empty(out_shape, torch.bfloat16, a) if out is None else out
    fn = getattr(_lib_raw(), name)
    _check(name, fn(recipe, _ptr(a), _ptr(a_scale), _ptr(b), _ptr(b_scale), _ptr(offs),
                    E, M, N, K, _ptr(out), _stream(stream)))
    return out


def fp8moe_scaled_grouped_mm_fwd(recipe, a, a_scale, w, w_scale, offs, out=None, stream=None):
    """a [M, K] e4m3 (uint8), w [E, N, K] e4m3 -> out [M, N] bf16."""
    M, K = a.shape
    E, N, _ = w.shape
    return _gemm("fp8moe_scaled_grouped_mm_fwd", recipe, a, a_scale, w, w_scale, offs, E, M, N, K,
                 out, (M, N), stream)


def fp8moe_scaled_grouped_mm_dgrad(recipe, dy, dy_scale, wt, wt_scale, offs, out=None, stream=None):
    """dy [M, N], wt [E, K, N] -> dA [M, K] bf16."""
    M, N = dy.shape
    E, K, _ = wt.shape
    return _gemm("fp8moe_scaled_grouped_mm_dgrad", recipe, dy, dy_scale, wt, wt_scale, offs, E, M, N, K,
                 out, (M, K), stream)


def fp8moe_scaled_grouped_mm_wgrad(recipe, dyt, dyt_scale, at, at_scale, offs, M: int, out=None,
                                   stream=None):
    """dyt [N, Mt], at [K, Mt] -> dW [E, N, K] bf16 (M = routed rows)."""
    N = dyt.shape[0]
    K = at.shape[0]
    E = offs.numel()
    return _gemm("fp8moe_scaled_grouped_mm_wgrad", recipe, dyt, dyt_scale, at, at_scale, offs, E, M, N, K,
                 out, (E, N, K), stream)


def fp8moe_mxfp8_grouped_mm_fwd_quant_a(a, w, w_scale, offs, out=None, a_q=None, a_s=None, keep_quantized=False,
                                        stream=None):
    """a [M, K] bf16, w [E, N, K] e4m3 (uint8) with its swizzled scales ->
    out [M, N] bf16; A is quantized to MXFP8 inside the GEMM.  With
    ``keep_quantized`` (or given buffers) also returns the codes [M, K] and
    row-major e8m0 scales [M, K/32] the kernel used: (out, a_q, a_s)."""
    torch = _torch()
    M, K = a.shape
    E, N, _ = w.shape
    if keep_quantized and a_q is None:
        a_q = _empty((M, K), torch.uint8, a)
        a_s = _empty((M, K // 32), torch.uint8, a)
    out = _empty((M, N), torch.bfloat16, a) if out is None else out
    _check("fp8moe_mxfp8_grouped_mm_fwd_quant_a", _lib_raw().fp8moe_mxfp8_grouped_mm_fwd_quant_a(
        _ptr(a), _ptr(w), _ptr(w_scale), _ptr(offs), E, M, N, K, _ptr(out), _ptr(a_q), _ptr(a_s),
        _stream(stream)))
    return (out, a_q, a_s) if a_q is not None else out


def fp8moe_mxfp8_grouped_mm_dgrad_quant_a(dy, wt, wt_scale, offs, out=None, dy_q=None, dy_s=None,
                                          keep_quantized=False, stream=None):
    """dy [M, N] bf16, wt [E, K, N] e4m3 with its swizzled scales -> dA
    [M, K] bf16; dY is quantized to MXFP8 inside the GEMM (codes / scales
    returned as for the forward when asked)."""
    torch = _torch()
    M, N = dy.shape
    E, K, _ = wt.shape
    if keep_quantized and dy_q is None:
        dy_q = _empty((M, N), torch.uint8, dy)
        dy_s = _empty((M, N // 32), torch.uint8, dy)
    out = _empty((M, K), torch.bfloat16, dy) if out is None else out
    _check("fp8moe_mxfp8_grouped_mm_dgrad_quant_a", _lib_raw().fp8moe_mxfp8_grouped_mm_dgrad_quant_a(
        _ptr(dy), _ptr(wt), _ptr(wt_scale), _ptr(offs), E, M, N, K, _ptr(out), _ptr(dy_q), _ptr(dy_s),
        _stream(stream)))
    return (out, dy_q, dy_s) if dy_q is not None else out


def fp8moe_quantize_blockwise_rows(x, kind: int = E4M3FN, q=None, scale_inv=None, stream=None):
    """1 x 128 tiles along the rows of x [R, C] -> (q [R, C], scale_inv [C/128, R])."""
    torch = _torch()
    R, C = x.shape
    q = _empty((R, C), torch.uint8, x) if q is None else q
    scale_inv = _empty((C // 128, R), torch.float32, x) if scale_inv is None else scale_inv
    _check("fp8moe_quantize_blockwise_rows", _lib_raw().fp8moe_quantize_blockwise_rows(
        _ptr(x), R, C, kind, _ptr(q), _ptr(scale_inv), _stream(stream)))
    return q, scale_inv


def fp8moe_quantize_blockwise_weight(w, kind: int = E4M3FN, plain: bool = True, transposed: bool = True,
                                     q=None, qt=None, scale_inv=None, stream=None):
    """128 x 128 tiles of w [E, N, K] -> (q [E, N, K] or None, qt [E, K, N] or
    None, scale_inv [E, N/128, K/128])."""
    torch = _torch()
    E, N, K = w.shape
    q = (_empty((E, N, K), torch.uint8, w) if q is None else q) if plain else None
    qt = (_empty((E, K, N), torch.uint8, w) if qt is None else qt) if transposed else None
    scale_inv = _empty((E, N // 128, K // 128), torch.float32, w) if scale_inv is None else scale_inv
    _check("fp8moe_quantize_blockwise_weight", _lib_raw().fp8moe_quantize_blockwise_weight(
        _ptr(w), E, N, K, kind, _ptr(q), _ptr(qt), _ptr(scale_inv), _stream(stream)))
    return q, qt, scale_inv


def fp8moe_blockwise_token_blocks(M: int, E: int) -> int:
    """Rows of the token-tile scale buffer (an upper bound on the blocks)."""
    return int(_lib_raw().fp8moe_blockwise_token_blocks(M, E))


def fp8moe_quantize_blockwise_tokens(x, offs, kind: int = E4M3FN, qt=None, scale_inv=None, stream=None):
    """128-token tiles per group of x [M, C] -> (qt [C, M], scale_inv
    [fp8moe_blockwise_token_blocks(M, E), C])."""
    torch = _torch()
    M, C = x.shape
    E = offs.numel()
    qt = _empty((C, M), torch.uint8, x) if qt is None else qt
    scale_inv = (_empty((fp8moe_blockwise_token_blocks(M, E), C), torch.float32, x)
                 if scale_inv is None else scale_inv)
    _check("fp8moe_quantize_blockwise_tokens", _lib_raw().fp8moe_quantize_blockwise_tokens(
        _ptr(x), M, C, _ptr(offs), E, kind, _ptr(qt), _ptr(scale_inv), _stream(stream)))
    return qt, scale_inv


def fp8moe_mxfp8_moe_workspace_bytes(E: int, M: int, N: int, K: int) -> int:
    """Bytes of the workspace the MXFP8 MoE layer composites keep between
    forward and backward (-1 for unsupported sizes)."""
    return int(_lib_raw().fp8moe_mxfp8_moe_workspace_bytes(E, M, N, K))


def fp8moe_mxfp8_moe_fwd(a, w, offs, workspace=None, out=None, stream=None):
    """a [M, K] bf16 routed rows, w [E, N, K] bf16, offs [E] int32 (device).

    Quantizes both operands to MXFP8 (both directions) and runs the grouped
    GEMM forward.  Returns (out [M, N] bf16, workspace); pass the workspace
    to fp8moe_mxfp8_moe_bwd."""
    torch = _torch()
    M, K = a.shape
    E, N, _ = w.shape
    n = fp8moe_mxfp8_moe_workspace_bytes(E, M, N, K)
    if n < 0:
        raise Fp8MoeError("fp8moe_mxfp8_moe_fwd", 2)
    workspace = _empty((n,), torch.uint8, a) if workspace is None else workspace
    out = _empty((M, N), torch.bfloat16, a) if out is None else out
    _check("fp8moe_mxfp8_moe_fwd", _lib_raw().fp8moe_mxfp8_moe_fwd(
        _ptr(a), _ptr(w), _ptr(offs), E, M, N, K, _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream)))
    return out, workspace


def fp8moe_mxfp8_moe_bwd(dy, offs, workspace, K: int, need_da: bool = True, need_dw: bool = True,
                         da=None, dw=None, stream=None):
    """dy [M, N] bf16 and the forward's workspace -> (dA [M, K], dW [E, N, K])
    bf16; a result not asked for is returned as None."""
    torch = _torch()
    M, N = dy.shape
    E = offs.numel()
    if need_da:
        da = _empty((M, K), torch.bfloat16, dy) if da is None else da
    else:
        da = None
    if need_dw:
        dw = _empty((E, N, K), torch.bfloat16, dy) if dw is None else dw
    else:
        dw = None
    _check("fp8moe_mxfp8_moe_bwd", _lib_raw().fp8moe_mxfp8_moe_bwd(
        _ptr(dy), _ptr(offs), E, M, N, K, _ptr(workspace), workspace.numel(), _ptr(da), _ptr(dw),
        _stream(stream)))
    return da, dw


def fp8moe_get_device_status(stream=None) -> int:
    """Synchronize the stream; return and clear the sticky device status code."""
    v = ctypes.c_int32(0)
    _check("fp8moe_get_device_status", _lib_raw().fp8moe_get_device_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)


def fp8moe_testing_stall_next_gemm() -> None:
    """Arm the one-shot stall of the next grouped GEMM launch (tests of the
    bounded-wait timeout path)."""
    _check("fp8moe_testing_stall_next_gemm", _lib_raw().fp8moe_testing_stall_next_gemm())


def fp8moe_testing_stall_next_tensorwise() -> None:
    """Arm the one-shot stall of the next one-launch tensorwise kernel (tests
    of its grid-wide meeting's timeout path)."""
    _check("fp8moe_testing_stall_next_tensorwise", _lib_raw().fp8moe_testing_stall_next_tensorwise())


def fp8moe_testing_stall_next_quant_ring() -> None:
    """Arm the one-shot stall of the next warp-specialised quantization launch
    (dual-direction MXFP8 or routed-rows transposed colwise; tests of their
    rings' timeout path)."""
    _check("fp8moe_testing_stall_next_quant_ring", _lib_raw().fp8moe_testing_stall_next_quant_ring())


def fp8moe_status_string(code: int) -> str:
    return _lib_raw().fp8moe_status_string(code).decode()
