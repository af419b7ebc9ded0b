"""The C-ABI library loads and exports every symbol its header declares; host-side
argument checks return their status before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as F
    return F.lib()


def _declared():
    hdr = open(os.path.join(ROOT, "include", "fp8moe.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8moe_[a-z0-9_]+)\s*\(", hdr)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    import mxfp8_moe_quantization_gb300 as F
    assert set(F.SYMBOLS) == set(names)


def test_status_strings(lib):
    """Every code of the header's fp8moe_status enum has its own message."""
    hdr = open(os.path.join(ROOT, "include", "fp8moe.h")).read()
    body = hdr[hdr.index("typedef enum {"):hdr.index("} fp8moe_status;")]
    codes = {name: int(v) for name, v in re.findall(r"(FP8MOE_\w+)\s*=\s*(\d+)", body)}
    assert codes["FP8MOE_OK"] == 0 and codes["FP8MOE_ERR_CONCURRENT"] == 8
    unknown = lib.fp8moe_status_string(max(codes.values()) + 1)
    msgs = [lib.fp8moe_status_string(c) for c in sorted(codes.values())]
    assert all(m and m != unknown for m in msgs)
    assert len(set(msgs)) == len(msgs)
    assert lib.fp8moe_version() >> 16 == 1


def test_sizes(lib):
    assert lib.fp8moe_jagged_t_cols(100, 4) == 224
    assert lib.fp8moe_jagged_t_cols(49152, 64) == (49152 + 31 * 64 + 15) // 16 * 16
    from oracle import swizzle as S, quant as Q
    for (B, R, Cs, E, ax) in [(1, 1024, 8, 4, 0), (1, 512, 32, 4, 1), (16, 8192, 160, 0, -1),
                              (1, 1, 1, 0, -1), (1, 0, 0, 0, -1)]:
        rp, cp = S.swizzled_shape(R, Cs, E, ax)
        assert lib.fp8moe_swizzled_scales_bytes(B, R, Cs, E, ax) == B * rp * cp
    assert Q.jagged_t_cols(100, 4) == lib.fp8moe_jagged_t_cols(100, 4)


def test_host_errors_before_launch(lib):
    """Invalid arguments are rejected on the host (no CUDA call is made)."""
    p = ctypes.c_void_p(1 << 20)     # aligned, never dereferenced
    mis = ctypes.c_void_p((1 << 20) + 8)
    INVALID, ALIGN, UNSUP = 1, 2, 3
    assert lib.fp8moe_quantize_rowwise(None, 4, 32, 32, 0, p, p, None) == INVALID
    assert lib.fp8moe_quantize_rowwise(p, 4, 24, 24, 0, p, p, None) == ALIGN       # C % 16
    assert lib.fp8moe_quantize_rowwise(mis, 4, 32, 32, 0, p, p, None) == ALIGN
    assert lib.fp8moe_quantize_rowwise(p, 4, 32, 32, 7, p, p, None) == INVALID     # bad kind
    assert lib.fp8moe_quantize_rowwise(p, 0, 32, 32, 0, p, p, None) == 0           # empty: no-op
    assert lib.fp8moe_mxfp8_quantize_dim0(p, 1, 4, 48, p, p, None) == ALIGN         # C % 32
    assert lib.fp8moe_mxfp8_quantize_dim1(p, 1, 48, 64, p, p, None) == ALIGN        # R % 32
    assert lib.fp8moe_mxfp8_quantize_dim0(p, 1, 0, 64, p, p, None) == 0
    assert lib.fp8moe_quantize_colwise_3d(p, 2, 24, 32, None, 1, 0, p, p, None) == ALIGN  # R % 16
    assert lib.fp8moe_swizzle_scales_128x4(p, 2, 128, 4, p, 4, 0, p, None) == INVALID    # B > 1 grouped
    assert lib.fp8moe_scaled_grouped_mm_fwd(1, p, p, p, p, p, 4, 64, 64, 48, p, None) == ALIGN  # K % 32
    assert lib.fp8moe_scaled_grouped_mm_fwd(5, p, p, p, p, p, 4, 64, 64, 64, p, None) == INVALID
    assert lib.fp8moe_scaled_grouped_mm_fwd(1, p, p, p, p, None, 4, 64, 64, 64, p, None) == INVALID
    assert lib.fp8moe_scaled_grouped_mm_wgrad(1, p, p, p, p, p, 4, 48, 64, 64, p, None) == ALIGN  # M % 32
    assert lib.fp8moe_get_device_status(None, None) == INVALID


def test_layer_workspace_and_host_errors(lib):
    """The MoE layer composites: workspace size = the kept A^T / W^T operands
    plus the larger of the forward-only and backward-only operands (each
    buffer rounded up to 256 bytes); host checks before any launch."""
    lib.fp8moe_mxfp8_moe_workspace_bytes.restype = ctypes.c_int64
    ws = lambda *a: lib.fp8moe_mxfp8_moe_workspace_bytes(*[ctypes.c_int64(v) for v in a])
    sw = lambda B, R, Cs, E, ax: lib.fp8moe_swizzled_scales_bytes(B, R, Cs, E, ax)
    up = lambda v: (v + 255) // 256 * 256
    for E, M, N, K in [(16, 16640, 8192, 5120), (4, 1024, 512, 256), (3, 0, 64, 96), (1, 32, 32, 32)]:
        kept = up(K * M) + up(sw(1, K, M // 32, E, 1)) + up(E * K * N) + up(sw(E, K, N // 32, 0, -1))
        fwd = up(M * K) + up(sw(1, M, K // 32, E, 0)) + up(E * N * K) + up(sw(E, N, K // 32, 0, -1))
        bwd = up(M * N) + up(sw(1, M, N // 32, E, 0)) + up(N * M) + up(sw(1, N, M // 32, E, 1))
        assert ws(E, M, N, K) == kept + max(fwd, bwd)
    assert ws(4, 64, 64, 48) == -1 and ws(0, 64, 64, 64) == -1 and ws(1025, 64, 64, 64) == -1
    p = ctypes.c_void_p(1 << 20)
    big = ctypes.c_int64(1 << 40)
    INVALID, ALIGN = 1, 2
    i64 = ctypes.c_int64
    assert lib.fp8moe_mxfp8_moe_fwd(p, p, p, i64(4), i64(64), i64(64), i64(48), p, p, big, None) == ALIGN
    assert lib.fp8moe_mxfp8_moe_fwd(p, p, p, i64(4), i64(64), i64(64), i64(64), p, p, i64(100), None) == INVALID
    assert lib.fp8moe_mxfp8_moe_fwd(p, p, None, i64(4), i64(64), i64(64), i64(64), p, p, big, None) == INVALID
    assert lib.fp8moe_mxfp8_moe_bwd(p, p, i64(4), i64(64), i64(64), i64(64), None, big, p, p, None) == INVALID
    assert lib.fp8moe_mxfp8_moe_bwd(p, p, i64(4), i64(64), i64(64), i64(64), p, big, None, None, None) == 0
    # jagged colwise takes at most FP8MOE_MAX_GROUPS groups
    assert lib.fp8moe_quantize_colwise_3d(p, i64(1025), i64(64), i64(32), p, 1, 0, p, p, None) == INVALID


def test_blockwise_host_errors(lib):
    p = ctypes.c_void_p(1 << 20)
    i64 = ctypes.c_int64
    INVALID, ALIGN = 1, 2
    assert lib.fp8moe_quantize_blockwise_rows(p, i64(4), i64(192), 0, p, p, None) == ALIGN        # C % 128
    assert lib.fp8moe_quantize_blockwise_rows(p, i64(0), i64(128), 0, p, p, None) == 0
    assert lib.fp8moe_quantize_blockwise_weight(p, i64(2), i64(128), i64(64), 0, p, p, p, None) == ALIGN
    assert lib.fp8moe_quantize_blockwise_weight(p, i64(2), i64(128), i64(128), 0, None, None, p, None) == INVALID
    assert lib.fp8moe_quantize_blockwise_tokens(p, i64(48), i64(32), p, i64(2), 0, p, p, None) == ALIGN  # M % 32
    assert lib.fp8moe_quantize_blockwise_tokens(p, i64(64), i64(32), None, i64(2), 0, p, p, None) == INVALID
    assert lib.fp8moe_blockwise_token_blocks(i64(16640), i64(16)) == 130 + 16
    assert lib.fp8moe_blockwise_token_blocks(i64(0), i64(0)) == -1
    # GEMM: weight tiles need N, K multiples of 128
    assert lib.fp8moe_scaled_grouped_mm_fwd(3, p, p, p, p, p, i64(4), i64(64), i64(256), i64(192), p, None) == ALIGN
    assert lib.fp8moe_scaled_grouped_mm_wgrad(3, p, p, p, p, p, i64(4), i64(48), i64(256), i64(256), p, None) == ALIGN
