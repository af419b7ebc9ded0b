"""Plain, slow CPU oracle for the FP8 / MXFP8 MoE hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it; the library itself never
does, and shares no code with it.

Modules:
    formats     e4m3fn / e4m3fnuz / e8m0 from their definitions
    quant       rowwise, colwise (3D dense, jagged), MXFP8 dim0 / dim1
    swizzle     128x4 tiled scale layout (plain and grouped)
    grouped_mm  forward / dgrad / wgrad grouped GEMM in float64

Every function is pinned by ``tests/test_oracle_*.py`` against something other
than itself (enumeration, closed forms, torch's CPU FP8 casts on in-range
values, brute force on tiny inputs).  No function here is "parity unpinned".
"""
from . import formats, quant, swizzle, grouped_mm  # noqa: F401
