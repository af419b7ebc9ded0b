"""Benchmark: one MXFP8 MoE training step of the Llama4-Scout-shaped layer.

A step is one pass of the whole hot path over one batch of synthetic routed
tokens, for both expert weights of the layer (W1 [16, 8192, 5120] and
W2 [16, 5120, 8192]):

    MXFP8 quantize A (dim0) + swizzle, W (dim0) + swizzle  -> grouped GEMM fwd
    MXFP8 quantize dY (dim0) + swizzle, W (dim1) + swizzle -> grouped GEMM dgrad
    MXFP8 quantize dY, A (dim1) + column-grouped swizzle   -> grouped GEMM wgrad

Prints one JSON line.  ``value`` is the effective MXFP8 grouped-GEMM
throughput of the step (GEMM FLOPs over the step time, quantization
included); the line also carries the GEMM-only TFLOP/s, the quantization
GB/s, the dominant kernel's roofline, an end-to-end number through host
buffers, and the CPU oracle timed on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "scout"
METRIC = "MXFP8 grouped-GEMM TFLOP/s (% FP8 peak); fused quant HBM GB/s (% peak)"


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the GEMM
# kernel per launch, averaged over one fwd, dgrad and wgrad launch of the Scout
# W1 layer: an ncu capture of those counters on the first 8 experts, scaled to
# the full layer by each mode's algorithmic bytes.  It is reported only while
# the kernel source is the one that was captured (same SHA-256).
GEMM_TRAFFIC = {"source": "mxfp8_moe_quantization_gb300/csrc/grouped_mm.cu",
                "sha256": "503e3ef16d9dc15f9d0b947bb3bd4d632d48e0ecca09219d9fef5ad1ae2d276e",
                # full-size Scout W1 fwd / dgrad / wgrad: algorithmic bytes x the
                # traffic / algorithmic ratio of an 8-expert capture
                "bytes_per_launch": (1030.3e6 + 1055.2e6 + 1474.9e6) / 3}


def gemm_traffic():
    import hashlib
    path = os.path.join(ROOT, GEMM_TRAFFIC["source"])
    try:
        h = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return GEMM_TRAFFIC["bytes_per_launch"] if h == GEMM_TRAFFIC["sha256"] else None


def max_over_ranks(value, pg=None, device="cpu"):
    """The largest of the ranks' values (a job takes as long as its slowest
    rank); the value itself on one rank."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank, world, ms_step):
    """Whole-job throughput: every rank runs the same step on its own batch
    (weak scaling), so the job does world x the flops of one rank per step."""
    return flops_per_rank * world / (ms_step * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# the step
# ----------------------------------------------------------------------------
class ScoutStep:
    """Buffers and launches of one step; every launch goes through the C ABI."""

    def __init__(self, F, wl, device, layers=2, fused=True):
        import torch
        import workloads as W
        self.F, self.wl, self.dev = F, wl, device
        self.fused = fused
        self.offs_np = wl.offs()
        self.offs = torch.from_numpy(self.offs_np).to(device)
        self.M = wl.M
        self.E = wl.E
        self.real_tokens = int(wl.group_plan()[0].sum())
        self.layers = []
        for wname, aname, dname in [("W1", "A", "dY"), ("W2", "A2", "dY2")][:layers]:
            w = W.make_weights(wl, wname, device=device)
            a = W.make_activations(wl, aname, device=device)
            dy = W.make_activations(wl, dname, device=device)
            self.layers.append(self._alloc(w, a, dy))
        # fused: 3 quantize calls (2 kernels each: dim0 and dim1 with final-layout
        # scales) + 3 GEMMs per weight; unfused: 6 quantize + 6 swizzle + 3 GEMMs
        self.launches_per_step = (6 if fused else 15) * len(self.layers)

    def _alloc(self, w, a, dy):
        import torch
        F, dev, M, E = self.F, self.dev, self.M, self.E
        _, N, K = w.shape
        u8 = torch.uint8
        L = dict(w=w, a=a, dy=dy, N=N, K=K)
        L["qa"] = torch.empty(M, K, dtype=u8, device=dev)
        L["sa"] = torch.empty(M, K // 32, dtype=u8, device=dev)
        # swizzled scale buffers start zeroed: the fused kernels write only real
        # scale bytes, so the padding stays 0
        L["sa_sw"] = torch.zeros(F.fp8moe_swizzled_scales_bytes(1, M, K // 32, E, F.GROUP_ROWS), dtype=u8, device=dev)
        L["qw"] = torch.empty(E, N, K, dtype=u8, device=dev)
        L["sw"] = torch.empty(E, N, K // 32, dtype=u8, device=dev)
        L["sw_sw"] = torch.zeros(F.fp8moe_swizzled_scales_bytes(E, N, K // 32), dtype=u8, device=dev)
        L["out"] = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        L["qdy"] = torch.empty(M, N, dtype=u8, device=dev)
        L["sdy"] = torch.empty(M, N // 32, dtype=u8, device=dev)
        L["sdy_sw"] = torch.zeros(F.fp8moe_swizzled_scales_bytes(1, M, N // 32, E, F.GROUP_ROWS), dtype=u8, device=dev)
        L["qwt"] = torch.empty(E, K, N, dtype=u8, device=dev)
        L["swt"] = torch.empty(E, K, N // 32, dtype=u8, device=dev)
        L["swt_sw"] = torch.zeros(F.fp8moe_swizzled_scales_bytes(E, K, N // 32), dtype=u8, device=dev)
        L["da"] = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        L["qdyt"] = torch.empty(N, M, dtype=u8, device=dev)
        L["sdyt"] = torch.empty(N, M // 32, dtype=u8, device=dev)
        L["sdyt_sw"] = torch.zeros(F.fp8moe_swizzled_scales_bytes(1, N, M // 32, E, F.GROUP_COLS), dtype=u8, device=dev)
        L["qat"] = torch.empty(K, M, dtype=u8, device=dev)
        L["sat"] = torch.empty(K, M // 32, dtype=u8, device=dev)
        L["sat_sw"] = torch.zeros(F.fp8moe_swizzled_scales_bytes(1, K, M // 32, E, F.GROUP_COLS), dtype=u8, device=dev)
        L["dw"] = torch.empty(E, N, K, dtype=torch.bfloat16, device=dev)
        return L

    # accounting -------------------------------------------------------
    def gemm_flops(self):
        """Per step: 3 GEMMs per weight, 2*T*N*K each over the real routed tokens."""
        return sum(3 * 2.0 * self.real_tokens * L["N"] * L["K"] for L in self.layers)

    def quant_bytes(self):
        """Algorithmic HBM bytes of the quantization launches per step.

        Each of A, W, dY is quantized along both dimensions.  Fused, one
        launch reads the tensor once (2 B/element) and writes both codes
        (2 x 1 B) and both scale sets (2 x 1 B per 32 elements).  Unfused,
        each direction reads the tensor and writes its codes and scales, and
        the swizzle reads and writes every scale byte once more.
        """
        tot = 0.0
        for L in self.layers:
            M, N, K, E = self.M, L["N"], L["K"], self.E
            elems = M * K + E * N * K + M * N               # A, W, dY
            if self.fused:
                tot += elems * (2 + 2 + 2 / 32)
            else:
                tot += elems * 2 * (3 + 1 / 32) + elems * 2 / 32 * 2
        return tot

    def quant_elements(self):
        """Elements quantized per step, counting each direction separately."""
        return sum(2 * (self.M * L["K"] + self.E * L["N"] * L["K"] + self.M * L["N"]) for L in self.layers)

    # launches -------------------------------------------------------
    def run(self, rec=None):
        """One step.  ``rec(kind, fn)`` wraps each launch for timing."""
        F, offs = self.F, self.offs
        rec = rec or (lambda kind, fn: fn())
        if self.fused:
            for L in self.layers:
                # A: dim0 (forward operand, row-grouped scales) + dim1 (wgrad operand,
                # column-grouped scales); W: both directions, per-expert scales;
                # dY: dim0 (dgrad) + dim1 (wgrad)
                rec("quant", lambda: F.fp8moe_mxfp8_quantize_dual(
                    L["a"], offs, F.GROUP_ROWS, F.GROUP_COLS, q0=L["qa"], s0=L["sa_sw"], q1=L["qat"], s1=L["sat_sw"]))
                rec("quant", lambda: F.fp8moe_mxfp8_quantize_dual(
                    L["w"], None, F.NO_GROUPS, F.NO_GROUPS, q0=L["qw"], s0=L["sw_sw"], q1=L["qwt"], s1=L["swt_sw"]))
                rec("gemm", lambda: F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, L["qa"], L["sa_sw"], L["qw"], L["sw_sw"],
                                                                   offs, out=L["out"]))
                rec("quant", lambda: F.fp8moe_mxfp8_quantize_dual(
                    L["dy"], offs, F.GROUP_ROWS, F.GROUP_COLS, q0=L["qdy"], s0=L["sdy_sw"], q1=L["qdyt"],
                    s1=L["sdyt_sw"]))
                rec("gemm", lambda: F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, L["qdy"], L["sdy_sw"], L["qwt"],
                                                                     L["swt_sw"], offs, out=L["da"]))
                rec("gemm", lambda: F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, L["qdyt"], L["sdyt_sw"], L["qat"],
                                                                     L["sat_sw"], offs, self.M, out=L["dw"]))
            return
        for L in self.layers:
            rec("quant", lambda: F.fp8moe_mxfp8_quantize_dim0(L["a"], L["qa"], L["sa"]))
            rec("quant", lambda: F.fp8moe_swizzle_scales_128x4(L["sa"], offs, F.GROUP_ROWS, out=L["sa_sw"]))
            rec("quant", lambda: F.fp8moe_mxfp8_quantize_dim0(L["w"], L["qw"], L["sw"]))
            rec("quant", lambda: F.fp8moe_swizzle_scales_128x4(L["sw"], out=L["sw_sw"]))
            rec("gemm", lambda: F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, L["qa"], L["sa_sw"], L["qw"], L["sw_sw"],
                                                               offs, out=L["out"]))
            rec("quant", lambda: F.fp8moe_mxfp8_quantize_dim0(L["dy"], L["qdy"], L["sdy"]))
            rec("quant", lambda: F.fp8moe_swizzle_scales_128x4(L["sdy"], offs, F.GROUP_ROWS, out=L["sdy_sw"]))
            rec("quant", lambda: F.fp8moe_mxfp8_quantize_dim1(L["w"], L["qwt"], L["swt"]))
            rec("quant", lambda: F.fp8moe_swizzle_scales_128x4(L["swt"], out=L["swt_sw"]))
            rec("gemm", lambda: F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, L["qdy"], L["sdy_sw"], L["qwt"],
                                                                 L["swt_sw"], offs, out=L["da"]))
            rec("quant", lambda: F.fp8moe_mxfp8_quantize_dim1(L["dy"], L["qdyt"], L["sdyt"]))
            rec("quant", lambda: F.fp8moe_swizzle_scales_128x4(L["sdyt"], offs, F.GROUP_COLS, out=L["sdyt_sw"]))
            rec("quant", lambda: F.fp8moe_mxfp8_quantize_dim1(L["a"], L["qat"], L["sat"]))
            rec("quant", lambda: F.fp8moe_swizzle_scales_128x4(L["sat"], offs, F.GROUP_COLS, out=L["sat_sw"]))
            rec("gemm", lambda: F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, L["qdyt"], L["sdyt_sw"], L["qat"],
                                                                 L["sat_sw"], offs, self.M, out=L["dw"]))


def run_e2e(F, sets, steps, warmup, stream_weights=False):
    """Same step through host buffers: every step copies its per-step inputs
    (the routed activations A and the output gradients dY of both weights)
    in from pinned host memory and its results (the layer outputs and the
    input gradients, out and dA) back to pinned host memory; the expert
    weights and their gradients stay on the device, as model state does in
    training.  ``stream_weights`` also moves W in and dW out every step (a
    weight-streaming setup).  The copies run on their own streams and the
    steps alternate between the given buffer sets (``sets``: ScoutStep objects
    of the same shapes), so that step i's download, step i+1's compute and
    step i+2's upload overlap, as a training loop with a prefetching loader
    would; every step's transfers are inside the timed region, which ends when
    the last download has landed (one copy stream per direction: spreading
    the transfers over four streams each way measured slower).  Before the
    steps, the same buffers' copies are timed alone and both ways at once
    (``host_link``): their rates and the per-step floor they set; inside the
    timed steps, the mean duration of each step's uploads, compute and
    downloads (``host_link.in_loop_ms_per_step``)."""
    import torch
    host_in, host_out = [], []
    for st in sets:
        hi, ho = [], []
        for L in st.layers:
            for k in ("a", "w", "dy") if stream_weights else ("a", "dy"):
                hi.append((L[k], torch.empty(L[k].shape, dtype=L[k].dtype, pin_memory=True).copy_(L[k].cpu())))
            for k in ("out", "da", "dw") if stream_weights else ("out", "da"):
                ho.append((L[k], torch.empty(L[k].shape, dtype=L[k].dtype, pin_memory=True)))
        host_in.append(hi)
        host_out.append(ho)
    def h2d_bytes(hs):
        return sum(h.numel() * h.element_size() for _, h in hs[0])

    d2h_bytes = h2d_bytes
    h2d = h2d_bytes(host_in)
    d2h = d2h_bytes(host_out)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ns = len(sets)

    # the host link on these buffers: one step's uploads alone, downloads
    # alone, and both at once (their own streams, CUDA events), so that the
    # end-to-end time can be read against the copies' own floor
    def copies(up, down, reps=3):
        for it in range(reps + 1):
            e0 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e1 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            torch.cuda.synchronize()
            if up:
                with torch.cuda.stream(s_in):
                    e0[0].record(s_in)
                    for d, h in host_in[0]:
                        d.copy_(h, non_blocking=True)
                    e1[0].record(s_in)
            if down:
                with torch.cuda.stream(s_out):
                    e0[1].record(s_out)
                    for d, h in host_out[0]:
                        h.copy_(d, non_blocking=True)
                    e1[1].record(s_out)
            torch.cuda.synchronize()
            if it == 0:
                ms = [0.0, 0.0]
                continue
            if up:
                ms[0] += e0[0].elapsed_time(e1[0]) / reps
            if down:
                ms[1] += e0[1].elapsed_time(e1[1]) / reps
        return ms

    up_ms = copies(True, False)[0]
    down_ms = copies(False, True)[1]
    both = copies(True, True)
    link = {"h2d_gbs": h2d_bytes(host_in) / up_ms / 1e6, "d2h_gbs": d2h_bytes(host_out) / down_ms / 1e6,
            "h2d_gbs_concurrent": h2d_bytes(host_in) / both[0] / 1e6,
            "d2h_gbs_concurrent": d2h_bytes(host_out) / both[1] / 1e6,
            "copies_floor_ms_per_step": max(both)}
    ev_in = [torch.cuda.Event() for _ in range(ns)]
    ev_comp = [torch.cuda.Event() for _ in range(ns)]
    ev_out = [torch.cuda.Event() for _ in range(ns)]

    # per timed step: start / end events of its uploads, compute and downloads
    # (each on its own stream), to tell in the report whether the copies ran
    # at the link's rate inside the loop
    marks = []

    def one(i, mark=False):
        k = i % ns
        m = [torch.cuda.Event(enable_timing=True) for _ in range(6)] if mark else None
        with torch.cuda.stream(s_in):
            if i >= ns:
                s_in.wait_event(ev_comp[k])   # the set's previous step has read its inputs
            if m:
                m[0].record(s_in)
            for d, h in host_in[k]:
                d.copy_(h, non_blocking=True)
            if m:
                m[1].record(s_in)
            ev_in[k].record(s_in)
        comp.wait_event(ev_in[k])
        if i >= ns:
            comp.wait_event(ev_out[k])        # the set's previous results have been copied out
        if m:
            m[2].record(comp)
        sets[k].run()
        if m:
            m[3].record(comp)
        ev_comp[k].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            if m:
                m[4].record(s_out)
            for d, h in host_out[k]:
                h.copy_(d, non_blocking=True)
            if m:
                m[5].record(s_out)
            ev_out[k].record(s_out)
        if m:
            marks.append(m)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(warmup + i, mark=True)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    n = len(marks)
    link["in_loop_ms_per_step"] = {
        "h2d": sum(m[0].elapsed_time(m[1]) for m in marks) / n,
        "compute": sum(m[2].elapsed_time(m[3]) for m in marks) / n,
        "d2h": sum(m[4].elapsed_time(m[5]) for m in marks) / n}
    return dt, h2d, d2h, link


# ----------------------------------------------------------------------------
# DeepSeek-V3 layer: HBM-bound GEMMs and the standalone weight quantization
# ----------------------------------------------------------------------------
def dsv3_measure(F, dev, iters=5, warmup=2):
    """The DeepSeek-V3-shaped MoE layer (256 experts, 7168 -> 2048, 36,448
    routed rows, Zipf-skewed loads with empty experts), measured the way the
    Scout step is (CUDA events around every launch on the launching stream,
    inputs larger than L2): the standalone MXFP8 quantization of all expert
    weights (W1 [256,2048,7168] and W2 [256,7168,2048], both directions, one
    launch each) and the MXFP8 grouped GEMM forward, dgrad and wgrad of both
    weights.  Every GEMM here is bound by HBM (arithmetic intensity 123-235
    FLOP/B against a ridge near 570), so each is reported against the
    measured copy bandwidth with its algorithmic bytes: fp8 codes and e8m0
    scales of both operands (the weights of experts with tokens) plus the
    bf16 output (wgrad: every expert's dW)."""
    import torch
    import workloads as W
    wl = W.get_workload("dsv3")
    offs = torch.from_numpy(wl.offs()).to(dev)
    M, E = wl.M, wl.E
    real = wl.group_plan()[0]
    T, live = int(real.sum()), int((real > 0).sum())
    stream = torch.cuda.current_stream()
    layers = []
    for wname, aname, dname in [("W1", "A", "dY"), ("W2", "A2", "dY2")]:
        w = W.make_weights(wl, wname, device=dev)
        a = W.make_activations(wl, aname, device=dev)
        dy = W.make_activations(wl, dname, device=dev)
        _, N, K = w.shape
        qw, sw, qwt, swt = F.fp8moe_mxfp8_quantize_dual(w, None, F.NO_GROUPS, F.NO_GROUPS)
        qa, sa, qat, sat = F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, F.GROUP_COLS)
        qdy, sdy, qdyt, sdyt = F.fp8moe_mxfp8_quantize_dual(dy, offs, F.GROUP_ROWS, F.GROUP_COLS)
        del a, dy
        L = dict(name=wname, N=N, K=K, w=w, qw=qw, sw=sw, qwt=qwt, swt=swt, qa=qa, sa=sa, qat=qat, sat=sat,
                 qdy=qdy, sdy=sdy, qdyt=qdyt, sdyt=sdyt,
                 out=torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                 da=torch.empty(M, K, dtype=torch.bfloat16, device=dev),
                 dw=torch.empty(E, N, K, dtype=torch.bfloat16, device=dev))
        layers.append(L)
    # launches of one pass, with their algorithmic bytes and flops
    c = 1 + 1 / 32                          # an fp8 code and its share of an e8m0 scale
    runs = []
    for L in layers:
        N, K = L["N"], L["K"]
        fl = 2.0 * T * N * K
        runs.append((f"{L['name']}_weight_quant", L["w"].numel() * (4 + 2 / 32), 0.0,
                     lambda L=L: F.fp8moe_mxfp8_quantize_dual(L["w"], None, F.NO_GROUPS, F.NO_GROUPS, q0=L["qw"],
                                                              s0=L["sw"], q1=L["qwt"], s1=L["swt"])))
        runs.append((f"{L['name']}_fwd", (M * K + live * N * K) * c + M * N * 2, fl,
                     lambda L=L: F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, L["qa"], L["sa"], L["qw"], L["sw"], offs,
                                                                out=L["out"])))
        runs.append((f"{L['name']}_dgrad", (M * N + live * N * K) * c + M * K * 2, fl,
                     lambda L=L: F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, L["qdy"], L["sdy"], L["qwt"], L["swt"],
                                                                  offs, out=L["da"])))
        runs.append((f"{L['name']}_wgrad", (N + K) * M * c + E * N * K * 2, fl,
                     lambda L=L: F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, L["qdyt"], L["sdyt"], L["qat"], L["sat"],
                                                                  offs, M, out=L["dw"])))
    for _ in range(warmup):
        for _, _, _, fn in runs:
            fn()
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0
    evs = {name: [] for name, _, _, _ in runs}
    for _ in range(iters):
        for name, _, _, fn in runs:
            s0 = torch.cuda.Event(enable_timing=True)
            e0 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            fn()
            e0.record(stream)
            evs[name].append((s0, e0))
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0
    peaks, _ = load_peaks()
    hbm, fp8 = peaks["hbm_gbs"], 2.0 * peaks["bf16_tflops"]
    res = {}
    for name, nbytes, fl, _ in runs:
        ms = sum(s0.elapsed_time(e0) for s0, e0 in evs[name]) / iters
        d = {"us": ms * 1e3, "gbs": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm}
        if fl:
            d["tflops"] = fl / ms / 1e9
            d["frac_fp8_peak"] = fl / ms / 1e9 / fp8
        res[name] = d
    q_bytes = sum(nb for name, nb, _, _ in runs if name.endswith("weight_quant"))
    q_ms = sum(res[n]["us"] for n in res if n.endswith("weight_quant")) / 1e3
    out = {
        "dsv3_gemm_frac_hbm": {L["name"]: {m: round(res[f"{L['name']}_{m}"]["frac_hbm"], 4)
                                           for m in ("fwd", "dgrad", "wgrad")} for L in layers},
        "dsv3_weight_quant_gbs": q_bytes / q_ms / 1e6,
        "dsv3_weight_quant_frac_hbm": q_bytes / q_ms / 1e6 / hbm,
        "dsv3": {"workload": f"dsv3: {wl.description}", "routed_rows_padded": M, "real_tokens_x_topk": T,
                 "experts_with_tokens": live, "launches": res, "launches_per_pass": len(runs),
                 "passes": iters, "bound": "hbm"},
    }
    del layers, runs
    torch.cuda.empty_cache()
    return out, len(evs) * iters


# ----------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ----------------------------------------------------------------------------
def oracle_sample_step(wl):
    """A fixed fraction of one step of the workload for the CPU oracle: the
    MXFP8 quantization of a slice of the routed activations (both directions)
    and a float64 grouped GEMM forward on a slice of one expert, sized so that
    their elements and flops stand in the step's own proportion.  Returns
    (fraction, the callable step, a description)."""
    import numpy as np
    from oracle import quant as OQ, grouped_mm as OG
    import workloads as W
    T = int(wl.group_plan()[0].sum())
    M = wl.M
    step_flops = sum(3 * 2.0 * T * n * k for n, k in [(wl.N, wl.K), (wl.K, wl.N)])
    step_elems = sum(2 * (M * k + wl.E * n * k + M * n) for n, k in [(wl.N, wl.K), (wl.K, wl.N)])
    rows_q = 256                                    # quantized rows of K columns, both directions
    frac = 2.0 * rows_q * wl.K / step_elems
    gemm_flops = frac * step_flops
    rows_g = 256
    cols_g = max(16, int(round(gemm_flops / (2.0 * rows_g * wl.K) / 16)) * 16)
    frac_g = 2.0 * rows_g * cols_g * wl.K / step_flops
    frac = 0.5 * (frac + frac_g)                    # the two parts' fractions agree to within rounding
    x = W.make_activations(wl, "A").float().numpy()[:rows_q]
    a = x[:rows_g].astype(np.float64)
    w = (np.random.default_rng(0).standard_normal((1, cols_g, wl.K)) * 0.02)

    def step():
        OQ.mxfp8_quantize_dim0(x)
        OQ.mxfp8_quantize_dim1(x)
        OG.grouped_mm_fwd(a, w, np.array([rows_g]))

    desc = (f"oracle: mxfp8_quantize_dim0 + dim1 of A[:{rows_q}] ([{rows_q},{wl.K}]) and float64 grouped_mm_fwd "
            f"{rows_g}x{cols_g}x{wl.K}; {frac:.3g} of one step's quantized elements and GEMM flops")
    return frac, step, desc


def cpu_baseline(wl, budget_s=20.0):
    """The oracle's step rate (GEMM flops of the step / time) from sample
    steps run for about ``budget_s`` seconds; (TFLOP/s, description)."""
    frac, step, desc = oracle_sample_step(wl)
    step_flops = sum(3 * 2.0 * int(wl.group_plan()[0].sum()) * n * k for n, k in [(wl.N, wl.K), (wl.K, wl.N)])
    step()
    t0 = time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < budget_s and reps < 200:
        step()
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return frac * step_flops / dt / 1e12, desc + f"; {reps} sample steps"


# ----------------------------------------------------------------------------
# --rows: every hot-path row timed at its configuration size
# ----------------------------------------------------------------------------
def bench_rows(F, iters=30, only=None):
    """One JSON line per kernel: each step of the path at the configuration
    sizes of the MoE layers (CUDA events on the launching stream, the mean of
    `iters` runs after warm-up, an L2 flush between runs), with the fraction
    of its roof: HBM bytes / measured copy bandwidth, or FLOPs / measured FP8
    peak (2 x the bf16 burst), whichever the kernel is bound by.

    The event clock of these GPUs advances in steps of about 2 us, so a
    single reading of a short kernel is off by up to a step; the start of a
    run falls at a random point between steps, which makes the mean of many
    readings unbiased where a median would stay on the step grid.  Readings
    more than twice the median (a run interrupted by something else) are
    left out."""
    import torch
    import workloads as W
    dev = torch.device("cuda")
    sections = set(only.split(",")) if only else None

    def want(name):
        return sections is None or name in sections

    peaks, peak_kind = load_peaks()
    hbm, fp8 = peaks["hbm_gbs"], 2.0 * peaks["bf16_tflops"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean = torch.zeros(64 << 20, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(iters):
            # L2 flush: write a buffer twice the size of L2, then read another
            # one, so that the write-backs of the flush's dirty lines finish
            # before the timed region (the kernel starts from a cold, clean L2)
            flush.fill_(1)
            clean.max()
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            # keep the GPU busy while the host enqueues the timed call, so
            # that its launch latency is not inside the events
            torch.cuda._sleep(200000)
            s.record(stream)
            fn()
            e.record(stream)
            torch.cuda.synchronize()
            ts.append(s.elapsed_time(e))
        assert F.fp8moe_get_device_status() == 0
        ts.sort()
        med = ts[len(ts) // 2]
        kept = [t for t in ts if t <= 2.0 * med]
        return sum(kept) / len(kept)

    def emit(row, kernel, config, ms, nbytes=None, flops=None, roof_of_hbm=False):
        d = {"row": row, "kernel": kernel, "config": config, "us": round(ms * 1e3, 1)}
        if flops is not None:
            d["tflops"] = round(flops / ms / 1e9, 1)
            d["frac_fp8_peak"] = round(flops / ms / 1e9 / fp8, 3)
        if nbytes is not None:
            d["gbs"] = round(nbytes / ms / 1e6, 1)
            d["frac_hbm"] = round(nbytes / ms / 1e6 / hbm, 3)
        if roof_of_hbm:
            d["bound"] = "hbm"
        d["peaks"] = peak_kind
        print(json.dumps(d), flush=True)

    def codes(*shape):
        return torch.randint(0, 120, shape, dtype=torch.uint8, device=dev)

    # ---- quantization rows (a1, a2, a10, tensorwise) on the rowwise configs
    ll, ds, sc, v3 = (W.get_workload(n) for n in ("llama3_8b", "dsmoe_16b", "scout", "dsv3"))
    x = W.make_activations(ll, "A", device=dev)
    wll = W.make_weights(ll, "W1", device=dev).reshape(ll.N, ll.K)
    if want("rowwise"):
        for kind, tag in ((F.E4M3FN, "a1"), (F.E4M3FNUZ, "a10")):
            for name, t in (("X [8192,4096]", x), ("W [14336,4096]", wll)):
                q = torch.empty(t.shape, dtype=torch.uint8, device=dev)
                inv = torch.empty(t.shape[0], dtype=torch.float32, device=dev)
                ms = timed(lambda: F.fp8moe_quantize_rowwise(t, kind=kind, q=q, scale_inv=inv))
                emit(tag, "k_quant_rowwise", f"llama3_8b {name}", ms, nbytes=t.numel() * 3 + t.shape[0] * 4)
        ads = W.make_activations(ds, "A", device=dev)
        qa = torch.empty(ads.shape, dtype=torch.uint8, device=dev)
        ia = torch.empty(ds.M, dtype=torch.float32, device=dev)
        ms = timed(lambda: F.fp8moe_quantize_rowwise(ads, q=qa, scale_inv=ia))
        emit("a1", "k_quant_rowwise", f"dsmoe_16b A [{ds.M},{ds.K}]", ms, nbytes=ads.numel() * 3 + ds.M * 4)
        del ads
    if want("colwise"):
        q = torch.empty(wll.shape[::-1], dtype=torch.uint8, device=dev)
        inv = torch.empty(1, ll.K, dtype=torch.float32, device=dev)
        ms = timed(lambda: F.fp8moe_quantize_colwise_3d(wll[None], None, True, q=q, scale_inv=inv))
        emit("a2", "k_cw_cluster (one pass)", "llama3_8b W^T [1,14336,4096] transposed", ms, nbytes=wll.numel() * 3 + ll.K * 4)
        dsoffs = torch.from_numpy(ds.offs()).to(dev)
        for which in ("W1", "W2"):
            wds = W.make_weights(ds, which, device=dev)
            q = torch.empty((wds.shape[0], wds.shape[2], wds.shape[1]), dtype=torch.uint8, device=dev)
            inv = torch.empty(wds.shape[0], wds.shape[2], dtype=torch.float32, device=dev)
            ms = timed(lambda: F.fp8moe_quantize_colwise_3d(wds, None, True, q=q, scale_inv=inv))
            emit("a2", "k_cw_cluster (one pass)", f"dsmoe_16b {which} {list(wds.shape)} transposed", ms,
                 nbytes=wds.numel() * 3 + wds.shape[0] * wds.shape[2] * 4)
            del wds
        ads = W.make_activations(ds, "A", device=dev)
        q = torch.empty((ds.K, F.fp8moe_jagged_t_cols(ds.M, ds.E)), dtype=torch.uint8, device=dev)
        inv = torch.empty(ds.E, ds.K, dtype=torch.float32, device=dev)
        ms = timed(lambda: F.fp8moe_quantize_colwise_3d(ads, dsoffs, True, q=q, scale_inv=inv))
        emit("a2", "k_cw_jag_ws (one pass, one CTA per group strip)", f"dsmoe_16b jagged A [{ds.M},{ds.K}] transposed", ms,
             nbytes=ads.numel() * 3 + ds.E * ds.K * 4)
        del ads
    if want("tensorwise"):
        for name, t in (("X [8192,4096]", x), ("W [14336,4096]", wll)):
            q = torch.empty(t.shape, dtype=torch.uint8, device=dev)
            inv = torch.empty(1, dtype=torch.float32, device=dev)
            ms = timed(lambda: F.fp8moe_quantize_tensorwise(t, q=q, scale_inv=inv))
            emit("next4", "k_tw_stream (one launch)", f"llama3_8b {name} tensorwise", ms, nbytes=t.numel() * 3)
    del x, wll

    # ---- MXFP8 quantization rows (a3, a4, a5, fused dual) on Scout and DeepSeek-V3
    soffs = torch.from_numpy(sc.offs()).to(dev)
    if want("mx") or want("swizzle"):
        a = W.make_activations(sc, "A", device=dev)
        w1 = W.make_weights(sc, "W1", device=dev)
    if want("mx"):
        for name, t, offs, l0, l1 in (("A [16640,5120]", a, soffs, F.GROUP_ROWS, F.GROUP_COLS),
                                      ("W1 [16,8192,5120]", w1, None, F.NO_GROUPS, F.NO_GROUPS)):
            o = F.fp8moe_mxfp8_quantize_dual(t, offs, l0, l1)
            n = t.numel()
            ms = timed(lambda: F.fp8moe_mxfp8_quantize_dim0(t, q=o[0]))
            emit("a3", "k_mx_dim0", f"scout {name}", ms, nbytes=n * (3 + 1 / 32))
            ms = timed(lambda: F.fp8moe_mxfp8_quantize_dim1(t, qt=o[2]))
            emit("a4", "k_mx_dual<dim1>", f"scout {name}", ms, nbytes=n * (3 + 1 / 32))
            ms = timed(lambda: F.fp8moe_mxfp8_quantize_dual(t, offs, l0, l1, q0=o[0], s0=o[1], q1=o[2], s1=o[3]))
            emit("next1", "k_mx_dual_ws (both directions, one read)", f"scout {name} final-layout scales", ms,
                 nbytes=n * (4 + 2 / 32))
    if want("swizzle"):
        s_rm = torch.empty(sc.E, sc.N, sc.K // 32, dtype=torch.uint8, device=dev)
        F.fp8moe_mxfp8_quantize_dim0(w1, scale=s_rm)
        s_sw = torch.zeros(F.fp8moe_swizzled_scales_bytes(sc.E, sc.N, sc.K // 32), dtype=torch.uint8, device=dev)
        ms = timed(lambda: F.fp8moe_swizzle_scales_128x4(s_rm, out=s_sw))
        emit("a5", "k_swizzle_rows (one bulk copy per 128-row block)", "scout W1 scales [16,8192,160]", ms, nbytes=s_rm.numel() * 2)
    if want("mx") or want("swizzle"):
        del a, w1
    if want("mx"):
        w3 = W.make_weights(v3, "W1", device=dev)
        o = F.fp8moe_mxfp8_quantize_dual(w3, None, F.NO_GROUPS, F.NO_GROUPS)
        ms = timed(lambda: F.fp8moe_mxfp8_quantize_dual(w3, None, F.NO_GROUPS, F.NO_GROUPS, q0=o[0], s0=o[1], q1=o[2],
                                                         s1=o[3]))
        emit("next1", "k_mx_dual_ws (both directions, one read)", "dsv3 W1 [256,2048,7168]", ms,
             nbytes=w3.numel() * (4 + 2 / 32))
        ms = timed(lambda: F.fp8moe_mxfp8_quantize_dim0(w3, q=o[0]))
        emit("a3", "k_mx_dim0", "dsv3 W1 [256,2048,7168]", ms, nbytes=w3.numel() * (3 + 1 / 32))
        del w3, o

    # ---- grouped GEMMs (a6-a8): MXFP8 on Scout and DeepSeek-V3, rowwise on
    # DeepSeek-MoE-16B and the dense Llama3 linear
    if want("gemm"):
        for wl in (sc, v3):
            offs = torch.from_numpy(wl.offs()).to(dev)
            M, E, T = wl.M, wl.E, int(wl.group_plan()[0].sum())
            live = int((wl.group_plan()[0] > 0).sum())
            for (N, K, wname) in ((wl.N, wl.K, "W1"), (wl.K, wl.N, "W2")):
                flops = 2.0 * T * N * K
                qa, qw, qdy, qwt = codes(M, K), codes(E, N, K), codes(M, N), codes(E, K, N)
                qdyt, qat = codes(N, M), codes(K, M)

                def sc_(n):
                    return torch.full((n,), 127, dtype=torch.uint8, device=dev)
                sa = sc_(F.fp8moe_swizzled_scales_bytes(1, M, K // 32, E, F.GROUP_ROWS))
                sw = sc_(F.fp8moe_swizzled_scales_bytes(E, N, K // 32))
                sdy = sc_(F.fp8moe_swizzled_scales_bytes(1, M, N // 32, E, F.GROUP_ROWS))
                swt = sc_(F.fp8moe_swizzled_scales_bytes(E, K, N // 32))
                sdyt = sc_(F.fp8moe_swizzled_scales_bytes(1, N, M // 32, E, F.GROUP_COLS))
                sat = sc_(F.fp8moe_swizzled_scales_bytes(1, K, M // 32, E, F.GROUP_COLS))
                out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
                da = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
                dw = torch.empty(E, N, K, dtype=torch.bfloat16, device=dev)
                # HBM bytes: fp8 operands (weights of live experts) + bf16 output
                fb = M * K + live * N * K + M * N * 2
                db = M * N + live * N * K + M * K * 2
                wb = (N + K) * M + E * N * K * 2
                cfg = f"{wl.name} {wname} M={M} N={N} K={K} E={E}"
                hb = wl.name == "dsv3"
                ms = timed(lambda: F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs, out=out))
                emit("a6", "k_grouped_mm<MX,fwd>", cfg, ms, nbytes=fb, flops=flops, roof_of_hbm=hb)
                ms = timed(lambda: F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qdy, sdy, qwt, swt, offs, out=da))
                emit("a7", "k_grouped_mm<MX,dgrad>", cfg, ms, nbytes=db, flops=flops, roof_of_hbm=hb)
                ms = timed(lambda: F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, offs, M, out=dw))
                emit("a8", "k_grouped_mm<MX,wgrad>", cfg, ms, nbytes=wb, flops=flops, roof_of_hbm=hb)
                del qa, qw, qdy, qwt, qdyt, qat, out, da, dw
    # the rowwise recipe's GEMMs also run alone (--only gemm_rowwise): under
    # 2 GB on the device, the case the profiler captures
    if want("gemm") or want("gemm_rowwise"):
        for wl in (ds, ll):
            offs = torch.from_numpy(wl.offs()).to(dev)
            M, E, N, K = wl.M, wl.E, wl.N, wl.K
            Mt = F.fp8moe_jagged_t_cols(M, E)
            flops = 2.0 * M * N * K
            qa, qw, qdy, qwt, qdyt, qat = codes(M, K), codes(E, N, K), codes(M, N), codes(E, K, N), codes(N, Mt), codes(K, Mt)
            s_m = torch.ones(M, dtype=torch.float32, device=dev)
            s_en = torch.ones(E, N, dtype=torch.float32, device=dev)
            s_ek = torch.ones(E, K, dtype=torch.float32, device=dev)
            cfg = f"{wl.name} M={M} N={N} K={K} E={E}"
            out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            ms = timed(lambda: F.fp8moe_scaled_grouped_mm_fwd(F.ROWWISE, qa, s_m, qw, s_en, offs, out=out))
            emit("a6", "k_grouped_mm<rowwise,fwd>", cfg, ms, flops=flops)
            da = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
            ms = timed(lambda: F.fp8moe_scaled_grouped_mm_dgrad(F.ROWWISE, qdy, s_m, qwt, s_ek, offs, out=da))
            emit("a7", "k_grouped_mm<rowwise,dgrad>", cfg, ms, flops=flops)
            dw = torch.empty(E, N, K, dtype=torch.bfloat16, device=dev)
            ms = timed(lambda: F.fp8moe_scaled_grouped_mm_wgrad(F.ROWWISE, qdyt, s_en, qat, s_ek, offs, M, out=dw))
            emit("a8", "k_grouped_mm<rowwise,wgrad>", cfg, ms, flops=flops)
            del qa, qw, qdy, qwt, qdyt, qat, out, da, dw

    # ---- activation quantization fused into the GEMM prologue (a9 and its
    # dgrad twin) against the unfused chain: the dim0 quantization of the
    # bf16 operand (scales straight into the grouped layout) then the GEMM
    if want("fused"):
        for wl in (sc, v3):
            offs = torch.from_numpy(wl.offs()).to(dev)
            M, E, N, K = wl.M, wl.E, wl.N, wl.K
            T = int(wl.group_plan()[0].sum())
            flops = 2.0 * T * N * K
            a = W.make_activations(wl, "A", device=dev)
            dy = W.make_activations(wl, "dY", device=dev)
            w = W.make_weights(wl, "W1", device=dev)
            qw, sw, qwt, swt = F.fp8moe_mxfp8_quantize_dual(w, None, F.NO_GROUPS, F.NO_GROUPS)
            del w
            out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            da = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
            qa, sa, _, _ = F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, dim1=False)
            qd, sd, _, _ = F.fp8moe_mxfp8_quantize_dual(dy, offs, F.GROUP_ROWS, dim1=False)
            cfg = f"{wl.name} W1 M={M} N={N} K={K} E={E}"

            def chain_fwd():
                F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, dim1=False, q0=qa, s0=sa)
                F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs, out=out)

            def chain_dgrad():
                F.fp8moe_mxfp8_quantize_dual(dy, offs, F.GROUP_ROWS, dim1=False, q0=qd, s0=sd)
                F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qd, sd, qwt, swt, offs, out=da)
            ms = timed(chain_fwd)
            emit("a9", "k_mx_dim0 + k_grouped_mm<MX,fwd> (unfused)", cfg, ms, flops=flops)
            ms = timed(lambda: F.fp8moe_mxfp8_grouped_mm_fwd_quant_a(a, qw, sw, offs, out=out))
            emit("a9", "k_grouped_mm<MX,fwd,quant-A prologue>", cfg, ms, flops=flops)
            ms = timed(chain_dgrad)
            emit("next1", "k_mx_dim0 + k_grouped_mm<MX,dgrad> (unfused)", cfg, ms, flops=flops)
            ms = timed(lambda: F.fp8moe_mxfp8_grouped_mm_dgrad_quant_a(dy, qwt, swt, offs, out=da))
            emit("next1", "k_grouped_mm<MX,dgrad,quant-dY prologue>", cfg, ms, flops=flops)
            del a, dy, qw, sw, qwt, swt, out, da, qa, sa, qd, sd

    # ---- MoE layer composites (next1) and blockwise scaling (next3) on the
    # Scout W1 layer
    if want("layer") or want("blockwise"):
        soffs = torch.from_numpy(sc.offs()).to(dev)
        M, E, N, K = sc.M, sc.E, sc.N, sc.K
        T = int(sc.group_plan()[0].sum())
        flops = 2.0 * T * N * K
        a = W.make_activations(sc, "A", device=dev)
        w = W.make_weights(sc, "W1", device=dev)
        dy = torch.randn(M, N, device=dev).to(torch.bfloat16)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        da = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dw = torch.empty(E, N, K, dtype=torch.bfloat16, device=dev)
        cfg = f"scout W1 M={M} N={N} K={K} E={E}"
    if want("layer"):
        ws = torch.empty(F.fp8moe_mxfp8_moe_workspace_bytes(E, M, N, K), dtype=torch.uint8, device=dev)
        ms = timed(lambda: F.fp8moe_mxfp8_moe_fwd(a, w, soffs, workspace=ws, out=out))
        emit("next1", "fp8moe_mxfp8_moe_fwd (2 dual quant + fwd GEMM)", cfg, ms, flops=flops)
        ms = timed(lambda: F.fp8moe_mxfp8_moe_bwd(dy, soffs, ws, K, da=da, dw=dw))
        emit("next1", "fp8moe_mxfp8_moe_bwd (dual quant + dgrad + wgrad)", cfg, ms, flops=2 * flops)
        del ws
    if want("blockwise"):
        qa, sa = F.fp8moe_quantize_blockwise_rows(a)
        ms = timed(lambda: F.fp8moe_quantize_blockwise_rows(a, q=qa, scale_inv=sa))
        emit("next3", "k_bw_rows", f"scout A [{M},{K}] 1x128", ms, nbytes=a.numel() * (3 + 4 / 128))
        qw, qwt, sw = F.fp8moe_quantize_blockwise_weight(w)
        ms = timed(lambda: F.fp8moe_quantize_blockwise_weight(w, q=qw, qt=qwt, scale_inv=sw))
        emit("next3", "k_bw_weight (both layouts)", f"scout W1 {list(w.shape)} 128x128", ms, nbytes=w.numel() * 4)
        qat, sat = F.fp8moe_quantize_blockwise_tokens(a, soffs)
        ms = timed(lambda: F.fp8moe_quantize_blockwise_tokens(a, soffs, qt=qat, scale_inv=sat))
        emit("next3", "k_bw_tokens", f"scout A [{M},{K}] 128-token tiles", ms, nbytes=a.numel() * (3 + 4 / 128))
        qdy, sdy = F.fp8moe_quantize_blockwise_rows(dy)
        qdyt, sdyt = F.fp8moe_quantize_blockwise_tokens(dy, soffs)
        ms = timed(lambda: F.fp8moe_scaled_grouped_mm_fwd(F.BLOCKWISE, qa, sa, qw, sw, soffs, out=out))
        emit("next3", "k_blockwise_mm<fwd>", cfg, ms, flops=flops)
        ms = timed(lambda: F.fp8moe_scaled_grouped_mm_dgrad(F.BLOCKWISE, qdy, sdy, qwt, sw, soffs, out=da))
        emit("next3", "k_blockwise_mm<dgrad>", cfg, ms, flops=flops)
        ms = timed(lambda: F.fp8moe_scaled_grouped_mm_wgrad(F.BLOCKWISE, qdyt, sdyt, qat, sat, soffs, M, out=dw))
        emit("next3", "k_blockwise_mm<wgrad>", cfg, ms, flops=flops)
        del qa, qw, qwt, qat, qdy, qdyt
    if want("layer") or want("blockwise"):
        del a, w, dy, out, da, dw

    # ---- routing (next2) on the Scout and DeepSeek-V3 token counts
    if want("routing"):
        for wl, k in ((sc, 1), (v3, 8)):
            T, E, H = wl.tokens, wl.E, wl.K
            g = torch.Generator(device=dev).manual_seed(wl.seed)
            idx = torch.stack([torch.randperm(E, device=dev, generator=g)[:k] for _ in range(T)]).to(torch.int32) \
                if k > 1 else torch.randint(0, E, (T, 1), device=dev, generator=g, dtype=torch.int32)
            xt = torch.randn(T, H, device=dev, generator=g).to(torch.bfloat16)
            wt = torch.rand(T, k, device=dev, generator=g)
            ws = torch.empty(max(F.fp8moe_route_workspace_bytes(T, k, E), 4), dtype=torch.uint8, device=dev)
            a, offs, row_of = F.fp8moe_route_permute(xt, idx, E, workspace=ws)
            ms = timed(lambda: F.fp8moe_route_permute(xt, idx, E, a=a, offs=offs, row_of=row_of, workspace=ws))
            emit("next2", "route_permute (count, scan, rank, copy)", f"{wl.name} T={T} k={k} E={E} H={H}", ms,
                 nbytes=T * H * 2 + a.numel() * 2)
            outt = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
            ms = timed(lambda: F.fp8moe_route_unpermute(a, row_of, wt, out=outt))
            emit("next2", "k_route_unpermute", f"{wl.name} T={T} k={k} N={H}", ms, nbytes=T * k * H * 2 + T * H * 2)
            del xt, a, outt


def dual_case(F, dev):
    """The fused dual-direction MXFP8 quantization of the Scout activations
    A [16640, 5120] (routing offsets of 16 experts, both code layouts with
    grouped 128x4 scales): the step's first k_mx_dual launch on its own, a
    case for profiler captures that holds under 1 GB on the device.  Runs
    once as warm-up and once timed, and prints the time."""
    import torch
    import workloads as W
    sc = W.get_workload("scout")
    a = W.make_activations(sc, "A", device=dev)
    offs = torch.from_numpy(sc.offs()).to(dev)
    run = lambda: F.fp8moe_mxfp8_quantize_dual(a, offs, F.GROUP_ROWS, F.GROUP_COLS)
    run()
    torch.cuda.synchronize()
    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    run()
    e0.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(e0)
    print(json.dumps({"case": "scout A dual-direction MXFP8", "shape": list(a.shape), "us": round(ms * 1e3, 1),
                      "gbs": round(a.numel() * (2 + 2 + 2 / 32) / ms / 1e6, 1)}))
    assert F.fp8moe_get_device_status() == 0


def gemm_case(F, dev, n_experts):
    """The Scout W1 grouped GEMMs restricted to the first ``n_experts`` experts
    and their routed rows (fp8 codes of random bytes, unit e8m0 scales): a
    reduced case of the same kernels for profiler captures.  Runs forward,
    dgrad and wgrad once as warm-up and once timed, and prints the times."""
    import torch
    import workloads as W
    E = n_experts
    sizes = W.group_sizes("scout")[:E]
    offs = torch.from_numpy(W.offsets_from_sizes(sizes)).to(dev)
    M, N, K = int(sum(sizes)), W.get_workload("scout").N, W.get_workload("scout").K
    g = torch.Generator(device=dev).manual_seed(0)

    def codes(*shape):
        return torch.randint(0, 120, shape, dtype=torch.uint8, device=dev, generator=g)

    def unit(n):
        return torch.full((n,), 127, dtype=torch.uint8, device=dev)
    qa, qw, qdy, qwt, qdyt, qat = codes(M, K), codes(E, N, K), codes(M, N), codes(E, K, N), codes(N, M), codes(K, M)
    sa = unit(F.fp8moe_swizzled_scales_bytes(1, M, K // 32, E, F.GROUP_ROWS))
    sw = unit(F.fp8moe_swizzled_scales_bytes(E, N, K // 32))
    sdy = unit(F.fp8moe_swizzled_scales_bytes(1, M, N // 32, E, F.GROUP_ROWS))
    swt = unit(F.fp8moe_swizzled_scales_bytes(E, K, N // 32))
    sdyt = unit(F.fp8moe_swizzled_scales_bytes(1, N, M // 32, E, F.GROUP_COLS))
    sat = unit(F.fp8moe_swizzled_scales_bytes(1, K, M // 32, E, F.GROUP_COLS))
    out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    da = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(E, N, K, dtype=torch.bfloat16, device=dev)
    runs = [("fwd", lambda: F.fp8moe_scaled_grouped_mm_fwd(F.MXFP8, qa, sa, qw, sw, offs, out=out)),
            ("dgrad", lambda: F.fp8moe_scaled_grouped_mm_dgrad(F.MXFP8, qdy, sdy, qwt, swt, offs, out=da)),
            ("wgrad", lambda: F.fp8moe_scaled_grouped_mm_wgrad(F.MXFP8, qdyt, sdyt, qat, sat, offs, M, out=dw))]
    for _, fn in runs:
        fn()
    torch.cuda.synchronize()
    for name, fn in runs:
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        fn()
        e0.record()
        torch.cuda.synchronize()
        ms = s0.elapsed_time(e0)
        print(json.dumps({"case": f"scout W1, first {E} experts", "mode": name, "M": M, "N": N, "K": K,
                          "us": round(ms * 1e3, 1), "tflops": round(2.0 * M * N * K / ms / 1e9, 1)}))
    assert F.fp8moe_get_device_status() == 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--layers", type=int, default=2, choices=[1, 2],
                    help="expert weights per step (2 = W1 and W2; 1 = W1 only, for profiling)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="separate dim0 / dim1 / swizzle launches instead of the fused dual-direction kernel")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-dsv3", action="store_true", help="skip the DeepSeek-V3 layer measurements")
    ap.add_argument("--only", default=None,
                    help="with --rows: comma-separated sections (rowwise, colwise, tensorwise, mx, swizzle, gemm, gemm_rowwise, "
                         "fused, layer, blockwise, routing)")
    ap.add_argument("--gemm-case", type=int, default=0, metavar="E",
                    help="run the Scout W1 grouped GEMMs on the first E experts only (a reduced case for "
                         "profiler captures) and exit")
    ap.add_argument("--dual-case", action="store_true",
                    help="run the fused dual-direction quantization of the Scout activations once (a reduced "
                         "case for profiler captures) and exit")
    ap.add_argument("--rows", action="store_true",
                    help="time every hot-path kernel at its configuration size (one JSON line each) and exit")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    import workloads as W
    wl = W.get_workload(WORKLOAD)

    if args.impl == "reference":
        # the reference arm is the CPU oracle (the pages ship no runnable
        # code): every step runs the oracle on the same fixed fraction of one
        # Scout step (its quantization and its GEMM work in the step's
        # proportion), so the rate is measured, not projected
        if rank != 0:
            return
        frac, sample_step, sample = oracle_sample_step(wl)
        step_flops = sum(3 * 2.0 * int(wl.group_plan()[0].sum()) * n * k
                         for n, k in [(wl.N, wl.K), (wl.K, wl.N)])
        for _ in range(args.warmup):
            sample_step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            sample_step()
        t_sample = (time.perf_counter() - t0) / args.steps
        val = frac * step_flops / t_sample / 1e12
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_sample * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl.name}: {wl.description}", "step": sample,
                       "step_fraction_of_workload_step": frac},
            "extrapolated": False,
            "full_step_ms_estimate": t_sample / frac * 1e3,
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return

    import torch
    from mxfp8_moe_quantization_gb300 import build as B
    B.build()
    import mxfp8_moe_quantization_gb300 as F

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if args.rows:
        bench_rows(F, only=args.only)
        return
    if args.gemm_case:
        gemm_case(F, dev, args.gemm_case)
        return
    if args.dual_case:
        dual_case(F, dev)
        return
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    step = ScoutStep(F, wl, dev, layers=args.layers, fused=not args.unfused)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    assert F.fp8moe_get_device_status() == 0

    # timed region: events around every launch on the launching stream
    ev = {"gemm": [], "quant": []}

    def rec(kind, fn):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        ev[kind].append((s, e))

    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clk:
        t_start.record(stream)
        for _ in range(args.steps):
            step.run(rec)
        t_end.record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), pg, dev)
    ms_step = ms_total / args.steps
    gemm_ms = sum(s.elapsed_time(e) for s, e in ev["gemm"]) / args.steps
    quant_ms = sum(s.elapsed_time(e) for s, e in ev["quant"]) / args.steps
    n_gemm = len(ev["gemm"]) // args.steps
    flops = step.gemm_flops()
    qbytes = step.quant_bytes()
    assert F.fp8moe_get_device_status() == 0

    peaks, peak_kind = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]          # nominal fp8:bf16 dense ratio 4.5 / 2.25
    gemm_launch_ms = gemm_ms / n_gemm
    achieved = flops / n_gemm / (gemm_launch_ms * 1e-3) / 1e12
    value = job_tflops(flops, world, ms_step)

    e2e = e2e_ws = None
    if not args.no_e2e:
        # a second buffer set of the same shapes lets transfers and compute
        # of neighbouring steps overlap
        step2 = ScoutStep(F, wl, dev, layers=args.layers, fused=not args.unfused)
        dt, h2d, d2h, link = run_e2e(F, [step, step2], max(4, args.steps // 3), 2)
        dt = max_over_ranks(dt, pg, dev)
        e2e = {"value": job_tflops(flops, world, dt * 1e3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3,
               "moves": "A, dY in; out, dA back (weights and weight gradients resident)", "host_link": link}
        dt, h2d, d2h, link = run_e2e(F, [step, step2], max(4, args.steps // 6), 2, stream_weights=True)
        del step2
        dt = max_over_ranks(dt, pg, dev)
        e2e_ws = {"value": job_tflops(flops, world, dt * 1e3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3,
                  "moves": "A, W, dY in; out, dA, dW back", "host_link": link}
    extra, extra_launches = ({}, 0) if args.no_dsv3 else dsv3_measure(F, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        rate, sample = cpu_baseline(wl)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle", "sample": sample}

    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 x e4m3 (e8m0 scales) -> fp32 accum -> bf16", "data": "synthetic",
            "config": {"workload": f"{wl.name}: {wl.description}", "experts": wl.E, "tokens": wl.tokens,
                       "routed_rows_padded": wl.M, "hidden": wl.K, "ffn": wl.N, "weights": args.layers,
                       "l2": "inputs larger than L2 (each expert weight is 1.34 GB bf16)",
                       "quant": "fused dual-direction" if step.fused else "separate dim0/dim1/swizzle"},
            "gemm_tflops": flops / (gemm_ms * 1e-3) / 1e12,
            "gemm_frac_fp8_peak": flops / (gemm_ms * 1e-3) / 1e12 / fp8_peak,
            "quant_gbs": qbytes / (quant_ms * 1e-3) / 1e9,
            "quant_frac_hbm": qbytes / (quant_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "gemm_ms_per_step": gemm_ms, "quant_ms_per_step": quant_ms,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                         "frac": achieved / fp8_peak, "traffic": gemm_traffic(),
                         "kernel": "k_grouped_mm<MX=true>", "peak_source":
                             f"{peak_kind}: 2 x bf16_tflops (nominal fp8/bf16 dense ratio)"},
            "clocks": clk.summary(),
            "e2e": e2e,
            "e2e_weights_streamed": e2e_ws,
            "cpu_baseline": cpu,
            "gpu_launches": step.launches_per_step * args.steps,
            **extra,
            "gpu_launches_dsv3": extra_launches,
        }))
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
