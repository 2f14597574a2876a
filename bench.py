"""Benchmark of the block-scaled 4-bit hot path on GB300.

Headline workload (one step): the decode qmv sweep over a hidden-5120 dense
stack -- 64 layers x (q, k, v, o 5120x5120; gate, up 17408x5120; down
5120x17408) -- against NVFP4 weights (group 16, E4M3 scales, fp32 global
scale), bf16 activations, fp32 accumulation.  `value` is weight-bytes GB/s
(packed codes + block scales) with weights resident in HBM; the stack (13.4 GB)
is far larger than L2, so no flush is needed between steps.  The same line
reports the other formats (MXFP4, affine-4 g64), the activation quantize, the
NVFP4 prefill qqmm and the MXFP4 MoE gather_qmm as components.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs an independent replica (the path has no
exchange step), timings are max-reduced, value = all ranks' bytes / time.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_scaled_fp4_fp_gb300 import synth  # noqa: E402

METRIC = "FP4 qmv weight GB/s (% of HBM peak); NVFP4 qqmm TFLOPS (% of FP4 peak)"
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / bf16 tensor ratio on GB300


# --------------------------------------------------------------------------- utils
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()  # start timing once sampling runs, so the samples cover the timed region
            while not self.lines and time.time() - t0 < 3.0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash(name: str) -> str:
    p = os.path.join(ROOT, "block_scaled_fp4_fp_gb300", "csrc", name)
    h = hashlib.sha256()
    for f in (p, os.path.join(ROOT, "block_scaled_fp4_fp_gb300", "csrc", "common.cuh")):
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_file: str, key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(key)
    if not d or d.get("source_hash") != kernel_source_hash(kernel_file):
        return None
    return d.get("dram_bytes_per_launch")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


@contextlib.contextmanager
def nvtx(name: str):
    """An NVTX range around a host-side region (visible to Nsight tools); a
    no-op where NVTX is unavailable."""
    pushed = False
    try:
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:
        pass
    try:
        yield
    finally:
        if pushed:
            try:
                torch.cuda.nvtx.range_pop()
            except Exception:
                pass


def device_info(index: int) -> dict:
    """Name, SM count and compute capability of the GPU, and the host's cores."""
    info = {"host_cores": os.cpu_count()}
    try:
        p = torch.cuda.get_device_properties(index)
        info.update(name=p.name, sm_count=p.multi_processor_count, cc=f"{p.major}.{p.minor}")
    except Exception as e:  # the line is still printed without them
        info["error"] = type(e).__name__
    return info


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the process group (the slowest
    rank's time is the job's); the values unchanged without one."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_gbs(bytes_per_rank: int, ms: float, world: int) -> float:
    """Whole-job weight throughput: every rank streams its own replica of the
    stack (replicas, weak scaling), so the job moves world x bytes per step."""
    return world * bytes_per_rank / ms / 1e6


# ----------------------------------------------------------------- decode stack
layer_groups = synth.layer_groups


class DecodeStack:
    """64-layer weight stack in one format, weights resident on the device."""

    def __init__(self, B, mode: int, layers: int, device, layout: str = "split", qx: bool = False,
                 prefetch: bool = False):
        """layout "split": one matrix per projection, 7 GEMVs a layer.  "fused":
        the projections that multiply the same x stored as one matrix, as serving
        engines store them -- q|k|v as [3*5120, 5120] and gate|up as [2*17408,
        5120] -- so a layer is 4 GEMVs (qkv, o, gate_up, down) over the same
        weights (each output slice is that projection's y).  "fused_qkv": only
        q|k|v fused, 5 GEMVs a layer.  qx: the quantized-activation route (qqmv:
        x quantized and dequantized inside each GEMV; NVFP4 with a static
        activation global scale, as a calibrated checkpoint carries one).  prefetch:
        every launch goes through qmv_grouped naming the next launch's weights, which
        it warms in L2 once its own weight loads are issued."""
        self.B, self.mode, self.layers, self.qx = B, mode, layers, qx
        self.mats = []
        self.bytes = 0
        # "split_grouped": one matrix per projection, as "split", but the projections
        # that multiply the same x (q, k, v; gate, up) run as one qmv_grouped launch
        self.grouped = layout == "split_grouped"
        self.launch_groups = []
        for l in range(layers):
            for N, K, grp in layer_groups("split" if self.grouped else layout):
                self.mats.append(self._make(l, N, K, grp, device))
            base = len(self.mats) - len(layer_groups("split" if self.grouped else layout))
            if self.grouped:
                self.launch_groups += [[base + p for p in g] for _, _, g in layer_groups("fused")]
            else:
                self.launch_groups += [[i] for i in range(base, len(self.mats))]
        self.x = {K: synth.decode_x(K, device=device) for K in {k for _, _, k in synth.LAYER_PROJECTIONS}}
        self.gs_x = {K: (B.fp4_amax_global_scale(v) if qx and mode == B.MODE_NVFP4 else None)
                     for K, v in self.x.items()}
        self.y = [torch.empty((m["N"],), dtype=torch.bfloat16, device=device) for m in self.mats]
        self.prefetch = prefetch and not qx
        self.mgroups = [B.matrix_group([(self.mats[i]["q"], self.mats[i]["s"], self.mats[i]["b"], self.mats[i]["gs"])
                                        for i in g]) for g in self.launch_groups]

    def _make(self, layer, N, K, grp, device):
        B = self.B
        if self.mode == B.MODE_AFFINE:
            # uniform synthetic codes (the library has no affine quantizer), seeded by the group's first projection
            q, s, b = synth.affine_synthetic(N, K, synth.layer_seed(layer, grp[0]), device=device)
            nbytes = q.numel() * 4 + s.numel() * 2 + b.numel() * 2
            self.bytes += nbytes
            return {"N": N, "K": K, "q": q, "s": s, "b": b, "gs": None, "bytes": nbytes}
        w = synth.decode_weight(layer, grp, device=device)
        gs = B.fp4_amax_global_scale(w) if self.mode == B.MODE_NVFP4 else None
        q, s = B.fp4_quantize(w, self.mode, global_scale=gs)
        del w
        nbytes = q.numel() * 4 + s.numel()
        self.bytes += nbytes
        return {"N": N, "K": K, "q": q, "s": s, "b": None, "gs": gs, "bytes": nbytes}

    def step(self, stream=None):
        B = self.B
        if self.prefetch:
            n = len(self.launch_groups)
            for j, g in enumerate(self.launch_groups):
                B.qmv_grouped(self.x[self.mats[g[0]]["K"]], self.mgroups[j], mode=self.mode,
                              ys=[self.y[i] for i in g], stream=stream, prefetch_next=self.mgroups[(j + 1) % n])
            return
        if self.grouped:
            for g in self.launch_groups:
                ms = [self.mats[i] for i in g]
                if len(g) == 1:
                    m = ms[0]
                    B.qmv(self.x[m["K"]], m["q"], m["s"], m["b"], m["gs"], mode=self.mode, y=self.y[g[0]],
                          stream=stream)
                else:
                    B.qmv_grouped(self.x[ms[0]["K"]], [(m["q"], m["s"], m["b"], m["gs"]) for m in ms],
                                  mode=self.mode, ys=[self.y[i] for i in g], stream=stream)
            return
        for m, y in zip(self.mats, self.y):
            if self.qx:
                B.qqmv(self.x[m["K"]], m["q"], m["s"], self.gs_x[m["K"]], m["gs"], mode=self.mode, y=y, stream=stream)
            else:
                B.qmv(self.x[m["K"]], m["q"], m["s"], m["b"], m["gs"], mode=self.mode, y=y, stream=stream)

    def stream_step(self, stream=None):
        """The same weights moved as the tensor-core GEMV moves them, with no
        compute (NVFP4 only): the launch-and-stream ceiling of that kernel shape."""
        for m in self.mats:
            self.B.fp4_debug_stream_weights(m["q"], m["s"], stream=stream)

    @property
    def launches(self):
        return len(self.launch_groups)


WORKLOAD = ("decode qmv over a 64-layer hidden-5120 stack (q,k,v,o 5120x5120; gate,up 17408x5120; "
            "down 5120x17408), NVFP4 g16 weights, bf16 x, one token")
LAYOUT = ("q|k|v stored as one [15360, 5120] matrix and gate|up as one [34816, 5120] matrix (they "
          "multiply the same x): 4 GEMVs a layer, the same weights and outputs; one matrix per "
          "projection (7 GEMVs a layer) is components.decode_qmv.nvfp4; every launch names the next "
          "launch's weights (qmv_grouped's L2 prefetch hint)")


def time_graph(graph, steps, warmup, stream):
    # replay() launches on the current stream: make it the stream the events see
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn(stream)  # warm (loads kernels, sets attributes) outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn(stream)
    torch.cuda.synchronize()
    return g


# ------------------------------------------------------------------ components
def bench_quantize(B, device, reps=200, windows=3):
    """Activation quantize 4096x5120 (0.1 % outliers x50), tiled scales; 4 rotating
    inputs.  A launch takes ~10 us, so one short window is noisy (+-5 % between
    windows): the median of `windows` windows of `reps` back-to-back launches."""
    xs = [synth.activations_with_outliers(4096, 5120, seed=i, outlier_seed=100 + i, device=device) for i in range(4)]
    res = {}
    for mode, name, sr in ((B.MODE_NVFP4, "nvfp4", False), (B.MODE_MXFP4, "mxfp4", False),
                           (B.MODE_NVFP4, "nvfp4_stochastic", True), (B.MODE_MXFP4, "mxfp4_stochastic", True)):
        gss = [B.fp4_amax_global_scale(x) if mode == B.MODE_NVFP4 else None for x in xs]
        outs = [B.fp4_quantize(x, mode, global_scale=g, layout=B.SCALES_TILED) for x, g in zip(xs, gss)]

        def call(r):
            i = r % 4
            if sr:  # a fresh offset per call: no random word is reused
                B.fp4_quantize_sr(xs[i], mode, 1234, r * (4096 * 5120 // 4), global_scale=gss[i],
                                  layout=B.SCALES_TILED, xq=outs[i][0], scales=outs[i][1])
            else:
                B.fp4_quantize(xs[i], mode, global_scale=gss[i], layout=B.SCALES_TILED, xq=outs[i][0],
                               scales=outs[i][1])

        for i in range(4):  # warm-up
            call(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        per = []
        for wdw in range(max(1, windows)):
            e0.record()
            for r in range(reps):  # back-to-back launches over 4 rotating inputs (4 x 84 MB > L2)
                call(wdw * reps + r)
            e1.record()
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / reps if reps else float("nan"))
        ms = statistics.median(per)
        nbytes = 4096 * 5120 * 2 + 4096 * 5120 // 2 + outs[0][1].numel()
        res[name] = {"ms": ms, "GB/s": nbytes / ms / 1e6, "bytes": nbytes, "windows_ms": per}
    return res


def bench_qqmm(B, device, Ms=(1024, 2048, 8192), reps=20):
    N, K = 17408, 5120
    w = synth.bf16_normal((N, K), 0.02, seed=1, device=device)
    gw = B.fp4_amax_global_scale(w)
    wq, ws_w = B.fp4_quantize(w, B.MODE_NVFP4, global_scale=gw, layout=B.SCALES_TILED)
    del w
    res = {}
    for M in Ms:
        x = synth.bf16_normal((M, K), 1.0, seed=2, device=device)
        gx = B.fp4_amax_global_scale(x)
        xq, xs = B.fp4_quantize(x, B.MODE_NVFP4, global_scale=gx, layout=B.SCALES_TILED)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        for _ in range(3):  # warm-up
            B.qqmm(xq, xs, wq, ws_w, gx, gw, mode=B.MODE_NVFP4, out=out)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            B.qqmm(xq, xs, wq, ws_w, gx, gw, mode=B.MODE_NVFP4, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps if reps else float("nan")
        # the activation's global scale and quantization (tiled scales) in front of each GEMM
        e0.record()
        for _ in range(reps):
            B.fp4_amax_global_scale_noalloc(x, gs_out=gx)
            B.fp4_quantize(x, B.MODE_NVFP4, global_scale=gx, layout=B.SCALES_TILED, xq=xq, scales=xs)
            B.qqmm(xq, xs, wq, ws_w, gx, gw, mode=B.MODE_NVFP4, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms_q = e0.elapsed_time(e1) / reps if reps else float("nan")
        # the same three steps fused into one cooperative launch (qqmm_quantize_x)
        ws = B.qqmm_quantize_x_workspace(M, K, B.MODE_NVFP4)
        for _ in range(3):
            B.qqmm_quantize_x(x, wq, ws_w, ws, None, gw, mode=B.MODE_NVFP4, out=out)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            B.qqmm_quantize_x(x, wq, ws_w, ws, None, gw, mode=B.MODE_NVFP4, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms_f = e0.elapsed_time(e1) / reps if reps else float("nan")
        flops = 2.0 * M * N * K
        # algorithmic bytes: both operands' codes and E4M3 scales once, the bf16 output once
        nbytes = (M + N) * K // 2 + (M + N) * (K // 16) + 2 * M * N
        res[f"M{M}"] = {"ms": ms, "TFLOP/s": flops / ms / 1e9, "flops": flops, "bytes": nbytes,
                        "GB/s": nbytes / ms / 1e6,
                        "ms_with_x_quantize": ms_q, "TFLOP/s_with_x_quantize": flops / ms_q / 1e9,
                        "ms_fused_x_quantize": ms_f, "TFLOP/s_fused_x_quantize": flops / ms_f / 1e9}
        del x, xq, xs, out
    return res


def bench_qqmm_mxfp4(B, device, Ms=(1024, 2048, 8192), reps=20):
    """The same GEMM with MXFP4 operands (E8M0 scales per 32, no global scale)."""
    N, K = 17408, 5120
    w = synth.bf16_normal((N, K), 0.02, seed=1, device=device)
    wq, ws_w = B.fp4_quantize(w, B.MODE_MXFP4, layout=B.SCALES_TILED)
    del w
    res = {}
    for M in Ms:
        x = synth.bf16_normal((M, K), 1.0, seed=2, device=device)
        xq, xs = B.fp4_quantize(x, B.MODE_MXFP4, layout=B.SCALES_TILED)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        for _ in range(3):  # warm-up
            B.qqmm(xq, xs, wq, ws_w, None, None, mode=B.MODE_MXFP4, out=out)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            B.qqmm(xq, xs, wq, ws_w, None, None, mode=B.MODE_MXFP4, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps if reps else float("nan")
        flops = 2.0 * M * N * K
        res[f"M{M}"] = {"ms": ms, "TFLOP/s": flops / ms / 1e9, "flops": flops}
        del x, xq, xs, out
    return res


def bench_qqmm_cublaslt(B, device, Ms=(1024, 2048, 8192), reps=20):
    """Side comparison only: the same FP4 GEMMs through cuBLASLt's block-scaled
    kernels (torch._scaled_mm on float4_e2m1fn_x2 operands), fed the very bytes
    this library's quantizer wrote: packed codes as [rows, K/2] bytes and the
    128x4-tiled scales as E4M3 (NVFP4) or E8M0 (MXFP4) bytes.  The output, times
    alpha, is compared with qqmm's, which also checks that the nibble order and
    the tile layout read the same way in both.  Never on the product path."""
    N, K = 17408, 5120
    f4 = getattr(torch, "float4_e2m1fn_x2", None)
    e8 = getattr(torch, "float8_e8m0fnu", None)
    if f4 is None:
        return {"unavailable": "this PyTorch has no float4_e2m1fn_x2"}
    res = {}
    for name, mode, sdt in (("nvfp4", B.MODE_NVFP4, torch.float8_e4m3fn), ("mxfp4", B.MODE_MXFP4, e8)):
        if sdt is None:
            res[name] = {"unavailable": "this PyTorch has no float8_e8m0fnu"}
            continue
        w = synth.bf16_normal((N, K), 0.02, seed=1, device=device)
        gw = B.fp4_amax_global_scale(w) if mode == B.MODE_NVFP4 else None
        wq, ws_w = B.fp4_quantize(w, mode, global_scale=gw, layout=B.SCALES_TILED)
        del w
        bt = wq.view(torch.uint8).view(f4).t()  # [K/2, N], column-major
        sb = ws_w.view(torch.uint8).view(sdt).reshape(-1)
        for M in Ms:
            x = synth.bf16_normal((M, K), 1.0, seed=2, device=device)
            gx = B.fp4_amax_global_scale(x) if mode == B.MODE_NVFP4 else None
            xq, xs = B.fp4_quantize(x, mode, global_scale=gx, layout=B.SCALES_TILED)
            a = xq.view(torch.uint8).view(f4)
            sa = xs.view(torch.uint8).view(sdt).reshape(-1)
            rec = {}
            try:
                ref = torch._scaled_mm(a, bt, sa, sb, out_dtype=torch.bfloat16)
                ours = B.qqmm(xq, xs, wq, ws_w, gx, gw, mode=mode)
                alpha = (gx * gw).item() if gx is not None else 1.0
                d = ref.float() * alpha - ours.float()
                rec["rel_l2_vs_qqmm"] = (d.norm() / ours.float().norm()).item()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                for _ in range(3):
                    torch._scaled_mm(a, bt, sa, sb, out_dtype=torch.bfloat16, out=ref)
                ts = []
                for _ in range(3):
                    e0.record()
                    for _ in range(reps):
                        torch._scaled_mm(a, bt, sa, sb, out_dtype=torch.bfloat16, out=ref)
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) / max(reps, 1))
                ms = statistics.median(ts)
                rec["ms"] = ms
                rec["TFLOP/s"] = 2.0 * M * N * K / ms / 1e9
            except Exception as e:  # cuBLASLt or this PyTorch may not take the shape or format
                rec = {"unavailable": f"{type(e).__name__}: {str(e).splitlines()[0][:200]}"}
            res.setdefault(name, {})[f"M{M}"] = rec
            del x, xq, xs, a, sa
        del wq, ws_w, bt, sb
    return res


def bench_qmm(B, device, Ms=(1024, 2048, 8192), reps=20):
    """Dense W4A16 prefill GEMM M x 17408 x 5120: bf16 activations against NVFP4
    (group 16, global scale) and affine-4 group-64 weights."""
    N, K = 17408, 5120
    res = {}
    for name, mode in (("nvfp4", B.MODE_NVFP4), ("affine_g64", B.MODE_AFFINE)):
        if mode == B.MODE_AFFINE:
            wq, ws, wb = synth.affine_synthetic(N, K, seed=1, device=device)
            gw = None
        else:
            w = synth.bf16_normal((N, K), 0.02, seed=1, device=device)
            gw = B.fp4_amax_global_scale(w)
            wq, ws = B.fp4_quantize(w, mode, global_scale=gw)
            wb = None
            del w
        for M in Ms:
            x = synth.bf16_normal((M, K), 1.0, seed=2, device=device)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
            for _ in range(3):  # warm-up
                B.qmm(x, wq, ws, wb, gw, mode=mode, out=out)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                B.qmm(x, wq, ws, wb, gw, mode=mode, out=out)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps if reps else float("nan")
            flops = 2.0 * M * N * K
            res.setdefault(name, {})[f"M{M}"] = {"ms": ms, "TFLOP/s": flops / ms / 1e9, "flops": flops}
            del x, out
    return res


def bench_gather(B, device, reps=20):
    """MoE grouped W4A16 GEMMs of 2048 tokens, 32 experts, top-4: gate/up
    (N 5760, K 2880) on the routed token rows, and down (N 2880, K 2880) on a
    fresh [8192, 2880] input already in routed order."""
    tokens, E, topk, H, F = 2048, 32, 4, 2880, 5760
    lhs, rhs = synth.moe_routing(tokens, E, topk, seed=0)
    rhs_d = torch.from_numpy(rhs).to(device)
    res = {}
    for name, N, K, x, lhs_rows in (
            ("gate_up", F, H, synth.bf16_normal((tokens, H), 1.0, seed=1, device=device), lhs),
            ("down", H, H, synth.bf16_normal((len(lhs), H), 1.0, seed=3, device=device),
             np.arange(len(lhs), dtype=np.int32))):
        lhs_d = torch.from_numpy(lhs_rows).to(device)
        w = synth.bf16_normal((E * N, K), 0.02, seed=2 if name == "gate_up" else 4, device=device)
        q, s = B.fp4_quantize(w, B.MODE_MXFP4)
        del w
        q3, s3 = q.view(E, N, K // 8), s.view(E, N, K // 32)
        out = torch.empty((len(lhs), N), dtype=torch.bfloat16, device=device)
        for _ in range(3):  # warm-up
            B.gather_qmm(x, lhs_d, rhs_d, q3, s3, out=out)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            B.gather_qmm(x, lhs_d, rhs_d, q3, s3, out=out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps if reps else float("nan")
        flops = 2.0 * len(lhs) * N * K
        res[name] = {"ms": ms, "TFLOP/s": flops / ms / 1e9, "flops": flops}
        if name == "gate_up":
            # the routed activations first put in routing order (gather_rows), then the
            # grouped GEMM on consecutive rows (whole tiles by TMA): both launches timed
            xr = torch.empty((len(lhs), K), dtype=torch.bfloat16, device=device)
            ident = torch.arange(len(lhs), dtype=torch.int32, device=device)

            def two_step():
                B.gather_rows(x, lhs_d, out=xr)
                B.gather_qmm(xr, ident, rhs_d, q3, s3, out=out)

            for _ in range(3):
                two_step()
            torch.cuda.synchronize()
            e0.record()
            for _ in range(reps):
                two_step()
            e1.record()
            torch.cuda.synchronize()
            ms2 = e0.elapsed_time(e1) / reps if reps else float("nan")
            res[name].update({"ms_routed_order": ms2, "TFLOP/s_routed_order": flops / ms2 / 1e9})
            del xr
        del x, q, s, out
    return res


# ------------------------------------------------------------------ CPU oracle
def oracle_layer_setup():
    """Layer 0's seven NVFP4 projections for the oracle: weights generated on the
    CPU and quantized by the oracle (untimed), and the two activation vectors."""
    import oracle
    mats = []
    for p, (name, N, K) in enumerate(synth.LAYER_PROJECTIONS):
        w = synth.to_u16(synth.bf16_normal((N, K), 0.02, seed=synth.layer_seed(0, p)))
        gs = oracle.global_scale(w)
        q, s = oracle.nvfp4_quantize(w, gs)
        mats.append((q, s, gs, K))
    xs = {K: synth.to_u16(synth.bf16_normal((K,), 1.0, seed=7 + K)) for K in (synth.HIDDEN, synth.MLP)}
    return mats, xs


def oracle_layer_time(mats, xs):
    """Oracle qmv over the seven projections; returns (seconds, weight bytes)."""
    import oracle
    nbytes = sum(q.nbytes + s.nbytes for q, s, _, _ in mats)
    t0 = time.perf_counter()
    for q, s, gs, K in mats:
        oracle.qmv(xs[K], q, s, None, oracle.MODE_NVFP4, 16, gs)
    return time.perf_counter() - t0, nbytes


def cpu_component_baselines():
    """The oracle timed on the host cores for the components, on bounded samples
    (each labelled): quantize in full, qqmm on a 4-row slice, MoE gate/up on 8
    routed rows of one expert."""
    import oracle
    res = {}
    x = synth.to_u16(synth.activations_with_outliers(4096, 5120, seed=0, outlier_seed=100))
    gs = oracle.global_scale(x)
    t0 = time.perf_counter()
    oracle.nvfp4_quantize(x, gs)
    t = time.perf_counter() - t0
    res["quantize_4096x5120"] = {"value": (x.nbytes + x.nbytes // 4 + x.nbytes // 32) / t / 1e9, "unit": "GB/s",
                                 "sample": "4096x5120 NVFP4 in full"}
    w = synth.to_u16(synth.bf16_normal((1024, 5120), 0.02, seed=1))  # 1024 of the 17408 weight rows
    gw = oracle.global_scale(w)
    wq, ws = oracle.nvfp4_quantize(w, gw)
    xs = synth.to_u16(synth.bf16_normal((32, 5120), 1.0, seed=2))
    gx = oracle.global_scale(xs)
    xq, sx = oracle.nvfp4_quantize(xs, gx)
    t0 = time.perf_counter()
    oracle.qqmm(xq, sx, wq, ws, oracle.MODE_NVFP4, alpha=gx * gw)
    t = time.perf_counter() - t0
    res["qqmm_nvfp4_Mx17408x5120"] = {"value": 2.0 * 32 * 1024 * 5120 / t / 1e12, "unit": "TFLOP/s",
                                      "sample": "32 rows x 1024 columns of M x 17408 x 5120"}
    del w, wq, ws
    lhs, rhs = synth.moe_routing(2048, 32, 4, seed=0)
    e0 = int(rhs[0])
    sel = np.nonzero(rhs == e0)[0][:8]
    xg = synth.to_u16(synth.bf16_normal((2048, 2880), 1.0, seed=1))
    we = synth.to_u16(synth.bf16_normal((5760, 2880), 0.02, seed=2))
    q, sc = oracle.mxfp4_quantize(we)
    t0 = time.perf_counter()
    oracle.gather_qmm(xg, lhs[sel], np.zeros(len(sel), np.int32), q.reshape(1, 5760, 360), sc.reshape(1, 5760, 90),
                      None, oracle.MODE_MXFP4, 32)
    t = time.perf_counter() - t0
    res["gather_qmm_mxfp4_moe"] = {"value": 2.0 * len(sel) * 5760 * 2880 / t / 1e12, "unit": "TFLOP/s",
                                   "sample": f"gate/up, {len(sel)} routed rows of one expert"}
    for v in res.values():
        v.update({"kind": "oracle", "cores": oracle.num_threads()})
    return res


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ---------------------------------------------------------- profiling cases
def run_case(args):
    """Small single-kernel workloads for ncu captures (a few launches each)."""
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp4_fp_gb300 import binding as B
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    B.fp4_init(0)
    c = args.case
    if c.startswith("qmv_") or c.startswith("qqmv_"):
        layout = "fused" if c.endswith("_fused") else "split"
        base = c.replace("_fused", "").replace("qqmv_", "qmv_")
        mode = {"qmv_nvfp4": B.MODE_NVFP4, "qmv_mxfp4": B.MODE_MXFP4, "qmv_affine": B.MODE_AFFINE}[base]
        # 4 layers: 0.84 GB of weights, well above L2
        qx = c.startswith("qqmv_")
        stack = DecodeStack(B, mode, 4, dev, layout=layout, qx=qx, prefetch=not qx)
        for _ in range(3):
            stack.step()
    elif c.startswith("qqmm_m"):
        bench_qqmm(B, dev, Ms=(int(c[len("qqmm_m"):]),), reps=1)
    elif c.startswith("cublaslt_m"):
        print(json.dumps(bench_qqmm_cublaslt(B, dev, Ms=(int(c[len("cublaslt_m"):]),), reps=5)))
    elif c == "quantize":
        bench_quantize(B, dev, reps=2)
    elif c.startswith("qqmm_fused_m"):
        M, N, K = int(c[len("qqmm_fused_m"):]), 17408, 5120
        w = synth.bf16_normal((N, K), 0.02, seed=1, device=dev)
        gw = B.fp4_amax_global_scale(w)
        wq, sw = B.fp4_quantize(w, B.MODE_NVFP4, global_scale=gw, layout=B.SCALES_TILED)
        x = synth.bf16_normal((M, K), 1.0, seed=2, device=dev)
        ws = B.qqmm_quantize_x_workspace(M, K, B.MODE_NVFP4)
        for _ in range(2):
            B.qqmm_quantize_x(x, wq, sw, ws, None, gw, mode=B.MODE_NVFP4)
    elif c == "gather":
        bench_gather(B, dev, reps=1)
    elif c.startswith("qmm_m"):
        bench_qmm(B, dev, Ms=(int(c[len("qmm_m"):]),), reps=1)
    torch.cuda.synchronize()
    st = B.fp4_check_device_error()
    print(json.dumps({"case": c, "status": B.status_string(st)}))
    if st != B.FP4_OK:
        sys.exit(3)


# ------------------------------------------------------------------------ main
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    mats, xs = oracle_layer_setup()
    times, nbytes = [], 0
    for i in range(args.warmup + args.steps):
        t, nbytes = oracle_layer_time(mats, xs)
        if i >= args.warmup:
            times.append(t)
    sec = statistics.median(times)
    v = nbytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "layout": LAYOUT,
                   "l2": "inputs larger than L2 per step"},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": "layer 0 of 64: q,k,v,o,gate,up,down NVFP4 GEMV in the C oracle (fp64)"},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp4_fp_gb300 import binding as B
    B.fp4_init(local)
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device)

    # the headline: NVFP4 weights in the fused layout (4 GEMVs a layer); the
    # per-projection layout and the other formats are components
    # (name, format, layout, quantized x, next-launch prefetch hints); the FP4 layouts run as
    # a serving loop runs them: every launch names the next launch's weights
    modes = [("nvfp4_fused", B.MODE_NVFP4, "fused", False, True)] + (
        [] if args.quick else [("nvfp4_fused_no_prefetch", B.MODE_NVFP4, "fused", False, False),
                               ("nvfp4", B.MODE_NVFP4, "split", False, True),
                               ("nvfp4_grouped", B.MODE_NVFP4, "split_grouped", False, True),
                               ("mxfp4_fused", B.MODE_MXFP4, "fused", False, True),
                               ("mxfp4", B.MODE_MXFP4, "split", False, True),
                               ("mxfp4_grouped", B.MODE_MXFP4, "split_grouped", False, True),
                               ("affine_g64", B.MODE_AFFINE, "split", False, True),
                               ("affine_g64_grouped", B.MODE_AFFINE, "split_grouped", False, True),
                               ("affine_g64_fused", B.MODE_AFFINE, "fused", False, True),
                               ("nvfp4_fused_quantized_x", B.MODE_NVFP4, "fused", True, False),
                               ("mxfp4_fused_quantized_x", B.MODE_MXFP4, "fused", True, False)])
    results = {}
    headline = None
    for name, mode, layout, qx, pf in modes:
        stack = DecodeStack(B, mode, args.layers, device, layout=layout, qx=qx, prefetch=pf)
        graph = capture(stack.step, stream)
        if name == "nvfp4_fused":
            with ClockSampler(local) as clk, nvtx(f"decode {name}"):
                if ws > 1:
                    torch.distributed.barrier()
                ms = time_graph(graph, args.steps, args.warmup, stream)
            clocks = clk.summary()
            headline = (stack, graph, ms)
        else:
            with nvtx(f"decode {name}"):
                ms = time_graph(graph, args.steps, args.warmup, stream)
        results[name] = {"ms_per_step": ms, "GB/s": stack.bytes / ms / 1e6, "bytes_per_step": stack.bytes,
                         "frac_of_hbm": stack.bytes / ms / 1e6 / peaks["hbm_gbs"],
                         "launches_per_step": stack.launches, "layout": layout,
                         "entry_point": ("qqmv (x quantized inside the GEMV)" if qx else
                                         "qmv_grouped, each launch naming the next one's weights (L2 prefetch hint)"
                                         if pf else "qmv"),
                         "prefetch_next": pf}
        if name != "nvfp4_fused":
            del stack, graph
            torch.cuda.empty_cache()

    stack, graph, ms = headline
    # the same launches streaming the same weights with no compute
    sgraph = capture(stack.stream_step, stream)
    with nvtx("stream ceiling"):
        stream_ms = time_graph(sgraph, args.steps, args.warmup, stream)
    del sgraph
    # e2e: pinned host activations in, every projection's output back, through the C ABI
    hx = {k: v.cpu().pin_memory() for k, v in stack.x.items()}
    hy = torch.empty((sum(m["N"] for m in stack.mats),), dtype=torch.bfloat16).pin_memory()
    dy = torch.empty_like(hy, device=device)
    ys = []
    off = 0
    for m in stack.mats:
        ys.append(dy[off:off + m["N"]])
        off += m["N"]
    stack.y = ys

    def e2e_step(s):
        for k in stack.x:
            stack.x[k].copy_(hx[k], non_blocking=True)
        stack.step(s)
        hy.copy_(dy, non_blocking=True)

    g2 = capture(e2e_step, stream)
    with nvtx("e2e"):
        e2e_ms = time_graph(g2, args.steps, args.warmup, stream)
    h2d = sum(v.numel() * 2 for v in hx.values())
    d2h = hy.numel() * 2

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], device)
    value = job_gbs(stack.bytes, ms, ws)
    comps = {"decode_qmv": results}
    if not args.quick and rank == 0:
        comps["quantize_4096x5120"] = bench_quantize(B, device)
        comps["qqmm_nvfp4_Mx17408x5120"] = bench_qqmm(B, device)
        comps["qqmm_mxfp4_Mx17408x5120"] = bench_qqmm_mxfp4(B, device)
        comps["qqmm_cublaslt_side_comparison"] = bench_qqmm_cublaslt(B, device)
        comps["gather_qmm_mxfp4_moe"] = bench_gather(B, device)
        comps["qmm_w4a16_Mx17408x5120"] = bench_qmm(B, device)
        for fmt in comps["qmm_w4a16_Mx17408x5120"].values():
            for v in fmt.values():
                v["frac_of_bf16_peak"] = v["TFLOP/s"] / peaks["bf16_tflops"]
        fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
        for k, v in comps["qqmm_nvfp4_Mx17408x5120"].items():
            v["frac_of_fp4_peak"] = v["TFLOP/s"] / fp4_peak
            v["frac_of_hbm"] = v["GB/s"] / peaks["hbm_gbs"]
        for k, v in comps["qqmm_mxfp4_Mx17408x5120"].items():
            v["frac_of_fp4_peak"] = v["TFLOP/s"] / fp4_peak
        for fmt, d in comps["qqmm_cublaslt_side_comparison"].items():
            ours = comps["qqmm_nvfp4_Mx17408x5120" if fmt == "nvfp4" else "qqmm_mxfp4_Mx17408x5120"]
            for M, v in (d.items() if isinstance(d, dict) else ()):
                if isinstance(v, dict) and "TFLOP/s" in v and M in ours:
                    v["qqmm_over_cublaslt"] = ours[M]["TFLOP/s"] / v["TFLOP/s"]
        for k, v in comps["gather_qmm_mxfp4_moe"].items():
            v["frac_of_bf16_peak"] = v["TFLOP/s"] / peaks["bf16_tflops"]
            if "TFLOP/s_routed_order" in v:
                v["frac_of_bf16_peak_routed_order"] = v["TFLOP/s_routed_order"] / peaks["bf16_tflops"]
        for k, v in comps["quantize_4096x5120"].items():
            v["frac_of_hbm"] = v["GB/s"] / peaks["hbm_gbs"]
        if ws == 1 and not args.no_cpu:
            import oracle
            oracle.build()
            comps["cpu_oracle"] = cpu_component_baselines()

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        sec, nb = oracle_layer_time(*oracle_layer_setup())
        cpu = {"value": nb / sec / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": "layer 0 of 64 (q,k,v,o,gate,up,down), NVFP4 GEMV in the C oracle, fp64, weights "
                         "quantized by the oracle (untimed)"}
    if rank == 0:
        per_launch_bytes = stack.bytes / stack.launches
        achieved = stack.bytes / ms / 1e6
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp4-e2m1 x bf16, f32 acc", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layout": LAYOUT,
                       "layers": args.layers, "weight_bytes_per_step": stack.bytes,
                       "tokens_per_s": 1e3 / ms, "l2": "inputs larger than L2 (13.4 GB stack)",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": committed_traffic("qmv_tc.cu", "qmv_tc_nvfp4_decode_layer"),
                         "kernel": "qmv_tc_kernel (tcgen05 NVFP4 GEMV)", "bytes_per_launch": per_launch_bytes,
                         "peak_src": peaks["src"] + " hbm_gbs",
                         "stream_ceiling": {"GB/s": stack.bytes / stream_ms / 1e6, "ms_per_step": stream_ms,
                                            "frac_of_peak": stack.bytes / stream_ms / 1e6 / peaks["hbm_gbs"],
                                            "qmv_frac_of_ceiling": stream_ms / ms,
                                            "what": f"fp4_debug_stream_weights over the same {stack.launches} "
                                                    "launches: the same plan, TMA boxes, ring and launch, no "
                                                    "compute"}},
            "cpu_baseline": cpu,
            "e2e": {"value": job_gbs(stack.bytes, e2e_ms, ws), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": stack.launches * args.steps,
            "clocks": clocks,
            "device": device_info(local),
            "components": comps,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=synth.LAYERS)
    ap.add_argument("--quick", action="store_true", help="headline only (no other formats/components)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--case", default=None,
                    help="profiling case: qmv_nvfp4[_fused]|qmv_mxfp4[_fused]|qmv_affine[_fused]|qqmv_nvfp4_fused|"
                         "qqmm_m<M>|qqmm_fused_m<M>|qmm_m<M>|cublaslt_m<M>|quantize|gather")
    args = ap.parse_args()
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
