"""Benchmark of the block-float decode-in-kernel matmul on GB300.

One step = one decode token through the projections of an 80-layer dense
model over MXFP4 weights at M = 1: per layer fused QKV 10240x8192, FFN
up/gate 57344x8192 and down 8192x28672, each through mx_qmv (240 launches,
33.5 GB of distinct weights per step).  The headline value is weight GB/s
(codes + block scales streamed per second); the same run also reports the
2048 x 2048 GEMV, M = 4, the MoE decode layer (128 experts, top-8: gate-up,
SwiGLU, down, combine) in tokens/s, the MXFP8 / NVFP4 format sweep and the
prefill GEMM in TFLOP/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Inputs are seeded synthetic tensors (see
gemm_decode_register_gb300/synth.py).  Every layer's 419 MB of weights is
larger than the 129 MB L2, so each step streams them from HBM.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 qmv weight GB/s (% of HBM peak); MoE tok/s; prefill qmm TFLOP/s"
DENSE = [("qkv", 10240, 8192, 1), ("up_gate", 57344, 8192, 2), ("down", 8192, 28672, 3)]
LAYERS = 80


def workload(layers):
    return (f"decode step of a {layers}-layer dense model's projections, MXFP4 weights (E2M1 codes, E8M0 "
            "scale per 32, exponents uniform in [118,132]), bf16 activations N(0,1), M=1 token: per layer "
            "fused QKV 10240x8192 + FFN up/gate 57344x8192 + down 8192x28672, one mx_qmv launch each, "
            "distinct weights per layer")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1939.6)), \
            float(d.get("bf16_tflops_sustained", 1726.2)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


QMV_SOURCES = ["gemm_decode_register_gb300/csrc/mx_qmv_stream.cu", "gemm_decode_register_gb300/csrc/mx_qmv_core.cuh",
               "gemm_decode_register_gb300/csrc/mx_common.cuh", "gemm_decode_register_gb300/csrc/mx_internal.h",
               "gemm_decode_register_gb300/csrc/mx_stream.cuh"]
TRAFFIC_PROFILE = "profiles/qmv_decode_layer_traffic.md"


def measured_traffic():
    """DRAM bytes per qmv launch from the committed ncu summary, or None when
    the kernel sources changed since that capture."""
    import hashlib

    try:
        h = hashlib.sha256()
        for f in QMV_SOURCES:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        fields = {}
        with open(os.path.join(ROOT, TRAFFIC_PROFILE)) as fh:
            for line in fh:
                if ":" in line and line.strip().split(":")[0] in ("source_sha256", "traffic_bytes_per_launch"):
                    k, v = line.strip().split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256") != h.hexdigest():
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def max_over_ranks(dist, value, device=None):
    """The largest value across ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((t, float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ helpers

def upload(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1)).cuda()


def bf16_dev(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def pinned_bf16(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).reshape(-1).view(np.int16)).view(torch.bfloat16).pin_memory()


def graph_of(torch, fn, reps=1):
    """Capture reps calls of fn (our kernel launches) into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm (first-call set-up happens outside the capture)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    torch.cuda.synchronize()
    return g


def time_region(torch, fn, iters, stream):
    """Average seconds per call of fn over iters calls (CUDA events)."""
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record(stream)
    for _ in range(iters):
        fn()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / 1e3 / iters


# ------------------------------------------------------------------ our arm

def run_ours(args, rank, world, dist):
    import torch

    from gemm_decode_register_gb300 import build as b
    from gemm_decode_register_gb300 import ops, synth

    b.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    hbm, bf16_burst, bf16_sust, peak_kind = peaks()
    F4 = synth.FMT_MXFP4

    # ---- the step: one decode token through LAYERS dense layers (distinct
    # weights, drawn on the device: 33.5 GB at 80 layers)
    L = args.layers
    projs = []
    xoff = yoff = 0
    for li in range(L):
        for name, N, K, seed in DENSE:
            codes, scales = synth.weights_device(F4, N, K, 100000 * (li + 1) + seed, dev, exp_lo=118, exp_hi=132)
            projs.append({"name": name, "N": N, "K": K, "codes": codes, "scales": scales, "xo": xoff, "yo": yoff,
                          "bytes": codes.numel() + scales.numel()})
            xoff += K
            yoff += N
    # every projection's activation row and output row live in one buffer each,
    # so that a step's inputs arrive in one host-to-device copy and its outputs
    # leave in one device-to-host copy
    x_host = pinned_bf16(torch, synth.activations(1, xoff, 100))
    x_dev = x_host.to(dev)
    y_dev = torch.empty(yoff, dtype=torch.float32, device=dev)
    y_host = torch.empty(yoff, dtype=torch.float32).pin_memory()
    for P in projs:
        P["x"] = x_dev[P["xo"]:P["xo"] + P["K"]].view(1, P["K"])
        P["y"] = y_dev[P["yo"]:P["yo"] + P["N"]].view(1, P["N"])
    wbytes = sum(P["bytes"] for P in projs)
    alg_bytes = sum(P["bytes"] + P["K"] * 2 + P["N"] * 4 for P in projs)
    n_launch = len(projs)

    def launches():
        for P in projs:
            ops.qmv(F4, P["codes"], P["scales"], P["x"], P["N"], y=P["y"])

    # the step's launches captured once in a CUDA graph (programmatic dependent
    # launch lets each overlap the previous one's tail); each of layer 0's
    # projections alone as well, for the per-projection figures
    step_graph = graph_of(torch, launches)
    for P in projs[:3]:
        P["graph"] = graph_of(torch, lambda P=P: ops.qmv(F4, P["codes"], P["scales"], P["x"], P["N"], y=P["y"]))
    for _ in range(max(3, args.warmup)):
        step_graph.replay()
    torch.cuda.synchronize()

    clk = ClockSampler(dev.index)
    clk.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clk.mark("t0")
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step_graph.replay()
    t_end.record(stream)
    torch.cuda.synchronize()
    clk.mark("t1")
    elapsed = max_over_ranks(dist, t_start.elapsed_time(t_end) / 1e3, dev)
    # The timed region holds only this library's qmv kernel, n_launch launches
    # per step back to back: its average launch duration there is the region's
    # time over n_launch * steps launches.
    launch_avg_s = elapsed / (n_launch * args.steps)
    # each projection of layer 0 alone (one-launch graphs, events between
    # them, the three in turn so that none stays in L2): per-projection figures
    nl = min(args.steps * 10, 300)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nl)]
    for i in range(nl):
        ev[i][0].record(stream)
        for j, P in enumerate(projs[:3]):
            P["graph"].replay()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    launch_s = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(nl)) / 1e3 / nl for j in range(3)]
    value = world * wbytes * args.steps / elapsed / 1e9
    ms_per_step = elapsed / args.steps * 1e3
    achieved = alg_bytes / n_launch / launch_avg_s / 1e9
    per_proj = {P["name"]: round(P["bytes"] / s / 1e9, 1) for P, s in zip(projs[:3], launch_s)}

    # ---- end to end through the public API with host buffers: every step
    # copies the step's activations in from pinned host memory, issues the
    # n_launch mx_qmv calls through the binding (no graph) and copies the
    # outputs back; the same with the captured step for comparison
    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        launches()
        y_host.copy_(y_dev, non_blocking=True)

    def e2e_step_graph():
        x_dev.copy_(x_host, non_blocking=True)
        step_graph.replay()
        y_host.copy_(y_dev, non_blocking=True)

    for _ in range(3):
        e2e_step()
    e2e_t = time_region(torch, e2e_step, args.steps, stream)
    for _ in range(3):
        e2e_step_graph()
    e2e_tg = time_region(torch, e2e_step_graph, args.steps, stream)
    clk.stop()
    h2d = xoff * 2
    d2h = yoff * 4

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16xf16->f32 (decoded MXFP4 x scaled bf16)", "data": "synthetic",
        "config": {"workload": workload(L), "layers": L, "launches_per_step": n_launch,
                   "weight_bytes_per_step": wbytes,
                   "l2": f"inputs larger than L2: {wbytes / 1e9:.1f} GB of distinct weights streamed per step "
                         "(L2 129 MB)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "per_projection_gbs": per_proj,
                   "per_projection_note": "layer 0's projections, each as a one-launch graph, in turn, outside the "
                                          "timed region"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": measured_traffic(),
                     "kernel": "qmv_stream_kernel<MXFP4, MC=1>", "peak_source": peak_kind,
                     "bytes_per_launch": round(alg_bytes / n_launch),
                     "launch_us": round(launch_avg_s * 1e6, 3),
                     "launch_timing": f"CUDA events over the timed region: its time over the {n_launch} launches "
                                      "per step",
                     "traffic_source": TRAFFIC_PROFILE},
        "e2e": {"value": round(world * wbytes / e2e_t / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_t * 1e3, 4),
                "note": f"weights resident (model state); each step copies the {n_launch} activation rows in "
                        f"from pinned host memory (one copy), calls mx_qmv {n_launch} times through the Python "
                        "binding (ctypes, no graph) and copies the outputs back (one copy)",
                "graph_value": round(world * wbytes / e2e_tg / 1e9, 1),
                "graph_note": "the same with the step's launches replayed from one captured CUDA graph"},
        "gpu_launches": n_launch * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_extras and rank == 0:
        out["extras"] = extras(torch, ops, synth, dev, stream, hbm, bf16_burst, bf16_sust, args)
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(synth, budget_s=args.cpu_seconds)
    return out


def extras(torch, ops, synth, dev, stream, hbm, bf16_burst, bf16_sust, args):
    """Secondary measurements of the other workloads (same run)."""
    res = {}
    F4, F8, NV = synth.FMT_MXFP4, synth.FMT_MXFP8, synth.FMT_NVFP4
    iters = max(20, args.extra_iters)
    res.update(extras_config0(torch, ops, synth, dev, stream, hbm, iters))

    # M = 4 dense layer
    mats = []
    for name, N, K, seed in DENSE:
        codes, scales = synth.weights(F4, N, K, seed, exp_lo=118, exp_hi=132)
        mats.append((N, K, upload(torch, codes), upload(torch, scales),
                     bf16_dev(torch, synth.activations(4, K, 200 + seed)), codes.nbytes + scales.nbytes))
    wb = sum(m[5] for m in mats)
    for M in (1, 4):
        def f(M=M):
            for N, K, c, s, x, _ in mats:
                ops.qmv(F4, c, s, x.reshape(-1)[: M * K].view(M, K), N)
        g = graph_of(torch, f)
        t = time_region(torch, g.replay, iters, stream)
        res[f"dense_layer_M{M}"] = {"gbs": round(wb / t / 1e9, 1), "frac_hbm": round(wb / t / 1e9 / hbm, 4),
                                   "us": round(t * 1e6, 2), "tok_s": round(M / t, 1)}
    del mats

    # each projection alone: a graph over distinct weight copies (more than 4x L2 in all), per launch
    L2 = 129 * 2 ** 20
    for name, N, K, seed in DENSE:
        wbytes = N * K // 2 + N * K // 32
        copies = max(2, -(-4 * L2 // wbytes))
        ws = [synth.weights_device(F4, N, K, 1000 * seed + i, dev) for i in range(copies)]
        for M in (1, 4):
            x = bf16_dev(torch, synth.activations(M, K, 400 + seed)).view(M, K)
            y = torch.empty((M, N), dtype=torch.float32, device=dev)

            def fp(ws=ws, x=x, y=y, N=N):
                for c, s in ws:
                    ops.qmv(F4, c, s, x, N, y=y)
            g = graph_of(torch, fp)
            t = time_region(torch, g.replay, max(5, iters // 4), stream) / copies
            res[f"projection_{name}_M{M}"] = {"us": round(t * 1e6, 2), "gbs": round(wbytes / t / 1e9, 1),
                                             "frac_hbm": round(wbytes / t / 1e9 / hbm, 4), "copies": copies}
        del ws

    # format sweep on the FFN up/gate shape
    N, K = 57344, 8192
    for fmt, fname, seed in ((F4, "mxfp4", 2), (F8, "mxfp8", 6), (NV, "nvfp4", 7)):
        codes, scales = synth.weights(fmt, N, K, seed, exp_lo=118, exp_hi=132)
        c, s = upload(torch, codes), upload(torch, scales)
        wbf = codes.nbytes + scales.nbytes
        for M in (1, 4):
            x = bf16_dev(torch, synth.activations(M, K, 300 + M)).view(M, K)
            g = graph_of(torch, lambda: ops.qmv(fmt, c, s, x, N))
            t = time_region(torch, g.replay, iters, stream)  # 250-480 MB per call: larger than L2
            res[f"sweep_{fname}_M{M}"] = {"gbs": round(wbf / t / 1e9, 1),
                                         "frac_hbm": round(wbf / t / 1e9 / hbm, 4), "us": round(t * 1e6, 2)}
        del c, s

    # MoE decode layer: 128 experts, top-8, hidden 2048, expert intermediate 768
    E, topk, H, I = 128, 8, 2048, 768
    c1, s1 = synth.weights(F4, 2 * I, H, 40, E=E, exp_lo=118, exp_hi=132)
    c2, s2 = synth.weights(F4, H, I, 41, E=E, exp_lo=118, exp_hi=132)
    per_expert = (c1.nbytes + s1.nbytes + c2.nbytes + s2.nbytes) // E
    d1, e1, d2, e2 = (upload(torch, a) for a in (c1, s1, c2, s2))
    for T in (1, 4):
        nsets = 64
        ids_all = [synth.expert_ids(T, E, topk, 1000 * T + i) for i in range(nsets)]
        uniq = [len(np.unique(a)) for a in ids_all]
        ids_dev = [torch.from_numpy(a).cuda() for a in ids_all]
        ids_flat = [a.reshape(-1, 1).contiguous() for a in ids_dev]
        r = torch.from_numpy(synth.router_weights(T, topk, 77)).cuda()
        x = bf16_dev(torch, synth.activations(T, H, 78)).view(T, H)
        gu = torch.empty((T, topk, 2 * I), dtype=torch.float32, device=dev)
        h = torch.empty((T * topk, I), dtype=torch.bfloat16, device=dev)
        yd = torch.empty((T * topk, 1, H), dtype=torch.float32, device=dev)
        out = torch.empty((T, H), dtype=torch.float32, device=dev)

        def layer(i):
            ops.moe_qmv(F4, d1, e1, x, ids_dev[i], E, 2 * I, y=gu)
            ops.swiglu(gu, I, h=h)
            ops.moe_qmv(F4, d2, e2, h, ids_flat[i], E, H, y=yd)
            ops.moe_combine(yd, r, out=out)

        def gemv_only(i):
            ops.moe_qmv(F4, d1, e1, x, ids_dev[i], E, 2 * I, y=gu)
            ops.moe_qmv(F4, d2, e2, h, ids_flat[i], E, H, y=yd)

        hf = torch.empty((T, topk, I), dtype=torch.bfloat16, device=dev)

        def fused(i):
            ops.moe_gate_up_swiglu(F4, d1, e1, x, ids_dev[i], E, I, h=hf)
            ops.moe_down_combine(F4, d2, e2, hf.view(T * topk, I), ids_dev[i], r, E, H, out=out)

        # one CUDA graph per variant holds nsets layers, each with its own routing
        graphs = {}
        for name, fn in (("layer", layer), ("gemv", gemv_only), ("fused", fused)):
            def allsets(fn=fn):
                for i in range(nsets):
                    fn(i)
            graphs[name] = graph_of(torch, allsets)
        reps = max(4, iters // 8)
        t = time_region(torch, graphs["layer"].replay, reps, stream) / nsets
        t2 = time_region(torch, graphs["gemv"].replay, reps, stream) / nsets
        tf = time_region(torch, graphs["fused"].replay, reps, stream) / nsets
        ub = statistics.mean(uniq) * per_expert
        res[f"moe_layer_T{T}"] = {"tok_s": round(T / tf, 1), "us_layer": round(tf * 1e6, 2),
                                  "unique_expert_gbs": round(ub / tf / 1e9, 1),
                                  "frac_hbm": round(ub / tf / 1e9 / hbm, 4),
                                  "path": "mx_moe_gate_up_swiglu + mx_moe_down_combine (2 launches)",
                                  "tok_s_unfused": round(T / t, 1), "us_layer_unfused": round(t * 1e6, 2),
                                  "us_gemv_only_unfused": round(t2 * 1e6, 2),
                                  "mean_unique_experts": round(statistics.mean(uniq), 2),
                                  "note": "CUDA graph of 64 layers, each with freshly drawn expert ids"}
    del d1, e1, d2, e2

    # prefill qmm
    if args.no_qmm:
        return res
    try:
        for N, K, seed in ((28672, 8192, 8), (8192, 28672, 9)):
            M = 4096
            codes, scales = synth.weights(F4, N, K, seed, exp_lo=118, exp_hi=132)
            c, s = upload(torch, codes), upload(torch, scales)
            X = torch.randn(M, K, device=dev).to(torch.bfloat16)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            g = graph_of(torch, lambda: ops.qmm(F4, c, s, X, N, Y=Y))
            t = time_region(torch, g.replay, max(5, iters // 4), stream)
            tf = 2.0 * M * N * K / t / 1e12
            res[f"prefill_qmm_{N}x{K}"] = {"tflops": round(tf, 1), "frac_bf16_burst": round(tf / bf16_burst, 4),
                                          "frac_bf16_sustained": round(tf / bf16_sust, 4),
                                          "ms": round(t * 1e3, 3)}
            del c, s, X, Y
    except Exception as exc:  # reported, not hidden
        res["prefill_qmm"] = {"error": str(exc).splitlines()[0][:200]}
    for name, fn in (("moe_prefill", extras_moe_prefill), ("crossover_upgate", extras_crossover),
                     ("quantize", extras_quantize), ("qmm_qx", extras_qmm_qx)):
        try:
            res.update(fn(torch, ops, synth, dev, stream, bf16_burst, iters))
        except Exception as exc:  # reported, not hidden
            res[name] = {"error": str(exc).splitlines()[0][:200]}
    return res


def extras_config0(torch, ops, synth, dev, stream, hbm, iters):
    """The 2048 x 2048 MXFP4 GEMV at M = 1 (E8M0 exponents in [120, 130]):
    256 distinct weight copies (570 MB, over four times the 129 MB L2)
    rotated through one CUDA graph, so every call streams its 2.2 MB from
    HBM; the same calls issued one by one through the binding; and the
    latency of one call from issue to completion (host clock)."""
    F4 = synth.FMT_MXFP4
    N = K = 2048
    copies = 256
    ws = [synth.weights_device(F4, N, K, 7000 + i, dev, exp_lo=120, exp_hi=130) for i in range(copies)]
    wb = ws[0][0].numel() + ws[0][1].numel()
    x = bf16_dev(torch, synth.activations(1, K, 1000)).view(1, K)
    y = torch.empty((1, N), dtype=torch.float32, device=dev)

    def calls():
        for c, s in ws:
            ops.qmv(F4, c, s, x, N, y=y)

    g = graph_of(torch, calls)
    reps = max(5, iters // 10)
    t = time_region(torch, g.replay, reps, stream) / copies
    calls()
    t_ng = time_region(torch, calls, reps, stream) / copies
    lat = []
    for i in range(60):
        c, s = ws[i % copies]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ops.qmv(F4, c, s, x, N, y=y)
        torch.cuda.synchronize()
        lat.append(time.perf_counter() - t0)
    lat = statistics.median(lat[10:])
    gbs = wb / t / 1e9
    return {"config0_gemv_2048": {
        "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4), "frac_hbm_nominal_8tbs": round(gbs / 8000.0, 4),
        "us_per_call_graph": round(t * 1e6, 3), "us_per_call_no_graph": round(t_ng * 1e6, 3),
        "single_call_latency_us": round(lat * 1e6, 1), "weight_bytes": wb,
        "note": f"{copies} distinct weight copies ({copies * wb / 1e6:.0f} MB, > 4x L2) rotated in one graph; "
                "no-graph: the same calls issued one by one; latency: one call issue to completion"}}


def extras_moe_prefill(torch, ops, synth, dev, stream, bf16_burst, iters):
    """Expert-batched MoE prefill: 4096 tokens, top-8 of 128 experts, hidden
    2048, expert intermediate 768 (weights 321 MB, larger than L2)."""
    res = {}
    F4 = synth.FMT_MXFP4
    E, topk, H, I, T = 128, 8, 2048, 768, 4096
    c1, s1 = synth.weights(F4, 2 * I, H, 40, E=E, exp_lo=118, exp_hi=132)
    c2, s2 = synth.weights(F4, H, I, 41, E=E, exp_lo=118, exp_hi=132)
    d1, e1, d2, e2 = (upload(torch, a) for a in (c1, s1, c2, s2))
    ids = torch.from_numpy(synth.expert_ids(T, E, topk, 500)).cuda()
    r = torch.from_numpy(synth.router_weights(T, topk, 501)).cuda()
    x = bf16_dev(torch, synth.activations(T, H, 502)).view(T, H)
    h = bf16_dev(torch, synth.activations(T * topk, I, 503)).view(T * topk, I)
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws = ops.moe_ffn_prefill_workspace(T, E, topk, H, I, device=dev)
    n = max(5, iters // 10)
    g = graph_of(torch, lambda: ops.moe_ffn_prefill(F4, d1, e1, d2, e2, x, ids, r, E, I, out=out, workspace=ws))
    t = time_region(torch, g.replay, n, stream)
    fl = 2.0 * T * topk * (2 * I * H + H * I)
    res["moe_prefill_ffn_T4096"] = {"tok_s": round(T / t, 1), "us": round(t * 1e6, 1),
                                    "tflops": round(fl / t / 1e12, 1),
                                    "frac_bf16_burst": round(fl / t / 1e12 / bf16_burst, 4),
                                    "path": "mx_moe_ffn_prefill: routing (count, scan, place + gather), grouped "
                                            "gate-up GEMM + SwiGLU, grouped down GEMM, combine (6 launches)"}
    for name, d, e, xin, idv, N, K in (("gate_up", d1, e1, x, ids, 2 * I, H),
                                       ("down", d2, e2, h, ids.reshape(-1, 1).contiguous(), H, I)):
        Tq, tk = idv.shape
        y = torch.empty((Tq, tk, N), dtype=torch.bfloat16, device=dev)
        wsq = torch.empty(ops.load().mx_moe_qmm_workspace_size(Tq, E, tk, K), dtype=torch.uint8, device=dev)
        gq = graph_of(torch, lambda: ops.moe_qmm(F4, d, e, xin, idv, E, N, y=y, workspace=wsq))
        tq = time_region(torch, gq.replay, n, stream)
        flq = 2.0 * Tq * tk * N * K
        res[f"moe_prefill_qmm_{name}"] = {"tflops": round(flq / tq / 1e12, 1), "us": round(tq * 1e6, 1),
                                          "frac_bf16_burst": round(flq / tq / 1e12 / bf16_burst, 4),
                                          "path": "mx_moe_qmm: count, scan, place + gather, grouped GEMM "
                                                  "(4 launches)"}
        del y, wsq
    return res


def extras_qmm_qx(torch, ops, synth, dev, stream, bf16_burst, iters):
    """The tensor pipe's dense rate per MMA kind (mx_mma_peak, zero operands),
    and the prefill GEMM over quantised activations (mx_quantize, then the
    block-scaled mx_qmm_qx) on the 4096 x 28672 x 8192 up projection in each
    format, next to the bf16-activation GEMM (mx_qmm) on the same weights:
    TFLOP/s, fraction of the measured peak of the GEMM's own MMA kind, and the
    relative L2 distance between the two products (a property of quantising
    the activations, not an error of either kernel)."""
    res = {}
    kinds = ("bf16", "e4m3", "mxfp8", "mxfp4", "nvfp4")
    peaks = {k: round(ops.mma_peak_tflops(k), 1) for k in kinds}
    filled = {k: round(ops.mma_peak_tflops(k, filled=True), 1) for k in kinds}
    res["tensor_peaks_tflops"] = dict(peaks, note="mx_mma_peak: one CTA per SM issuing 128x256xK tcgen05.mma "
                                                  "(cta_group::1) on zero operands, best of 5")
    res["tensor_peaks_filled_tflops"] = dict(filled, note="the same on random finite operands (unit block "
                                                          "scales), the same shared-memory tiles every MMA: the "
                                                          "data does not slow the tensor pipe")
    probes = {}
    for k in ("mxfp8", "mxfp4"):
        for name, fl in (("rotate", ops.PEAK_ROTATE), ("rotate_smem_stores", ops.PEAK_ROTATE | ops.PEAK_SMEM_STORES),
                         ("rotate_tmem_stores", ops.PEAK_ROTATE | ops.PEAK_TMEM_STORES)):
            probes[f"{k}_{name}"] = round(ops.mma_peak_tflops(k, reps=3, filled=True, flags=fl), 1)
    res["tensor_peak_probes_tflops"] = dict(probes, note="random operands; MMAs rotating through 4 (3) stages of "
                                                         "48 KB; meanwhile 3 warps store 16-byte vectors into "
                                                         "shared memory, or into tensor memory, at full rate")
    M, N, K = 4096, 28672, 8192
    X = bf16_dev(torch, synth.activations(M, K, 58)).view(M, K)
    n = max(5, iters // 10)
    for fmt, fname, kind in ((synth.FMT_MXFP4, "mxfp4", "mxfp4"), (synth.FMT_MXFP8, "mxfp8", "mxfp8"),
                             (synth.FMT_NVFP4, "nvfp4", "nvfp4")):
        codes, scales = synth.weights_device(fmt, N, K, 8, dev, exp_lo=118, exp_hi=132)
        xc, xs = ops.quantize(fmt, X)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        Yb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        tg = time_region(torch, graph_of(torch, lambda: ops.qmm_qx(fmt, codes, scales, xc, xs, M, N, K, Y=Y)).replay,
                         n, stream)
        tq = time_region(torch, graph_of(torch, lambda: ops.quantize(fmt, X, xc, xs)).replay, n, stream)
        tb = time_region(torch, graph_of(torch, lambda: ops.qmm(fmt, codes, scales, X, N, Y=Yb)).replay, n, stream)
        ops.qmm_qx(fmt, codes, scales, xc, xs, M, N, K, Y=Y)
        ops.qmm(fmt, codes, scales, X, N, Y=Yb)
        dist = (torch.linalg.vector_norm((Y.float() - Yb.float())) / torch.linalg.vector_norm(Yb.float())).item()
        fl = 2.0 * M * N * K
        res[f"prefill_qmm_qx_{fname}_28672x8192"] = {
            "tflops": round(fl / tg / 1e12, 1), "ms": round(tg * 1e3, 3),
            "frac_measured_peak": round(fl / tg / 1e12 / peaks[kind], 4), "peak_kind": kind,
            "frac_filled_peak": round(fl / tg / 1e12 / filled[kind], 4),
            "quantize_us": round(tq * 1e6, 1), "tflops_with_quantize": round(fl / (tg + tq) / 1e12, 1),
            "bf16_path_tflops": round(fl / tb / 1e12, 1), "bf16_path_ms": round(tb * 1e3, 3),
            "rel_l2_vs_bf16_activations": round(dist, 4),
            "path": "mx_quantize (X to the weights' format) + mx_qmm_qx (block-scaled tcgen05.mma), against "
                    "mx_qmm (in-SMEM decode to bf16 + tcgen05 bf16 MMA)"}
        del codes, scales, xc, xs, Y, Yb
    return res


def extras_quantize(torch, ops, synth, dev, stream, bf16_burst, iters):
    """On-device quantisation of the prefill activations (4096 x 8192 bf16,
    67 MB in: larger than L2): bytes read and written per second."""
    res = {}
    M, K = 4096, 8192
    x = bf16_dev(torch, synth.activations(M, K, 600)).view(M, K)
    hbm = peaks()[0]
    for fmt, name in ((synth.FMT_MXFP4, "mxfp4"), (synth.FMT_MXFP8, "mxfp8"), (synth.FMT_NVFP4, "nvfp4")):
        codes, scales = ops.quantize(fmt, x)
        t = time_region(torch, graph_of(torch, lambda: ops.quantize(fmt, x, codes, scales)).replay,
                        max(10, iters // 4), stream)
        nbytes = 2 * M * K + codes.numel() + scales.numel() + (2 * M * K if fmt == synth.FMT_NVFP4 else 0)
        res[f"quantize_{name}"] = {"us": round(t * 1e6, 2), "gbs": round(nbytes / t / 1e9, 1),
                                   "frac_hbm": round(nbytes / t / 1e9 / hbm, 4),
                                   "bytes": nbytes,
                                   "note": "x read once (NVFP4: twice, tensor maximum then blocks) + codes and "
                                           "scales written"}
    return res


def extras_crossover(torch, ops, synth, dev, stream, bf16_burst, iters):
    """Decode GEMV against prefill GEMM as the token count grows, on the FFN
    up/gate shape (57344 x 8192, 250 MB of weights: larger than L2)."""
    F4 = synth.FMT_MXFP4
    N, K = 57344, 8192
    codes, scales = synth.weights(F4, N, K, 2, exp_lo=118, exp_hi=132)
    c, s = upload(torch, codes), upload(torch, scales)
    rows, first = {}, None
    n = max(3, iters // 20)
    for M in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        X = bf16_dev(torch, synth.activations(M, K, 400 + M)).view(M, K)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        tv = time_region(torch, graph_of(torch, lambda: ops.qmv(F4, c, s, X, N, y=y)).replay, n, stream)
        tm = time_region(torch, graph_of(torch, lambda: ops.qmm(F4, c, s, X, N, Y=Y)).replay, n, stream)
        rows[str(M)] = {"qmv_us": round(tv * 1e6, 1), "qmm_us": round(tm * 1e6, 1)}
        if first is None and tm < tv:
            first = M
    return {"crossover_upgate": {"rows": rows, "qmm_faster_from_M": first,
                                 "note": "qmv: 8 tokens per pass over the weights; qmm: 256-row pair tiles"}}


# ------------------------------------------------------------------ oracle

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(synth, budget_s=12.0):
    """The oracle (plain C, fp64) on a bounded sample of the same projections
    -- the leading rows of each, growing until about budget_s / 2 of host
    time per leg -- first single-threaded, then with the rows cut into
    ranges over every core of the process's affinity set; value in the same
    unit (weight GB/s), the all-core figure as the value."""
    import oracle

    orc = oracle.get()
    F4 = synth.FMT_MXFP4
    data = []
    for name, N, K, seed in DENSE:
        codes, scales = synth.weights(F4, N, K, seed, exp_lo=118, exp_hi=132)
        data.append((name, N, K, codes, scales, synth.activations(1, K, 100 + seed)))
    cores = host_cores()

    def leg(nthreads, start_rows):
        rows, spent, done_bytes, done_rows = start_rows, 0.0, 0, 0
        while spent < budget_s / 2:
            for name, N, K, codes, scales, x in data:
                r = np.arange(min(rows, N))
                t0 = time.perf_counter()
                if nthreads == 1:
                    orc.qmv_rows(F4, codes, scales, x, 1, N, K, r)
                else:
                    orc.qmv_rows_mt(F4, codes, scales, x, 1, N, K, r, nthreads)
                spent += time.perf_counter() - t0
                done_bytes += r.size * (K // 2 + K // 32)
                done_rows += r.size
            rows = min(2 * rows, 57344)
        return done_bytes / spent / 1e9, done_rows, spent

    v1, r1, s1 = leg(1, 16)
    vn, rn, sn = leg(cores, 16 * cores)
    return {"value": round(vn, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{rn} weight rows (leading rows of QKV, up/gate, down) on {cores} threads, {sn:.1f} s",
            "single_core": {"value": round(v1, 4), "cores": 1,
                            "sample": f"{r1} weight rows, {s1:.1f} s single-threaded"}}


def run_reference(args, rank, world):
    """The oracle arm: the same metric on the host cores (the oracle's rows
    cut into ranges over every core of the process's affinity set), each
    step a bounded sample of the projections (leading rows of each)."""
    from gemm_decode_register_gb300 import synth
    import oracle

    if rank != 0:
        return None
    orc = oracle.get()
    F4 = synth.FMT_MXFP4
    data = []
    for name, N, K, seed in DENSE:
        codes, scales = synth.weights(F4, N, K, seed, exp_lo=118, exp_hi=132)
        data.append((N, K, codes, scales, synth.activations(1, K, 100 + seed)))
    cores = host_cores()
    rows = args.ref_rows * cores

    def step():
        b = 0
        for N, K, codes, scales, x in data:
            r = min(rows, N)
            orc.qmv_rows_mt(F4, codes, scales, x, 1, N, K, np.arange(r), cores)
            b += r * (K // 2 + K // 32)
        return b

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    tot = 0
    for _ in range(args.steps):
        tot += step()
    el = time.perf_counter() - t0
    v = tot / el / 1e9
    sample = f"{rows} leading rows of each projection per step, {cores} host threads"
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": workload(args.layers), "sample": sample},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


CASES = {
    # name: (kind, fmt, M or T, N, K)
    "qmv_tiny_m1": ("qmv", 0, 1, 304, 8192),
    "qmv_2k_m1": ("qmv", 0, 1, 2048, 8192),
    "qmv_tinydown_m1": ("qmv", 0, 1, 304, 28672),
    "qmv_qkv_m1": ("qmv", 0, 1, 10240, 8192),
    "qmv_20k_m1": ("qmv", 0, 1, 20480, 8192),
    "qmv_upgate_m1": ("qmv", 0, 1, 57344, 8192),
    "qmv_upgate_m4": ("qmv", 0, 4, 57344, 8192),
    "qmv_down_m1": ("qmv", 0, 1, 8192, 28672),
    "qmv_down_m4": ("qmv", 0, 4, 8192, 28672),
    "qmv_mxfp8_m1": ("qmv", 1, 1, 57344, 8192),
    "qmv_nvfp4_m1": ("qmv", 2, 1, 57344, 8192),
    "moe_gateup_t4": ("moe", 0, 4, 1536, 2048),
    "moe_ffn_t1": ("moe_ffn", 0, 1, 2048, 768),  # fused gate-up/SwiGLU + down/combine, hidden 2048, I 768
    "moe_ffn_t4": ("moe_ffn", 0, 4, 2048, 768),
    "qmm_up": ("qmm", 0, 4096, 28672, 8192),
    "qmm_down": ("qmm", 0, 4096, 8192, 28672),
    "qmm_small": ("qmm", 0, 1024, 4096, 4096),
    "qmm_mid": ("qmm", 0, 2048, 8192, 4096),
    # block-scaled GEMM over quantised activations, 4096 x 28672 x 8192 (and a small case for captures)
    "qmm_qx_up_mxfp4": ("qmm_qx", 0, 4096, 28672, 8192),
    "qmm_qx_up_mxfp8": ("qmm_qx", 1, 4096, 28672, 8192),
    "qmm_qx_up_nvfp4": ("qmm_qx", 2, 4096, 28672, 8192),
    "qmm_qx_mid_mxfp4": ("qmm_qx", 0, 2048, 8192, 4096),
    # expert-batched MoE FFN prefill: 4096 tokens, top-8 of 128 experts, hidden 2048, I 768
    "moe_prefill_ffn_t4096": ("moe_prefill", 0, 4096, 2048, 768),
    # on-device quantisation of 4096 x 8192 bf16 activations
    "quantize_mxfp4": ("quantize", 0, 4096, 0, 8192),
    "quantize_mxfp8": ("quantize", 1, 4096, 0, 8192),
    "quantize_nvfp4": ("quantize", 2, 4096, 0, 8192),
}


def run_case(args):
    """One kernel configuration for a few launches (profiling runs); prints
    the mean launch time."""
    import torch

    from gemm_decode_register_gb300 import build as b
    from gemm_decode_register_gb300 import ops, synth

    b.build()
    kind, fmt, M, N, K = CASES[args.case]
    stream = torch.cuda.current_stream()
    if kind == "quantize":
        x = bf16_dev(torch, synth.activations(M, K, 600)).view(M, K)
        qc, qs = ops.quantize(fmt, x)
        f = lambda: ops.quantize(fmt, x, qc, qs)  # noqa: E731
        wb = 2 * M * K + qc.numel() + qs.numel()
    elif kind == "moe_prefill":
        E, topk, H, I = 128, 8, N, K
        c1, s1 = synth.weights(fmt, 2 * I, H, 40, E=E)
        c2, s2 = synth.weights(fmt, H, I, 41, E=E)
        d1, e1, d2, e2 = (upload(torch, a) for a in (c1, s1, c2, s2))
        ids = torch.from_numpy(synth.expert_ids(M, E, topk, 5)).cuda()
        r = torch.from_numpy(synth.router_weights(M, topk, 7)).cuda()
        x = bf16_dev(torch, synth.activations(M, H, 6)).view(M, H)
        out = torch.empty((M, H), dtype=torch.float32, device="cuda")
        ws = ops.moe_ffn_prefill_workspace(M, E, topk, H, I)
        f = lambda: ops.moe_ffn_prefill(fmt, d1, e1, d2, e2, x, ids, r, E, I, out=out, workspace=ws)  # noqa: E731
        wb = c1.nbytes + s1.nbytes + c2.nbytes + s2.nbytes
    elif kind == "qmm_qx":
        codes, scales = synth.weights_device(fmt, N, K, 2, "cuda")
        X = bf16_dev(torch, synth.activations(M, K, 3)).view(M, K)
        xc, xs = ops.quantize(fmt, X)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        f = lambda: ops.qmm_qx(fmt, codes, scales, xc, xs, M, N, K, Y=Y)  # noqa: E731
        wb = codes.numel() + scales.numel()
    elif kind == "moe_ffn":
        E, topk, H, I = 128, 8, N, K
        c1, s1 = synth.weights(fmt, 2 * I, H, 40, E=E)
        c2, s2 = synth.weights(fmt, H, I, 41, E=E)
        d1, e1, d2, e2 = (upload(torch, a) for a in (c1, s1, c2, s2))
        ids = torch.from_numpy(synth.expert_ids(M, E, topk, 5)).cuda()
        r = torch.from_numpy(synth.router_weights(M, topk, 7)).cuda()
        x = bf16_dev(torch, synth.activations(M, H, 6)).view(M, H)
        hf = torch.empty((M * topk, I), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((M, H), dtype=torch.float32, device="cuda")

        def f():
            ops.moe_gate_up_swiglu(fmt, d1, e1, x, ids, E, I, h=hf)
            ops.moe_down_combine(fmt, d2, e2, hf, ids, r, E, H, out=out)
        nu = len(np.unique(ids.cpu().numpy()))
        wb = (c1.nbytes + s1.nbytes + c2.nbytes + s2.nbytes) / E * nu
    elif kind == "moe":
        E, topk = 128, 8
        codes, scales = synth.weights(fmt, N, K, 40, E=E)
        c, s = upload(torch, codes), upload(torch, scales)
        ids = torch.from_numpy(synth.expert_ids(M, E, topk, 5)).cuda()
        x = bf16_dev(torch, synth.activations(M, K, 6)).view(M, K)
        f = lambda: ops.moe_qmv(fmt, c, s, x, ids, E, N)  # noqa: E731
        wb = (codes.nbytes + scales.nbytes) / E * len(np.unique(ids.cpu().numpy()))
    else:
        codes, scales = synth.weights(fmt, N, K, 2, exp_lo=118, exp_hi=132)
        c, s = upload(torch, codes), upload(torch, scales)
        if kind == "qmv":
            x = bf16_dev(torch, synth.activations(M, K, 3)).view(M, K)
            f = lambda: ops.qmv(fmt, c, s, x, N)  # noqa: E731
        else:
            X = torch.randn(M, K, device="cuda").to(torch.bfloat16)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            f = lambda: ops.qmm(fmt, c, s, X, N, Y=Y)  # noqa: E731
        wb = codes.nbytes + scales.nbytes
    g = graph_of(torch, f)
    t = time_region(torch, g.replay, args.iters, stream)
    out = {"case": args.case, "iters": args.iters, "us": round(t * 1e6, 2),
           "weight_gbs": round(wb / t / 1e9, 1)}
    if kind in ("qmm", "qmm_qx"):
        out["tflops"] = round(2.0 * M * N * K / t / 1e12, 1)
    if kind == "moe_prefill":
        out["tflops"] = round(2.0 * M * 8 * 3 * N * K / t / 1e12, 1)
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-qmm", action="store_true")
    ap.add_argument("--extra-iters", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=256, help="reference arm: rows per projection per host thread")
    ap.add_argument("--layers", type=int, default=LAYERS, help="dense layers per step")
    ap.add_argument("--case", choices=sorted(CASES), help="time one kernel configuration only")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    out = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
