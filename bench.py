#!/usr/bin/env python3
"""Benchmark of the DFlash 2 draft tail on one GB300 (one rank per GPU).

A step is one pass of the whole hot path over one draft block: the fused tail
(top-16 -> pair scores -> walk) plus the 20 two-tap conv calls of the drafter
(5 layers x 4 insertion points).  The headline workload is the 4B-drafter
block at batch 1 (B=1, L=16, V=151,936, d=2560): value = microseconds per draft
block.  The batched serving block (B=64) is measured in the same run and
reported as blocks/s and HBM GB/s against the roofline.

Timing: CUDA events on the launching stream around each step (a CUDA graph
replay of the step), L2 flushed by a 256 MB write between steps, the GPU kept
busy with a sleep kernel while the host enqueues so no host latency is timed.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from draft_selection_gb300 import workloads as wl  # noqa: E402

HEADLINE = "drafter4b_l16"
BATCHED = "serving_b64"
METRIC = "µs per draft block at B=1; blocks/s and HBM GB/s vs roofline at B=64"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of an op's
# kernel, by (op, workload), from one ncu capture of the kernel as it is now;
# an op whose kernel changed since its capture has no entry and reports null.
NCU_TRAFFIC = {
    ("topk", "drafter4b_l16"): 4940544,
    ("topk", "serving_b64"): 314891008,
    ("conv", "drafter4b_l16"): 1766656,
    ("conv", "serving_b64"): 7283200,
    ("lmhead", "drafter4b_l16"): 781673728,
    ("lmhead", "serving_b64"): 786832384,
}


# --------------------------------------------------------------------------- bytes


def tail_bytes(w: wl.Workload, es: int) -> dict:
    """Algorithmic HBM bytes of one tail call, by kernel (each needed byte once)."""
    R = w.rows
    d = w.d
    cand_rows = w.B * (16 * w.L + 1)
    topk = R * w.V * es + R * 16 * 8
    select = cand_rows * d * 2 + 3 * 256 * d * 2 + R * d * 2 + w.B * 4 + R * 16 * 8 + R * 256 * 4
    walk = R * 16 * 4 + R * 16 * 4 + R * 4 + R * 16 * 4
    return {"topk": topk, "select": select, "walk": walk, "total": topk + select + walk}


def tail_tables_bytes(w: wl.Workload, es: int) -> int:
    """Algorithmic HBM bytes of one table tail: logits, the gathered table rows
    (A rows of the predecessors, B rows of the candidates, float32), hidden,
    W_H and the outputs."""
    R = w.rows
    rows_a = w.B * (16 * (w.L - 1) + 1)
    rows_b = w.B * 16 * w.L
    return (R * w.V * es + (rows_a + rows_b) * 256 * 4 + R * w.d * 2 + 256 * w.d * 2
            + w.B * 4 + R * 16 * 8 + R * 4 + R * 16 * 4)


def conv_bytes(w: wl.Workload) -> int:
    d = w.d
    return (2 * w.B * w.L * d * 2 + w.B * d * 2 + 2 * d * 4 + (2 * d // 16) * d * 2)


def select_flops(w: wl.Workload) -> float:
    return 2.0 * w.B * (16 * w.L + 1) * w.d * 512 + 2.0 * w.rows * w.d * 256


def conv_flops(w: wl.Workload) -> float:
    return 2.0 * w.B * w.L * w.d * (2 * w.d // 16)


# --------------------------------------------------------------------------- setup


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = os.path.join("/tmp", f"dfl2_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


class Staged:
    """Tensors packed into one device buffer (each slice 256-byte aligned), so
    that a step's inputs (or outputs) move between host and device in one copy."""

    def __init__(self, tensors, device):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        self.buf = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        self.views = []
        for t, o in zip(tensors, offs):
            nb = t.numel() * t.element_size()
            v = self.buf[o:o + nb].view(t.dtype).view(t.shape)
            v.copy_(t)
            self.views.append(v)
        self.nbytes = n


class Case:
    """One workload resident on the device, with its step as callables.  The
    step's inputs that change every step (logits, hidden states, verified
    tokens, Philox keys, and each conv call's x and x_prev) sit in one staging
    buffer, and its outputs (tokens, q) in another."""

    def __init__(self, w: wl.Workload, T: float, device):
        import draft_selection_gb300 as dfl2
        self.dfl2 = dfl2
        self.w, self.T = w, T
        gen_dev = "cpu" if w.B == 1 else device
        logits = wl.make_logits(w, gen_dev).to(device)
        inp = wl.make_tail_inputs(w, gen_dev)
        self.inp = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        seeds = torch.from_numpy(inp["seeds"].view(np.int64)).to(device)
        self.convs = []
        for k in range(w.conv_calls):
            c = wl.make_conv_inputs(w, k, gen_dev)
            c = {n: t.to(device) for n, t in c.items()}
            self.convs.append(c)
        per_step = [logits, self.inp["hidden"], self.inp["verified"], seeds]
        for c in self.convs:
            per_step += [c["x"], c["x_prev"]]
        self.staged_in = Staged(per_step, device)
        v = iter(self.staged_in.views)
        self.logits, self.inp["hidden"], self.inp["verified"], self.seeds = (
            next(v), next(v), next(v), next(v))
        for c in self.convs:
            c["x"], c["x_prev"] = next(v), next(v)
            c["y"] = torch.empty_like(c["x"])
        del per_step, logits
        # one conv workspace serves the block's calls: they run one after another
        n = dfl2.dfl2_conv2_workspace_size(w.B, w.L, w.d)
        self.conv_ws = dfl2.workspace(n, device) if n else None
        B, L = w.B, w.L
        outs = [torch.empty(B, L, dtype=torch.int32, device=device)]
        if T > 0:
            outs.append(torch.empty(B, L, 16, dtype=torch.float32, device=device))
        self.staged_out = Staged(outs, device)
        self.tokens = self.staged_out.views[0]
        self.q = self.staged_out.views[1] if T > 0 else None
        self.ws = dfl2.workspace(dfl2.dfl2_tail_workspace_size(B, L, w.V, w.d), device)
        self.idx = torch.empty(B, L, 16, dtype=torch.int32, device=device)
        self.val = torch.empty(B, L, 16, dtype=torch.float32, device=device)
        self.scores = torch.empty(B, L, 16, 16, dtype=torch.float32, device=device)
        self.ws_topk = dfl2.workspace(dfl2.dfl2_topk_workspace_size(B, L, w.V), device)
        self.ws_sel = dfl2.workspace(dfl2.dfl2_select_workspace_size(B, L, w.d), device)
        self.es = self.logits.element_size()

    def tail(self):
        i = self.inp
        self.dfl2.dfl2_tail(self.logits, i["verified"], i["hidden"], i["E"], i["W_A"], i["W_B"],
                            i["W_H"], self.T, self.seeds, 0, self.tokens, self.ws, q=self.q)

    def conv(self, k=0, plain=False):
        """One conv call through dfl2_conv2_ws (plain: dfl2_conv2, no workspace)."""
        c = self.convs[k]
        if plain:
            self.dfl2.dfl2_conv2(c["x"], c["x_prev"], c["base"], c["W_c"], c["y"])
        else:
            self.dfl2.dfl2_conv2_ws(c["x"], c["x_prev"], c["base"], c["W_c"], c["y"], self.conv_ws)

    def convs20(self):
        for k in range(len(self.convs)):
            self.conv(k)

    def step(self):
        self.tail()
        self.convs20()

    def topk(self):
        self.dfl2.dfl2_topk(self.logits, self.idx, self.val, self.ws_topk)

    def select(self):
        i = self.inp
        self.dfl2.dfl2_select(self.idx, self.val, i["verified"], i["hidden"], i["E"], i["W_A"],
                              i["W_B"], i["W_H"], self.scores, self.ws_sel)

    def walk(self):
        self.dfl2.dfl2_walk(self.scores, self.idx, self.T, self.seeds, 0, self.tokens, q=self.q)

    def build_tables(self):
        """P_A, P_B (float32 [V,256]) for the table variant; returns the build time (ms)."""
        V = self.w.V
        dev = self.logits.device
        self.PA = torch.empty(V, 256, dtype=torch.float32, device=dev)
        self.PB = torch.empty_like(self.PA)
        i = self.inp
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.dfl2.dfl2_tables_build(i["E"], i["W_A"], i["W_B"], self.PA, self.PB)  # warm
        a.record()
        self.dfl2.dfl2_tables_build(i["E"], i["W_A"], i["W_B"], self.PA, self.PB)
        b.record()
        b.synchronize()
        return a.elapsed_time(b)

    def tail_tables(self):
        i = self.inp
        self.dfl2.dfl2_tail_tables(self.logits, i["verified"], i["hidden"], i["W_H"], self.PA,
                                   self.PB, self.T, self.seeds, 0, self.tokens, self.ws, q=self.q)


def capture(fn):
    """CUDA graph of fn (warmed up twice first); returns (graph, kernels per replay)."""
    import draft_selection_gb300 as dfl2
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    n0 = dfl2.dfl2_launch_count()
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        fn()
    torch.cuda.synchronize()
    return g, dfl2.dfl2_launch_count() - n0


def time_graph(g, steps, warmup, flush):
    """Per-replay device time (ms) with L2 flushed before every replay."""
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(warmup + steps):
        flush.fill_(i & 0xFF)
        torch.cuda._sleep(20000)  # keeps the GPU busy while the host enqueues the replay
        if i >= warmup:
            ev[i - warmup][0].record(stream)
        g.replay()
        if i >= warmup:
            ev[i - warmup][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def graph_floor(steps, warmup, flush):
    """Device time of a graph replay holding one trivial kernel (a 4-byte fill),
    timed like the ops: the launch and event overhead inside every per-op number."""
    tiny = torch.zeros(1, dtype=torch.int32, device=flush.device)
    g, _ = capture(lambda: tiny.fill_(1))
    return summarize(time_graph(g, steps, warmup, flush))


def sustained(g, seconds):
    """Mean device time per replay of g run back to back (no flush, no host gap)
    for about `seconds`: the steady state, and load for the clock sampler."""
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    b.synchronize()
    per = max(a.elapsed_time(b), 1e-3)
    n = max(10, int(seconds * 1e3 / per))
    done, total_ms = 0, 0.0
    while done < n:
        k = min(n - done, 2000)
        a.record(stream)
        for _ in range(k):
            g.replay()
        b.record(stream)
        b.synchronize()
        total_ms += a.elapsed_time(b)
        done += k
    return total_ms / done


def summarize(ts):
    return {"mean_ms": float(np.mean(ts)), "median_ms": float(np.median(ts)),
            "min_ms": float(np.min(ts))}


def roofline_obj(bytes_per_launch, ms, peak_gbs, which, traffic=None):
    gbs = bytes_per_launch / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_gbs, "unit": "GB/s",
            "frac": round(gbs / peak_gbs, 4), "traffic": traffic, "peak_kind": which}


# --------------------------------------------------------------------------- runs


def measure_native(case: Case, steps: int, warmup: int, flush, pk, which):
    w = case.w
    tb = tail_bytes(w, case.es)
    cb = conv_bytes(w)
    g_step, k_step = capture(case.step)
    g_tail, _ = capture(case.tail)
    g_topk, _ = capture(case.topk)
    case.topk()
    g_sel, _ = capture(case.select)
    case.select()
    g_walk, _ = capture(case.walk)
    g_conv, _ = capture(lambda: case.conv(0))
    g_c20, _ = capture(case.convs20)
    sub = max(3, min(steps, 400))
    res = {"step": summarize(time_graph(g_step, steps, warmup, flush)),
           "tail": summarize(time_graph(g_tail, sub, warmup, flush)),
           "topk": summarize(time_graph(g_topk, sub, warmup, flush)),
           "select": summarize(time_graph(g_sel, sub, warmup, flush)),
           "walk": summarize(time_graph(g_walk, sub, warmup, flush)),
           "conv_alone": summarize(time_graph(g_conv, sub, warmup, flush))}
    # A conv call as it runs in the step: the graph of the block's conv calls
    # back to back (one graph launch amortised over them), per call.
    c20 = summarize(time_graph(g_c20, sub, warmup, flush))
    res["conv"] = {k: v / w.conv_calls for k, v in c20.items()}
    res["floor"] = graph_floor(sub, warmup, flush)
    res["kernels_per_step"] = k_step
    build_ms = case.build_tables()
    g_tt, _ = capture(case.tail_tables)
    tt = summarize(time_graph(g_tt, sub, warmup, flush))["mean_ms"]
    ttb = tail_tables_bytes(w, case.es)
    res["tables"] = {"tail_us": round(tt * 1e3, 2), "build_ms": round(build_ms, 3),
                     "tail_bytes": ttb,
                     "tail_frac_of_hbm": round(ttb / (tt * 1e-3) / 1e9 / pk["hbm_gbs"], 4)}
    del case.PA, case.PB
    if w.B == 1:
        # the split-K projection on its warp-level engine (mma.sync), same graphs
        prev = case.dfl2.dfl2_set_projection_engine(case.dfl2.PROJ_WARP)
        try:
            g_tw, _ = capture(case.tail)
            case.topk()
            g_sw, _ = capture(case.select)
        finally:
            case.dfl2.dfl2_set_projection_engine(prev)
        res["proj_engines"] = {
            "tensor": {"tail_us": round(res["tail"]["mean_ms"] * 1e3, 2),
                       "select_us": round(res["select"]["mean_ms"] * 1e3, 2)},
            "warp": {"tail_us": round(summarize(time_graph(g_tw, sub, warmup, flush))["mean_ms"] * 1e3, 2),
                     "select_us": round(summarize(time_graph(g_sw, sub, warmup, flush))["mean_ms"] * 1e3, 2)},
        }
    peak = pk["hbm_gbs"]
    shares = {"topk": res["topk"]["mean_ms"], "select": res["select"]["mean_ms"],
              "walk": res["walk"]["mean_ms"], "conv": res["conv"]["mean_ms"] * w.conv_calls}
    dominant = max(shares, key=shares.get)
    tr = lambda op: NCU_TRAFFIC.get((op, w.name))
    per_kernel = {
        "topk": roofline_obj(tb["topk"], res["topk"]["mean_ms"], peak, which, tr("topk")),
        "select": roofline_obj(tb["select"], res["select"]["mean_ms"], peak, which, tr("select")),
        "walk": roofline_obj(tb["walk"], res["walk"]["mean_ms"], peak, which, tr("walk")),
        "conv": roofline_obj(cb, res["conv"]["mean_ms"], peak, which, tr("conv")),
    }
    per_kernel["select"]["tflops"] = round(select_flops(w) / (res["select"]["mean_ms"] * 1e-3)
                                           / 1e12, 2)
    per_kernel["conv"]["tflops"] = round(conv_flops(w) / (res["conv"]["mean_ms"] * 1e-3) / 1e12, 2)
    res["shares_ms"] = shares
    res["dominant"] = dominant
    res["per_kernel"] = per_kernel
    res["tail_bytes"] = tb["total"]
    res["conv_bytes_per_call"] = cb
    return res, g_step


def measure_verify(w: wl.Workload, device, steps, warmup, flush, peak_gbs):
    """Block verification (dfl2_verify) after the walk, each mode in its own
    graph: sampling reads one row of target probabilities per sequence, greedy
    ranks all L+1 rows."""
    import draft_selection_gb300 as dfl2
    inp = wl.make_verify_inputs(w, device=device)
    B, L, V = w.B, w.L, w.V
    n = torch.empty(B, dtype=torch.int32, device=device)
    out = torch.empty(B, L + 1, dtype=torch.int32, device=device)
    ws = dfl2.workspace(dfl2.dfl2_verify_workspace_size(B, L, V), device)
    seeds = torch.from_numpy(inp["seeds"].view(np.int64)).to(device)
    res = {}
    for mode in ("sampling", "greedy"):
        fn = lambda g=(mode == "greedy"): dfl2.dfl2_verify(
            inp["p"], inp["tokens"], n, out, greedy=g, slots=inp["slots"], q=inp["q"],
            cand_idx=inp["cand_idx"], seeds=seeds, cycle_offset=0, ws=ws)
        graph, _ = capture(fn)
        ms = summarize(time_graph(graph, max(3, min(steps, 200)), warmup, flush))["mean_ms"]
        nbytes = B * (V * 4 + L * 16) if mode == "sampling" else B * (L + 1) * V * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[mode] = {"us": round(ms * 1e3, 2), "bytes": nbytes, "gbs": round(gbs, 1),
                     "frac_of_hbm": round(gbs / peak_gbs, 4)}
    del inp
    return res


def measure_lmhead(w: wl.Workload, device, steps, warmup, flush, pk):
    """LM head + top-16 from the last hidden state: the fused kernel
    (dfl2_lmhead_topk, logits never written) against the unfused pair a
    library user would otherwise run, a cuBLAS bf16 GEMM writing the [B*L, V]
    logits followed by dfl2_topk over them.  Each arm in its own graph, L2
    flushed before every replay (W_lm alone is larger than L2)."""
    import draft_selection_gb300 as dfl2
    inp = wl.make_lmhead_inputs(w, device, "gauss")
    B, L, V, d = w.B, w.L, w.V, w.d
    R = B * L
    h, W = inp["hidden"], inp["W_lm"]
    idx = torch.empty(B, L, 16, dtype=torch.int32, device=device)
    val = torch.empty(B, L, 16, dtype=torch.float32, device=device)
    ws = dfl2.workspace(dfl2.dfl2_lmhead_topk_workspace_size(B, L, V, d), device)
    logits = torch.empty(R, V, dtype=torch.bfloat16, device=device)
    ws_t = dfl2.workspace(dfl2.dfl2_topk_workspace_size(B, L, V), device)
    h2 = h.view(R, d)
    fused = lambda: dfl2.dfl2_lmhead_topk(h, W, idx, val, ws)
    gemm = lambda: torch.matmul(h2, W.t(), out=logits)
    unfused = lambda: (gemm(), dfl2.dfl2_topk(logits.view(B, L, V), idx, val, ws_t))
    n = max(3, min(steps, 100))
    res = {}
    for name, fn in (("fused", fused), ("cublas_gemm", gemm), ("cublas_gemm_plus_topk", unfused)):
        graph, k = capture(fn)
        ms = summarize(time_graph(graph, n, warmup, flush))["mean_ms"]
        res[name + "_us"] = round(ms * 1e3, 2)
        if name == "fused":
            res["fused_launches"] = k
            fused_ms = ms
    torch.cuda.synchronize()
    assert dfl2.dfl2_device_error() == 0
    flops = 2.0 * R * V * d
    nbytes = V * d * 2 + R * d * 2 + R * 16 * 8
    tflops = flops / (fused_ms * 1e-3) / 1e12
    gbs = nbytes / (fused_ms * 1e-3) / 1e9
    # memory-bound while the weight read outlasts the MMAs at the measured peaks
    hbm_s = nbytes / (pk["hbm_gbs"] * 1e9)
    tc_s = flops / (pk["bf16_tflops"] * 1e12)
    if hbm_s >= tc_s:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm_gbs"], 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(tflops, 1), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(tflops / pk["bf16_tflops"], 4)}
    roof["traffic"] = NCU_TRAFFIC.get(("lmhead", w.name))
    res.update({"workload": w.name, "rows": R, "V": V, "d": d, "flops": flops, "bytes": nbytes,
                "tflops": round(tflops, 1), "gbs": round(gbs, 1), "roofline": roof,
                "speedup_vs_cublas_plus_topk": round(res["cublas_gemm_plus_topk_us"] /
                                                     res["fused_us"], 3),
                "inputs": "h ~ N(0,1), W_lm ~ N(0, 1/sqrt(d)), bf16"})
    del inp, logits
    return res


def measure_e2e(case: Case, g_step, steps, warmup, flush):
    """The same step with its inputs copied from pinned host memory (one copy of
    the staging buffer) and its outputs read back (one copy) inside the timed
    region."""
    pinned_in = case.staged_in.buf.detach().cpu().pin_memory()
    pinned_out = torch.empty(case.staged_out.buf.shape, dtype=torch.uint8, pin_memory=True)
    h2d = case.staged_in.nbytes
    d2h = case.staged_out.nbytes
    stream = torch.cuda.current_stream()
    ts = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(warmup + steps)]
    for i in range(warmup + steps):
        flush.fill_(i & 0xFF)
        # the GPU sleeps while the host enqueues the copies and the replay, so that
        # no host-side enqueue time falls inside the timed region
        torch.cuda._sleep(200000)
        a, b = ev[i]
        a.record(stream)
        case.staged_in.buf.copy_(pinned_in, non_blocking=True)
        g_step.replay()
        pinned_out.copy_(case.staged_out.buf, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= warmup:
            ts.append(a.elapsed_time(b))
    return float(np.mean(ts)), h2d, d2h


def cpu_baseline(case: Case, budget_s: float = 12.0):
    """The oracle, as it stands, on this host's cores: whole draft blocks of the
    same workload (tail + 20 conv calls) until the time budget is spent."""
    import oracle
    w = case.w
    lg = wl.host(case.logits)
    i = {k: (wl.host(v) if isinstance(v, torch.Tensor) else v) for k, v in case.inp.items()}
    convs = [{k: wl.host(v) for k, v in c.items() if k != "y"} for c in case.convs]
    n, t0 = 0, time.perf_counter()
    while True:
        idx, val = oracle.topk(lg, 16)
        S = oracle.select(idx, val, i["verified"], i["hidden"], i["E"], i["W_A"], i["W_B"],
                          i["W_H"])
        oracle.walk(S, idx, case.T, i["seeds"], 0)
        for c in convs:
            oracle.conv2(c["x"], c["x_prev"], c["base"], c["W_c"])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(dt / n * 1e6, 1), "unit": "µs per draft block",
            "cores": oracle.get_threads(), "kind": "oracle",
            "sample": f"{n} whole {w.name} blocks (tail + {w.conv_calls} conv calls), "
                      f"{dt:.1f} s of host time"}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = wl.WORKLOADS[args.workload]
    T = 1.0
    lg = wl.host(wl.make_logits(w, "cpu"))
    i = {k: (wl.host(v) if isinstance(v, torch.Tensor) else v)
         for k, v in wl.make_tail_inputs(w, "cpu").items()}
    convs = [{k: wl.host(v) for k, v in wl.make_conv_inputs(w, c, "cpu").items()}
             for c in range(w.conv_calls)]

    def block():
        idx, val = oracle.topk(lg, 16)
        S = oracle.select(idx, val, i["verified"], i["hidden"], i["E"], i["W_A"], i["W_B"],
                          i["W_H"])
        oracle.walk(S, idx, T, i["seeds"], 0)
        for c in convs:
            oracle.conv2(c["x"], c["x_prev"], c["base"], c["W_c"])

    for _ in range(args.warmup):
        block()
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        block()
        ts.append(time.perf_counter() - t0)
    us = float(np.mean(ts)) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1),
            "unit": "µs per draft block", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "V": w.V, "d": w.d, "T": T,
                       "conv_calls": w.conv_calls},
            "cpu_baseline": {"value": round(us, 1), "unit": "µs per draft block",
                             "cores": oracle.get_threads(), "kind": "oracle",
                             "sample": f"{args.steps} whole {w.name} blocks per the step count"},
            "e2e": {"value": round(us, 1), "unit": "µs per draft block",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profile_op(args) -> int:
    """Runs one op of the path --steps times on --workload with no timing, for a
    profiler to capture (e.g. ncu -k regex:topk16 ... bench.py --profile-op topk)."""
    from draft_selection_gb300 import build
    build.build()
    import draft_selection_gb300 as dfl2
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if args.proj_engine == "warp":
        dfl2.dfl2_set_projection_engine(dfl2.PROJ_WARP)
    if args.profile_op == "lmhead":
        w = wl.WORKLOADS[args.workload]
        lm = wl.make_lmhead_inputs(w, dev, "gauss")
        lm_idx = torch.empty(w.B, w.L, 16, dtype=torch.int32, device=dev)
        lm_val = torch.empty(w.B, w.L, 16, dtype=torch.float32, device=dev)
        lm_ws = dfl2.workspace(dfl2.dfl2_lmhead_topk_workspace_size(w.B, w.L, w.V, w.d), dev)
        case = None
    else:
        case = Case(wl.WORKLOADS[args.workload], 1.0, dev)
    if args.profile_op in ("select", "walk"):
        case.topk()
    if args.profile_op == "walk":
        case.select()
    if case is None:
        fn = lambda: dfl2.dfl2_lmhead_topk(lm["hidden"], lm["W_lm"], lm_idx, lm_val, lm_ws)
    else:
        fn = {"topk": case.topk, "select": case.select, "walk": case.walk,
              "conv": lambda: case.conv(0), "conv_plain": lambda: case.conv(0, plain=True),
              "tail": case.tail, "step": case.step}[args.profile_op]
    for _ in range(args.steps):
        fn()
    torch.cuda.synchronize()
    err = dfl2.dfl2_device_error()
    print(json.dumps({"profile_op": args.profile_op, "workload": args.workload,
                      "calls": args.steps, "device_error": err}), flush=True)
    return 0 if err == 0 else 1


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--batched", default=BATCHED, help="second workload ('' to skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back steps after the timed region")
    ap.add_argument("--proj-engine", choices=["tensor", "warp"], default="tensor",
                    help="engine of the split-K projection in --profile-op runs")
    ap.add_argument("--profile-op",
                    choices=["topk", "select", "walk", "conv", "conv_plain", "tail", "step",
                             "lmhead"],
                    help="run one op --steps times, untimed, for a profiler; no JSON line")
    args = ap.parse_args()
    if args.profile_op:
        return profile_op(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_init()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    from draft_selection_gb300 import build
    build.build()
    import draft_selection_gb300 as dfl2
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pk, which = peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    w = wl.WORKLOADS[args.workload]
    T = 1.0
    case = Case(w, T, device)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    res, g_step = measure_native(case, args.steps, args.warmup, flush, pk, which)
    step_ms = max_over_ranks(res["step"]["mean_ms"], world)
    # the step back to back for a few seconds: steady state with warm L2 and the
    # GPU under load while the clocks are sampled
    sustained_ms = sustained(g_step, args.sustain_s)
    barrier(world)
    e2e_ms, h2d, d2h = measure_e2e(case, g_step, max(3, min(args.steps, 200)), args.warmup, flush)
    e2e_ms = max_over_ranks(e2e_ms, world)
    verify = {w.name: measure_verify(w, device, args.steps, args.warmup, flush, pk["hbm_gbs"])}

    batched = None
    if args.batched:
        wb = wl.WORKLOADS[args.batched]
        cb = Case(wb, 1.0, device)
        rb, _ = measure_native(cb, max(3, min(args.steps, 200)), args.warmup, flush, pk, which)
        tail_ms = max_over_ranks(rb["tail"]["mean_ms"], world)
        step_b = max_over_ranks(rb["step"]["mean_ms"], world)
        tb = tail_bytes(wb, cb.es)["total"]
        batched = {
            "workload": wb.name, "B": wb.B,
            "blocks_per_s": round(world * wb.B / (step_b * 1e-3), 1),
            "tail_blocks_per_s": round(world * wb.B / (tail_ms * 1e-3), 1),
            "step_us": round(step_b * 1e3, 2), "tail_us": round(tail_ms * 1e3, 2),
            "conv_us_per_call": round(rb["conv"]["mean_ms"] * 1e3, 2),
            "conv_alone_us": round(rb["conv_alone"]["mean_ms"] * 1e3, 2),
            "tail_hbm_gbs": round(tb / (tail_ms * 1e-3) / 1e9, 1),
            "tail_frac_of_hbm": round(tb / (tail_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "tail_bytes": tb,
            "roofline": rb["per_kernel"][rb["dominant"]] | {"kernel": rb["dominant"]},
            "per_kernel": rb["per_kernel"],
            "kernel_ms": {k: round(rb[k]["mean_ms"], 5) for k in
                          ("topk", "select", "walk", "conv")},
            "tables": rb["tables"],
        }
        del cb
        verify[wb.name] = measure_verify(wb, device, args.steps, args.warmup, flush, pk["hbm_gbs"])
    lmhead = {}
    for name in (w.name, args.batched):
        if name:
            lmhead[name] = measure_lmhead(wl.WORKLOADS[name], device, args.steps, args.warmup,
                                          flush, pk)
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, args.cpu_budget)

    if rank == 0:
        us_block = step_ms * 1e3 / world
        line = {
            "metric": METRIC, "value": round(us_block, 2), "unit": "µs per draft block",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_ms, 5), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "V": w.V, "d": w.d, "T": T,
                       "conv_calls": w.conv_calls, "step": "tail + 20 conv (CUDA graph)",
                       "l2": "flushed (256 MB write) before every timed step"},
            "tail_us": round(res["tail"]["mean_ms"] * 1e3, 2),
            "conv20_us": round(res["conv"]["mean_ms"] * 1e3 * w.conv_calls, 2),
            "kernel_us": {k: round(res[k]["mean_ms"] * 1e3, 2) for k in
                          ("topk", "select", "walk", "conv", "conv_alone")},
            # per-op graphs minus the one-kernel graph floor (launch + events),
            # comparable with ncu's per-launch durations; conv is already per
            # call of a 20-call graph, so it keeps its value
            "graph_floor_us": round(res["floor"]["mean_ms"] * 1e3, 2),
            "kernel_us_net": {k: round((res[k]["mean_ms"] - res["floor"]["mean_ms"]) * 1e3, 2)
                              for k in ("topk", "select", "walk", "tail", "conv_alone")},
            "sustained_step_us": round(sustained_ms * 1e3, 2),
            "roofline": res["per_kernel"][res["dominant"]] | {"kernel": res["dominant"]},
            "per_kernel": res["per_kernel"],
            "tables": res["tables"],
            "proj_engines": res.get("proj_engines"),
            "b64": batched,
            "verify": verify,
            "lmhead_topk": lmhead,
            "e2e": {"value": round(e2e_ms * 1e3 / world, 2), "unit": "µs per draft block",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": res["kernels_per_step"] * args.steps,
            "kernels_per_step": res["kernels_per_step"],
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
