"""Benchmark: MoE dispatch + combine on one GB300 (µs per layer, HBM GB/s).

One step = one pass of the whole path over one synthetic layer: route
(top-K), dispatch (count, scan, scatter [+ FP8 quantise]), the per-expert
scale stand-in for the grouped GEMM, combine.  The metric is dispatch +
combine µs per layer (CUDA events on the launching stream around each call;
the L2 is flushed by a 256 MiB write before dispatch and before combine,
outside those events).  ``value`` is that time; the roofline object reports
the dominant call's algorithmic bytes / its event time against the measured
HBM copy bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 (torchrun, one process per GPU) runs N independent replicas of the
layer; ranks do not exchange data.  ``--impl reference`` times the CPU oracle
(single-threaded C) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "dispatch+combine µs/layer and achieved HBM GB/s (% of 8 TB/s) on 1 GB300"
UNIT = "us/layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# algorithmic bytes (the minimum each call must move)
# ---------------------------------------------------------------------------

def dispatch_bytes(T, E, R, K, H, fp8):
    payload = T * K * H * (1 if fp8 else 2)
    scales = T * K * (H // 128) * 4 if fp8 else 0
    return T * H * 2 + payload + scales + T * K * 4 + 2 * T * K * 4 + 2 * E * R * 4


def combine_bytes(T, K, H):
    return T * K * H * 2 + T * H * 2 + T * K * 4 + T * K * 4


def route_bytes(T, E, K):
    return T * E * 4 + T * K * 8


def routing_load(counts, E: int, R: int) -> dict:
    """How evenly the routing spreads the rows, from dispatch's count matrix
    (counts[e*R + s] = tokens of rank s routed to expert e): rows per expert
    and rows per destination rank (its E/R experts), max, min and max/mean."""
    c = np.asarray(counts, dtype=np.int64).reshape(E, R)
    per_expert = c.sum(axis=1)
    per_rank = per_expert.reshape(R, E // R).sum(axis=1)

    def stats(v):
        mean = float(v.mean())
        return {"max": int(v.max()), "min": int(v.min()), "mean": mean,
                "max_over_mean": float(v.max()) / mean if mean > 0 else None}

    return {"rows_per_expert": stats(per_expert), "rows_per_dest_rank": stats(per_rank)}


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel_file: str, summary_name: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", summary_name)
    src = os.path.join(ROOT, "combine_moe_route_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-* ")
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in a child process."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, "t_" + which, time.time())

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._reader.join(timeout=2)

    def summary(self):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        inside = [r for r in rows if self.t_start and self.t_stop and self.t_start <= r[0] <= self.t_stop + 0.06]
        window = "timed"
        if not inside:
            inside, window = rows, "warmup+timed (timed region shorter than the 50 ms sampling period)"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(v: float, world: int, device) -> float:
    if world <= 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def time_call(fn, stream, reps: int = 50) -> float:
    """Mean µs of fn() over reps calls, CUDA events on the launching stream, after 3 warm-ups."""
    for _ in range(3):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        fn()
    z.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(z) * 1e3 / reps


def time_flushed(fn, stream, flush, reps: int = 50) -> float:
    """Median µs of fn() with the L2 flushed (outside the events) before every call.

    A call here is tens of µs of GPU work, so a host pause of a millisecond (a garbage
    collection) can drain the queue inside one sample; the collector is off while the calls
    are enqueued, and the median ignores a stray sample."""
    for _ in range(3):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    gc_was_on = gc.isenabled()
    gc.disable()
    try:
        for a, z in ev:
            flush.fill_(3)
            a.record(stream)
            fn()
            z.record(stream)
        torch.cuda.synchronize()
    finally:
        if gc_was_on:
            gc.enable()
    return statistics.median(a.elapsed_time(z) for a, z in ev) * 1e3


def time_flushed_after(first, fn, stream, flush, reps: int = 50) -> float:
    """Median µs of fn() when each call follows first() (L2 flushed before first(), outside
    the events): for a receive half, which has something to receive only after its send."""
    for _ in range(3):
        first()
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    gc_was_on = gc.isenabled()
    gc.disable()
    try:
        for a, z in ev:
            flush.fill_(3)
            first()
            a.record(stream)
            fn()
            z.record(stream)
        torch.cuda.synchronize()
    finally:
        if gc_was_on:
            gc.enable()
    return statistics.median(a.elapsed_time(z) for a, z in ev) * 1e3


def measure_workload(name, dev, stream, flush, peak):
    """One workload on its own (the benchmark line's headline is the prefill layer; this covers
    every other one): T, dispatch and combine µs (flushed medians of 50 calls), their
    algorithmic bytes, the fraction of the measured copy peak and the % of 8 TB/s, and the
    CUDA-graph replay of dispatch + combine.  For the bf16 decode layers also the low-latency
    rectangle (chunk cap C = the largest rank; slots in token order, by atomic increments, and
    with the FP8 payload), its combine, and the graph replays of those forms."""
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    B, T, E, K, H, R = inp["B"], inp["T"], w.E, w.K, w.H, w.R
    x = inp["x"].to(dev)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    idx, wts = b.route_topk(logits, K)
    d = b.dispatch(x, idx, B, E, fp8=w.fp8)
    y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E)
    out = b.combine(y, d.tok2row, wts)
    torch.cuda.synchronize()
    db = dispatch_bytes(T, E, R, K, H, w.fp8)
    cb = combine_bytes(T, K, H)
    res = {"T": T, "R": R, "E": E, "K": K, "H": H, "payload": "fp8_e4m3" if w.fp8 else "bf16",
           "route_us": time_flushed(lambda: b.route_topk(logits, K, topk_idx=idx, topk_w=wts), stream, flush),
           "dispatch_us": time_flushed(lambda: b.dispatch(x, idx, B, E, fp8=w.fp8, out=d), stream, flush),
           "combine_us": time_flushed(lambda: b.combine(y, d.tok2row, wts, out=out), stream, flush),
           "algorithmic_bytes": {"dispatch": db, "combine": cb}}
    res["dispatch_plus_combine_us"] = res["dispatch_us"] + res["combine_us"]
    # What a flushed call's time holds besides its kernels: the event pair itself; the write-back
    # of the flush's own dirty lines (a 256 MiB read of another buffer after the flush leaves the
    # L2 holding only clean lines); and the combine as a layer runs it, right after the expert
    # stage that wrote its input (the L2 flushed before the expert stage).
    clean = torch.ones(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sink = torch.empty((), dtype=torch.int64, device=dev)

    def read_clean():
        torch.sum(clean, (0,), dtype=torch.int64, out=sink)

    def comb():
        b.combine(y, d.tok2row, wts, out=out)

    res["fixed_costs"] = {
        "events_only_us": time_flushed(lambda: None, stream, flush),
        "combine_us_clean_l2": time_flushed_after(read_clean, comb, stream, flush),
        "combine_us_after_expert": time_flushed_after(
            lambda: b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E, out=y), comb, stream, flush)}
    del clean
    res["frac_of_measured_peak"] = {"dispatch": db / (res["dispatch_us"] * 1e-6) / 1e9 / peak,
                                    "combine": cb / (res["combine_us"] * 1e-6) / 1e9 / peak}
    res["pct_of_8TBs"] = {"dispatch": 100 * db / (res["dispatch_us"] * 1e-6) / 1e9 / NOMINAL_HBM_GBS,
                          "combine": 100 * cb / (res["combine_us"] * 1e-6) / 1e9 / NOMINAL_HBM_GBS}
    res["floor_us_at_8TBs"] = {"dispatch": db / 8e6, "combine": cb / 8e6}
    res["floor_us_at_measured_peak"] = {"dispatch": db / (peak * 1e3), "combine": cb / (peak * 1e3)}
    graphs = []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        b.dispatch(x, idx, B, E, fp8=w.fp8, out=d)
        b.combine(y, d.tok2row, wts, out=out)
    graphs.append(g)
    torch.cuda.synchronize()
    res["graph_dispatch_plus_combine_us"] = time_flushed(g.replay, stream, flush)
    if not w.fp8:
        C = max(1, int(B.max()))
        eo = torch.arange(E + 1, dtype=torch.int32, device=dev) * (R * C)
        dl = b.dispatch_ll(x, idx, B, E, C)
        du = b.dispatch_ll(x, idx, B, E, C, unordered=True)
        dl8 = b.dispatch_ll(x, idx, B, E, C, fp8=True)
        du8 = b.dispatch_ll(x, idx, B, E, C, fp8=True, unordered=True)
        yl = b.expert_scale(dl.recv_x, None, eo, E)
        yu = b.expert_scale(du.recv_x, None, eo, E)
        outl = b.combine_ll(yl, E, R, C, dl.tok2row, wts)
        outu = b.combine_ll(yu, E, R, C, du.tok2row, wts)
        torch.cuda.synchronize()
        ll = {"C": C, "rectangle_rows": E * R * C,
              "ordered_dispatch_us": time_flushed(lambda: b.dispatch_ll(x, idx, B, E, C, out=dl), stream, flush),
              "unordered_dispatch_us": time_flushed(
                  lambda: b.dispatch_ll(x, idx, B, E, C, unordered=True, out=du), stream, flush),
              "ordered_fp8_dispatch_us": time_flushed(
                  lambda: b.dispatch_ll(x, idx, B, E, C, fp8=True, out=dl8), stream, flush),
              "unordered_fp8_dispatch_us": time_flushed(
                  lambda: b.dispatch_ll(x, idx, B, E, C, fp8=True, unordered=True, out=du8), stream, flush),
              "rectangle_combine_us": time_flushed(lambda: b.combine_ll(yl, E, R, C, dl.tok2row, wts, out=outl),
                                                   stream, flush)}
        gl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gl):
            b.dispatch_ll(x, idx, B, E, C, out=dl)
            b.combine_ll(yl, E, R, C, dl.tok2row, wts, out=outl)
        gu = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gu):
            b.dispatch_ll(x, idx, B, E, C, unordered=True, out=du)
            b.combine_ll(yu, E, R, C, du.tok2row, wts, out=outu)
        graphs += [gl, gu]
        torch.cuda.synchronize()
        ll["graph_ordered_dispatch_plus_combine_us"] = time_flushed(gl.replay, stream, flush)
        ll["graph_unordered_dispatch_plus_combine_us"] = time_flushed(gu.replay, stream, flush)
        res["low_latency"] = ll
    res["routing_load"] = routing_load(d.counts.cpu().numpy(), E, R)
    del graphs
    return _rounded(res)


def _rounded(v):
    if isinstance(v, float):
        return round(v, 4)
    if isinstance(v, dict):
        return {k: _rounded(u) for k, u in v.items()}
    return v


def measure_eager_layers(dev, stream):
    """Whole eager DeepSeek-V3 decode layers (route, dispatch, expert stand-in, combine) enqueued
    back to back: through the package functions, whose per-call checks cost host time, and
    through BoundLayer."""
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS["dsv3_decode"]
    inp = wl.generate(w, seed=0)
    B, E, K = inp["B"], w.E, w.K
    x = inp["x"].to(dev)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    bound = b.BoundLayer(x, logits, B, E, K)

    def eager_us(fn, n=50):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        z.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(z) * 1e3 / n

    return {"eager_dsv3_decode_layer": {"package_us": round(eager_us(lambda: b.moe_layer(x, logits, B, E, K)), 2),
                                        "bound_us": round(eager_us(bound), 2)}}


def measure_split_halves(name, dev, stream, flush, inter=2048, reps=20):
    """The split dispatch and combine on one workload: each half timed alone (flushed medians),
    against the one-call forms; then Dispatch Overlap ([DSD] "Computation and communication
    overlap"): the send half on a side stream while a dummy shared expert -- silu(x W1) W2,
    bf16 cuBLAS GEMMs of intermediate size `inter` -- runs on the main stream, then the receive
    half behind an event.  The send half is given every SM or a capped budget, so that the
    shared expert keeps the rest.  Reported per budget: serialised (one stream) and overlapped
    µs, and the fraction of the dispatch hidden."""
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    B, T, E, K, H, R = inp["B"], inp["T"], w.E, w.K, w.H, w.R
    x = inp["x"].to(dev)
    idx, wts = b.route_topk(torch.from_numpy(inp["logits"]).to(dev), K)
    d = b.dispatch(x, idx, B, E, fp8=w.fp8)
    ds = b.dispatch_send(x, idx, B, E, fp8=w.fp8)
    b.dispatch_recv(ds, B, E, K)
    y = b.expert_scale(ds.recv_x, ds.recv_scale, ds.expert_offsets, E)
    out = b.combine(y, ds.tok2row, wts)
    torch.cuda.synchronize()
    res = {"T": T,
           "dispatch_us": time_flushed(lambda: b.dispatch(x, idx, B, E, fp8=w.fp8, out=d), stream, flush),
           "dispatch_send_us": time_flushed(lambda: b.dispatch_send(x, idx, B, E, fp8=w.fp8, out=ds), stream, flush),
           "dispatch_recv_us": time_flushed_after(lambda: b.dispatch_send(x, idx, B, E, fp8=w.fp8, out=ds),
                                                  lambda: b.dispatch_recv(ds, B, E, K), stream, flush),
           "dispatch_send_plus_recv_us": time_flushed(
               lambda: (b.dispatch_send(x, idx, B, E, fp8=w.fp8, out=ds), b.dispatch_recv(ds, B, E, K)),
               stream, flush),
           "combine_us": time_flushed(lambda: b.combine(y, ds.tok2row, wts, out=out), stream, flush),
           "combine_send_plus_recv_us": time_flushed(
               lambda: (b.combine_send(ds.workspace, R), b.combine_recv(y, ds.tok2row, wts, ds.workspace, R, out=out)),
               stream, flush)}
    st, code = b.get_device_error(ds.workspace)
    if st != 0:
        raise RuntimeError(f"device error word {code:#x} in the split halves")

    gen = torch.Generator(device=dev).manual_seed(0)
    w1 = (torch.randn((H, inter), device=dev, generator=gen) * H ** -0.5).to(torch.bfloat16)
    w2 = (torch.randn((inter, H), device=dev, generator=gen) * inter ** -0.5).to(torch.bfloat16)
    side = torch.cuda.Stream(dev)

    def shared():
        return torch.nn.functional.silu(x @ w1) @ w2

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.fill_(4)
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            z.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(z) * 1e3)
        return statistics.median(ts)

    res["shared_expert_us"] = timed(shared)
    overlap = {}
    for max_sms in (0, 114, 76):
        def serial():
            b.dispatch_send(x, idx, B, E, fp8=w.fp8, max_sms=max_sms, out=ds)
            shared()
            b.dispatch_recv(ds, B, E, K)

        def overlapped():
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                b.dispatch_send(x, idx, B, E, fp8=w.fp8, max_sms=max_sms, out=ds)
                sent = torch.cuda.Event()
                sent.record(side)
            shared()
            stream.wait_event(sent)
            b.dispatch_recv(ds, B, E, K)

        send_alone = timed(lambda: b.dispatch_send(x, idx, B, E, fp8=w.fp8, max_sms=max_sms, out=ds))
        ser, ovl = timed(serial), timed(overlapped)
        overlap[f"max_sms_{max_sms or 'all'}"] = {
            "send_alone_us": send_alone, "serialised_us": ser, "overlapped_us": ovl,
            "hidden_frac_of_dispatch": (ser - ovl) / res["dispatch_us"]}
    res["dispatch_overlap"] = overlap
    st, code = b.get_device_error(ds.workspace)
    if st != 0:
        raise RuntimeError(f"device error word {code:#x} in the overlap runs")
    return _rounded(res)


def measure_partial_combine(b, y, d, idx, wts, out, E, R, K, H, T, stream, flush):
    """Sender-side partial accumulation on the benchmark layer: time of the send and receive
    halves, rows that would travel back (one per (token, expert rank) instead of one per copy),
    and the error of both combine forms against an fp64 sum on 256 sampled tokens."""
    part = b.combine_partial_send(y, d.tok2row, idx, wts, E, R)
    op = b.combine_partial_recv(part, idx, E, R)
    torch.cuda.synchronize()
    send_us = time_flushed(lambda: b.combine_partial_send(y, d.tok2row, idx, wts, E, R, out=part), stream, flush)
    recv_us = time_flushed(lambda: b.combine_partial_recv(part, idx, E, R, out=op), stream, flush)
    ranks = (idx // (E // R)).cpu().numpy()
    distinct = int(sum(len(np.unique(r)) for r in ranks))
    # precision on a sample of tokens: both forms against an fp64 sum of the same bf16 inputs
    rng = np.random.default_rng(0)
    g = np.sort(rng.choice(T, size=min(256, T), replace=False))
    rows = d.tok2row.view(T, K)[torch.from_numpy(g).to(y.device)].reshape(-1).long()
    yv = y.index_select(0, rows).float().cpu().numpy().astype(np.float64).reshape(len(g), K, H)
    wv = wts.cpu().numpy()[g].astype(np.float64)
    exact = np.einsum("tk,tkh->th", wv, yv)
    errs = {}
    for name, o in (("receive_side", out), ("sender_side", op)):
        ov = o.float().cpu().numpy()[g].astype(np.float64)
        err = np.abs(ov - exact)
        ulp = np.maximum(np.abs(exact), 2.0**-126) * 2.0**-8
        errs[name] = {"rms_rel": float(np.sqrt((err**2).mean() / (exact**2).mean())),
                      "max_bf16_ulp": float((err / ulp).max())}
    return {"partial_combine": {
        "send_us": round(send_us, 2), "recv_us": round(recv_us, 2),
        "rows_returned": distinct, "rows_returned_receive_side": T * K,
        "return_bytes_saved_frac": round(1.0 - distinct / (T * K), 4),
        "error_vs_fp64": errs}}


def replica_value(per_rank_us: float, world: int) -> float:
    """Whole-job µs per layer for N independent replicas: the slowest rank's
    time per layer divided by the N layers processed in that time."""
    return per_rank_us / world


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ---------------------------------------------------------------------------

def oracle_sample(workload, tokens_per_rank: int, seed: int = 0):
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[workload]
    B = np.full(w.R, tokens_per_rank, np.int32)
    inp = wl.generate(w, seed=seed, B=B)
    return w, inp


class OracleLayer:
    """The oracle's inputs for one sample, with routing and expert outputs prepared once."""

    def __init__(self, w, inp):
        import oracle
        from combine_moe_route_gb300 import workloads as wl
        self.o, self.w, self.inp = oracle, w, inp
        self.x = wl.bf16_bits(inp["x"])
        self.idx, self.wts = oracle.route_topk(inp["logits"], w.K)
        d = oracle.dispatch(self.x, self.idx, inp["B"], w.E, fp8=w.fp8)
        self.tok2row = d["tok2row"]
        self.y = oracle.expert_scale(d["recv"], d["recv_scale"], d["expert_offsets"], w.E)

    def time_step(self):
        """Seconds of one oracle dispatch plus one oracle combine on this sample."""
        t0 = time.perf_counter()
        self.o.dispatch(self.x, self.idx, self.inp["B"], self.w.E, fp8=self.w.fp8)
        t1 = time.perf_counter()
        self.o.combine(self.y, self.tok2row, self.wts, out="bf16")
        t2 = time.perf_counter()
        return t2 - t0


def pct(ms: list) -> list:
    """[p10, p90] of a list of millisecond timings, in µs."""
    q = sorted(ms)
    at = lambda f: q[min(len(q) - 1, int(round(f * (len(q) - 1))))] * 1e3
    return [at(0.10), at(0.90)]


def host_cpu() -> dict:
    """The host's logical CPU count and model: lscpu's "Model name" (on Arm hosts lscpu names
    the core, e.g. Neoverse-V2, where /proc/cpuinfo has no model line), else /proc/cpuinfo;
    on Arm also the main ID register (implementer 0x41 = Arm; part 0xd4f = Neoverse V2)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip().lower() == "model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    key = line.split(":", 1)[0].strip().lower()
                    if key in ("model name", "cpu model", "hardware"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    info = {"nproc": os.cpu_count(), "model": model or platform.processor() or platform.machine(),
            "machine": platform.machine()}
    try:
        with open("/sys/devices/system/cpu/cpu0/regs/identification/midr_el1") as f:
            info["midr_el1"] = f.read().strip()
    except OSError:
        pass
    return info


def path_dtype(w) -> str:
    """The arithmetic types the path computes in, for the bench line's ``dtype``."""
    if w.fp8:
        return "e4m3 dispatch payload + f32 scale per 128 channels; bf16 rows; f32 accumulate"
    return "bf16 rows; f32 accumulate"


L2_NOTE = (f"flushed by a {L2_FLUSH_BYTES >> 20} MiB write before route, dispatch and combine "
           "(outside their events)")


def cpu_baseline(workload: str, T_full: int):
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[workload]
    tpr = max(1, (T_full // w.R) // 8)
    w, inp = oracle_sample(workload, tpr)
    layer = OracleLayer(w, inp)
    t_start = time.perf_counter()
    times = []
    while True:
        times.append(layer.time_step())
        if time.perf_counter() - t_start > 10.0 or len(times) >= 20:
            break
    T_s = inp["T"]
    per_layer_us = statistics.median(times) * 1e6 * (T_full / T_s)
    return {"value": per_layer_us, "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
            "sample": f"{workload} with {tpr} tokens/rank (T={T_s} of {T_full}); median of {len(times)} "
                      "runs of oracle dispatch + combine, scaled by T_full/T_sample; single-threaded C"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    T_full = int(wl.draw_B(w, 0).sum())
    # each step: the oracle on 1/64 of the layer's tokens (at least 1 per rank), scaled to the layer
    tpr = max(1, (T_full // w.R) // 64)
    w, inp = oracle_sample(args.workload, tpr)
    layer = OracleLayer(w, inp)
    for _ in range(args.warmup):
        layer.time_step()
    times = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        times.append(layer.time_step() * 1e6 * (T_full / inp["T"]))
    wall = time.perf_counter() - t0
    value = statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(1, args.steps),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": path_dtype(w),
        "data": "synthetic", "config": bench_config(w, T_full, L2_NOTE),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "host": host_cpu(),
                         "sample": f"{args.workload} with {tpr} tokens/rank per step (T={inp['T']} of {T_full}), "
                                   "oracle dispatch + combine scaled by T_full/T_sample; single-threaded C"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def bench_config(w, T, l2, tokens_per_rank=None):
    tpr = tokens_per_rank if tokens_per_rank is not None else (
        f"{w.b_lo}" if w.b_lo == w.b_hi else f"U{{{w.b_lo}..{w.b_hi}}}")
    return {"workload": w.name, "R": w.R, "E": w.E, "K": w.K, "H": w.H, "T": T, "tokens_per_rank": tpr,
            "dispatch_payload": "fp8_e4m3 + fp32 scale per 128 channels" if w.fp8 else "bf16",
            "combine_out": "bf16 (fp32 accumulate)", "l2": l2, "seed": 0, "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, world, rank, local):
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import build
    from combine_moe_route_gb300 import workloads as wl

    if not os.path.exists(build.library_path()):
        build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    if args.tokens_per_rank is not None:          # a smaller case of the same layer (profiling)
        inp = wl.generate(w, seed=0, B=np.full(w.R, args.tokens_per_rank, np.int32))
    else:
        inp = wl.generate(w, seed=0)
    B, T, E, K, H = inp["B"], inp["T"], w.E, w.K, w.H
    stream = torch.cuda.current_stream(dev)

    x = inp["x"].to(dev)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    wts = torch.empty((T, K), dtype=torch.float32, device=dev)
    b.route_topk(logits, K, topk_idx=idx, topk_w=wts)
    d = b.dispatch(x, idx, B, E, fp8=w.fp8)                 # allocates outputs + workspace once
    y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E)
    out = b.combine(y, d.tok2row, wts)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    st, code = b.get_device_error(d.workspace)
    if st != 0:
        raise RuntimeError(f"device error word {code:#x} after the first layer")

    def step(ev=None):
        # every timed call follows an L2 flush: cold caches, and GPU work queued ahead of the
        # call so that its events time the kernels, not the host issuing them
        flush.fill_(0)
        if ev is not None:
            ev[0].record(stream)
        b.route_topk(logits, K, topk_idx=idx, topk_w=wts)
        if ev is not None:
            ev[1].record(stream)
        flush.fill_(1)
        if ev is not None:
            ev[2].record(stream)
        b.dispatch(x, idx, B, E, fp8=w.fp8, out=d)
        if ev is not None:
            ev[3].record(stream)
        b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E, out=y)
        if ev is not None:
            ev[4].record(stream)
        flush.fill_(2)
        if ev is not None:
            ev[5].record(stream)
        b.combine(y, d.tok2row, wts, out=out)
        if ev is not None:
            ev[6].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    clocks.mark("start")
    t_all0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_all1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("stop")
    barrier(world)
    clocks.stop()

    route_ms = [e[0].elapsed_time(e[1]) for e in evs]
    disp_ms = [e[2].elapsed_time(e[3]) for e in evs]
    exp_ms = [e[3].elapsed_time(e[4]) for e in evs]
    comb_ms = [e[5].elapsed_time(e[6]) for e in evs]
    total_ms = t_all0.elapsed_time(t_all1)
    dc_us = statistics.mean(a + c for a, c in zip(disp_ms, comb_ms)) * 1e3
    dc_us_max = max_over_ranks(dc_us, world, dev)
    step_ms_max = max_over_ranks(total_ms / args.steps, world, dev)

    # everything after the timed region (warm-L2 calls, end to end through host memory, the
    # "next" rows, the other workloads) is skipped with --kernels-only, which profiling uses
    unflushed = e2e_us = e2e_serial_us = x_h = lg_h = out_h = None
    next_rows, others = {}, {}
    if not args.kernels_only:
        # the same calls with the L2 left warm (no flush between them), outside the timed region
        uev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(20)]
        for e in uev:
            e[0].record(stream)
            b.dispatch(x, idx, B, E, fp8=w.fp8, out=d)
            e[1].record(stream)
            e[2].record(stream)
            b.combine(y, d.tok2row, wts, out=out)
            e[3].record(stream)
        torch.cuda.synchronize()
        unflushed = {"dispatch": statistics.mean(e[0].elapsed_time(e[1]) for e in uev[2:]) * 1e3,
                     "combine": statistics.mean(e[2].elapsed_time(e[3]) for e in uev[2:]) * 1e3,
                     "note": "back-to-back calls without an L2 flush; the expert stand-in does not run between them"}

        # end to end through the public API: pinned host inputs -> device -> layer -> pinned host output.
        # Serial: one layer after another on one stream.  Pipelined (HostLayerPipeline): the input copy
        # of layer i+1 and the output copy of layer i-1 overlap the compute of layer i.
        from combine_moe_route_gb300.pipeline import HostLayerPipeline
        x_h = inp["x"].pin_memory()
        lg_h = torch.from_numpy(inp["logits"]).pin_memory()
        out_h = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        e2e_steps = max(3, min(args.steps, 20))

        def e2e_step():
            x.copy_(x_h, non_blocking=True)
            logits.copy_(lg_h, non_blocking=True)
            b.route_topk(logits, K, topk_idx=idx, topk_w=wts)
            b.dispatch(x, idx, B, E, fp8=w.fp8, out=d)
            b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E, out=y)
            b.combine(y, d.tok2row, wts, out=out)
            out_h.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_serial_us = max_over_ranks(e0.elapsed_time(e1) * 1e3 / e2e_steps, world, dev)

        pipe = HostLayerPipeline(B, E, K, H, fp8=w.fp8, device=dev, depth=2)
        outs_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        for i in range(2):
            pipe.submit(x_h, lg_h, outs_h[i % 2])
        pipe.synchronize()
        barrier(world)
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(pipe.h2d)
        for i in range(e2e_steps):
            pipe.submit(x_h, lg_h, outs_h[i % 2])
        p1.record(pipe.d2h)
        pipe.synchronize()
        e2e_us = max_over_ranks(p0.elapsed_time(p1) * 1e3 / e2e_steps, world, dev)
        del pipe

        # the "next" rows, each timed on its own after the main region (not part of value)
        next_rows = {}
        if E % 8 == 0 and K <= 4 * (E // 8):
            g_idx = torch.empty_like(idx)
            g_w = torch.empty_like(wts)

            def grouped():
                b.route_topk_grouped(logits, K, 8, 4, topk_idx=g_idx, topk_w=g_w)

            us = time_call(grouped, stream, reps=50)
            next_rows["route_grouped_G8_M4"] = {"us": us, "GBps": route_bytes(T, E, K) / (us * 1e-6) / 1e9}

        next_rows.update(measure_partial_combine(b, y, d, idx, wts, out, E, w.R, K, H, T, stream, flush))
        next_rows.update(measure_eager_layers(dev, stream))
        peak_gbs, _ = measured_peaks()
        split = {}
        if args.tokens_per_rank is None:
            split[args.workload] = measure_split_halves(args.workload, dev, stream, flush)
            if args.workload != "dsv3_decode":
                split["dsv3_decode"] = measure_split_halves("dsv3_decode", dev, stream, flush)
        next_rows["split_halves"] = split
        # every other workload, each on its own (parity cases of the same path, not the headline)
        others = {}
        if args.tokens_per_rank is None and not args.headline_only:
            for name in ("toy", "dsv3_decode", "kimi_decode", "wide_ep_decode", "dsv3_prefill"):
                if name != args.workload:
                    others[name] = measure_workload(name, dev, stream, flush, peak_gbs)
                    torch.cuda.empty_cache()

    # correctness of what was timed: the last step's outputs equal the first layer's
    st, code = b.get_device_error(d.workspace)
    if st != 0:
        raise RuntimeError(f"device error word {code:#x} during the timed steps")

    if rank != 0:
        return

    peak, peak_kind = measured_peaks()
    db = dispatch_bytes(T, E, w.R, K, H, w.fp8)
    cb = combine_bytes(T, K, H)
    d_us = statistics.mean(disp_ms) * 1e3
    c_us = statistics.mean(comb_ms) * 1e3
    r_us = statistics.mean(route_ms) * 1e3
    d_gbs = db / (d_us * 1e-6) / 1e9
    c_gbs = cb / (c_us * 1e-6) / 1e9
    if c_us >= d_us:
        dom = {"kernel": "combine_kernel (moe_combine, 1 launch)", "bytes": cb, "us": c_us,
               "traffic": profile_traffic("combine.cu", "combine_dsv3_prefill.md")}
    else:
        dom = {"kernel": "moe_dispatch (hist + scan + scatter launches)", "bytes": db, "us": d_us,
               "traffic": profile_traffic("dispatch.cu", "scatter_dsv3_prefill.md")}
    achieved = dom["bytes"] / (dom["us"] * 1e-6) / 1e9
    cpu = cpu_baseline(args.workload, T) if (world == 1 and not args.no_cpu_baseline) else None
    if args.tokens_per_rank is not None:
        line_note = f"tokens_per_rank overridden to {args.tokens_per_rank} (not the benchmark workload)"
    else:
        line_note = None
    clk = clocks.summary()
    load = routing_load(d.counts.cpu().numpy(), E, w.R)
    line = {
        "metric": METRIC,
        "value": replica_value(dc_us_max, world),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms_max,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": path_dtype(w),
        "data": "synthetic (seeded N(0,1) tokens and router logits, see combine_moe_route_gb300/workloads.py)",
        "config": bench_config(w, T, L2_NOTE, args.tokens_per_rank),
        "roofline": {"bound": "hbm", "kernel": dom["kernel"], "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} (hbm_gbs)", "unit": "GB/s", "frac": achieved / peak,
                     "traffic": dom["traffic"], "algorithmic_bytes": dom["bytes"]},
        "kernels_us": {"route": r_us, "dispatch": d_us, "expert_stand_in": statistics.mean(exp_ms) * 1e3,
                       "combine": c_us},
        "hbm": {"dispatch_GBps": d_gbs, "dispatch_pct_of_8TBs": 100 * d_gbs / NOMINAL_HBM_GBS,
                "combine_GBps": c_gbs, "combine_pct_of_8TBs": 100 * c_gbs / NOMINAL_HBM_GBS,
                "dispatch_frac_of_measured": d_gbs / peak, "combine_frac_of_measured": c_gbs / peak,
                "route_GBps": route_bytes(T, E, K) / (r_us * 1e-6) / 1e9},
        "routing_load": load,
        "p50_us": {"dispatch": statistics.median(disp_ms) * 1e3, "combine": statistics.median(comb_ms) * 1e3},
        "p10_p90_us": {"dispatch": pct(disp_ms), "combine": pct(comb_ms)},
        "unflushed_us": unflushed,
        "e2e": None if e2e_us is None else {
                "value": replica_value(e2e_us, world), "unit": UNIT,
                "h2d_bytes_per_step": int(x_h.numel() * 2 + lg_h.numel() * 4),
                "d2h_bytes_per_step": int(out_h.numel() * 2),
                "serial_us": replica_value(e2e_serial_us, world),
                "note": "per layer: tokens and logits host->device, route + dispatch + expert stand-in + combine, "
                        "output device->host, through the package API; value: HostLayerPipeline (copies of "
                        "neighbouring layers overlap the compute), serial_us: one stream"},
        # per step: route, dispatch (prep + one kernel up to 16384 (token, slot) items, else
        # histogram + scan + scatter), expert stand-in, combine
        "gpu_launches": (3 + (2 if T * K <= 16384 else 3)) * args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"], "window": clk["window"]},
        "cpu_baseline": cpu,
        "workloads": others,
        "next_rows": next_rows,
    }
    if line_note:
        line["note"] = line_note
    print(json.dumps(line))


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="dsv3_prefill")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--headline-only", action="store_true",
                   help="skip the per-workload measurements of the other four layers")
    p.add_argument("--kernels-only", action="store_true",
                   help="only the timed steps (no end-to-end, next-row or other-workload measurements): "
                        "a small device footprint for profiling")
    p.add_argument("--tokens-per-rank", type=int, default=None,
                   help="override B (every rank) for a smaller case of the workload, e.g. for ncu captures")
    args = p.parse_args()
    args.warmup = max(3, args.warmup)        # at least 3 untimed warm-up steps
    world, rank, local = dist_init()
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
