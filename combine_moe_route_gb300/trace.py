"""Phase timeline of dispatch and combine, from a build of the library with -DMOE_TRACE.

    python -m combine_moe_route_gb300.trace [WORKLOAD ...] [--reps N] [--path one|three|both]

The traced build stamps %globaltimer at each phase boundary of the dispatch kernels
(histogram, scan, scatter; or the one-kernel path's prep, staging, counting, layout and
stores) and at the start and end of every combine block, keeping the earliest and the
latest stamp of each phase.  For each workload this prints, per dispatch path, the median
over ``reps`` calls of each phase's first and last stamp in microseconds from the call's
first stamp, next to the call's CUDA-event time; the L2 is flushed (a 256 MiB write)
before every call, as in the benchmark.  The default library is not touched: the traced
build goes to its own folder and the package functions are routed through it only here.
It needs a GPU.
"""
from __future__ import annotations

import argparse
import ctypes
import functools
import os
import statistics

import torch

from . import binding as b
from . import build
from . import workloads as wl

DISPATCH_PHASES = {
    0: "prep kernel starts", 2: "block starts", 36: "routing table staged", 4: "counting done",
    6: "layout done", 8: "row stores issued", 10: "warp done",
    12: "histogram block starts", 14: "histogram block done", 16: "scan block starts",
    18: "scan wait returned", 20: "scan ticket taken", 22: "scan loads and local scan done",
    24: "scan lookback done", 26: "scan block done", 28: "scatter block starts",
    30: "scatter wait returned", 32: "scatter row stores issued", 34: "scatter warp done",
}
COMBINE_PHASES = {0: "combine block starts", 2: "combine block done"}
SLOTS = 48
UNSET = (1 << 64) - 1
FLUSH_BYTES = 256 << 20


@functools.lru_cache(maxsize=None)
def traced_library(three_kernel: bool) -> ctypes.CDLL:
    """Build (once per folder) and load the traced library; three_kernel forces the
    histogram / scan / scatter path for every batch size."""
    defines = ("MOE_TRACE",) + (("MOE_SMALL_DISPATCH_ITEMS=0",) if three_kernel else ())
    out = os.path.join(build.PKG, "_build", "trace_three" if three_kernel else "trace_one")
    return b.load_library(build.build(out_dir=out, defines=defines))


def _phases(raw, names):
    """µs of each phase's first and last stamp from the call's first stamp."""
    mins = [raw[i] for i in range(0, SLOTS, 2) if raw[i] != UNSET]
    if not mins:
        return {}
    t0 = min(mins)
    out = {}
    for slot, name in names.items():
        if raw[slot] != UNSET:
            out[name] = ((raw[slot] - t0) / 1e3, (raw[slot + 1] - t0) / 1e3)
    return out


def timeline(workload: str, three_kernel: bool, reps: int = 25, device=None) -> dict:
    """Median phase times of ``reps`` flushed calls of dispatch and of combine."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    lib = traced_library(three_kernel)
    w = wl.WORKLOADS[workload]
    inp = wl.generate(w, seed=0)
    B, E, K = inp["B"], w.E, w.K
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    buf = (ctypes.c_ulonglong * SLOTS)()
    result = {}
    with b.using_library(lib):
        x = inp["x"].to(dev)
        lg = torch.from_numpy(inp["logits"]).to(dev)
        idx, wts = b.route_topk(lg, K)
        d = b.dispatch(x, idx, B, E, fp8=w.fp8)
        y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E)
        out = b.combine(y, d.tok2row, wts)
        torch.cuda.synchronize(dev)
        calls = {"dispatch": (lambda: b.dispatch(x, idx, B, E, fp8=w.fp8, out=d), lib.moe_trace_dispatch,
                              DISPATCH_PHASES),
                 "combine": (lambda: b.combine(y, d.tok2row, wts, out=out), lib.moe_trace_combine,
                             COMBINE_PHASES)}
        for name, (call, reader, names) in calls.items():
            runs, events = [], []
            for _ in range(reps):
                if reader(1, None) != 0:
                    raise RuntimeError("trace reset failed")
                flush.fill_(1)
                a = torch.cuda.Event(enable_timing=True)
                z = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                call()
                z.record(stream)
                torch.cuda.synchronize(dev)
                if reader(0, ctypes.cast(buf, ctypes.c_void_p)) != 0:
                    raise RuntimeError("trace read failed")
                runs.append(_phases(list(buf), names))
                events.append(a.elapsed_time(z) * 1e3)
            phases = {}
            for ph in names.values():
                got = [r[ph] for r in runs if ph in r]
                if got:
                    phases[ph] = (statistics.median(v[0] for v in got), statistics.median(v[1] for v in got))
            result[name] = {"event_us": statistics.median(events), "phases": phases}
    return result


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("workloads", nargs="*", default=["dsv3_decode"], choices=sorted(wl.WORKLOADS))
    ap.add_argument("--reps", type=int, default=25)
    ap.add_argument("--path", choices=["one", "three", "both"], default="both",
                    help="dispatch path: the library's choice (one), always three kernels, or both")
    args = ap.parse_args(argv)
    paths = {"one": [False], "three": [True], "both": [False, True]}[args.path]
    for name in args.workloads:
        for three in paths:
            label = "three-kernel dispatch forced" if three else "library's dispatch path"
            res = timeline(name, three, args.reps)
            print(f"## {name}: {label}\n")
            for call, r in res.items():
                print(f"{call}: CUDA-event time {r['event_us']:.2f} µs (median of {args.reps})\n")
                print("| phase | first µs | last µs |\n|---|---|---|")
                for ph, (lo, hi) in sorted(r["phases"].items(), key=lambda kv: kv[1][0]):
                    print(f"| {ph} | {lo:.2f} | {hi:.2f} |")
                print()


if __name__ == "__main__":
    main()
