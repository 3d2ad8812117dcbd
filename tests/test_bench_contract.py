"""bench.py's output contract, on the CPU.

The GPU arm needs a GPU; what can be checked here is the reference arm (the
CPU oracle timed on a sample of the workload), its behaviour under two ranks,
and the GPU arm's host-side pieces: the algorithmic-byte accounting that the
roofline fraction divides by, the ncu traffic lookup, the clock summary, the
CPU-baseline object and the routing-load summary."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CONTRACT_KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _json_lines(text):
    out = []
    for line in text.splitlines():
        line = line.strip()
        if line.startswith("{"):
            out.append(json.loads(line))
    return out


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "toy", "--steps", "2",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert CONTRACT_KEYS <= set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is False and d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["unit"] == "us/layer" and d["value"] > 0
    assert d["config"]["workload"] == "toy"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_warmup_is_at_least_three():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "toy", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    (d,) = _json_lines(r.stdout)
    assert d["warmup"] == 3


def test_reference_arm_under_two_ranks_prints_once():
    # torchrun with two gloo ranks on this host: rank 0 alone times the oracle
    # and prints; rank 1 exits 0 without work.  On a machine with a GPU the
    # ranks would take NCCL and one GPU each, so it needs two there.
    import torch
    if torch.cuda.is_available() and torch.cuda.device_count() < 2:
        pytest.skip("two ranks on a CUDA machine need two GPUs")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--workload", "toy",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


@pytest.mark.parametrize("name", ["dsv3_decode", "dsv3_prefill"])
def test_algorithmic_bytes_of_the_deepseek_layers(name):
    # The per-layer bytes each call must move, term by term: the source rows
    # read once, K copies written once (1 byte per channel in FP8, 2 in bf16),
    # the fp32 scale per 128 channels, the routing read, both maps written and
    # the count matrices; the combine reads K bf16 rows per token, writes one,
    # and reads the weights and the gather map.
    sys.path.insert(0, ROOT)
    import bench
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    T = int(wl.draw_B(w, 0).sum())
    assert T == (32768 if name == "dsv3_prefill" else 1024)
    rows = T * w.K
    src = T * w.H * 2
    copies = rows * w.H * (1 if w.fp8 else 2)
    scales = rows * (w.H // 128) * 4 if w.fp8 else 0
    maps = rows * 4 + 2 * rows * 4 + 2 * w.E * w.R * 4
    assert bench.dispatch_bytes(T, w.E, w.R, w.K, w.H, w.fp8) == src + copies + scales + maps
    assert bench.combine_bytes(T, w.K, w.H) == rows * w.H * 2 + T * w.H * 2 + 2 * rows * 4
    # the figures quoted beside the measurements, in MB
    want = {"dsv3_prefill": (2410.7, 4230.0), "dsv3_decode": (132.2, 132.2)}[name]
    assert round(bench.dispatch_bytes(T, w.E, w.R, w.K, w.H, w.fp8) / 1e6, 1) == want[0]
    assert round(bench.combine_bytes(T, w.K, w.H) / 1e6, 1) == want[1]


def test_routing_load_summary():
    sys.path.insert(0, ROOT)
    import bench
    # E = 4 experts on R = 2 ranks; counts[e*R + s]
    counts = np.array([3, 1,    # expert 0: 4 rows
                       0, 0,    # expert 1: 0
                       2, 2,    # expert 2: 4
                       4, 0])   # expert 3: 4
    got = bench.routing_load(counts, 4, 2)
    assert got["rows_per_expert"] == {"max": 4, "min": 0, "mean": 3.0, "max_over_mean": 4 / 3}
    # destination rank 0 holds experts 0-1 (4 rows), rank 1 experts 2-3 (8 rows)
    assert got["rows_per_dest_rank"] == {"max": 8, "min": 4, "mean": 6.0, "max_over_mean": 8 / 6}
    assert bench.routing_load(np.zeros(8, np.int32), 4, 2)["rows_per_expert"]["max_over_mean"] is None


def test_routing_load_shows_the_zipf_skew(oracle):
    # the Kimi-K2-style workload adds a Zipf(1.2) bias per expert to the logits,
    # so its rows pile onto a few experts; the toy workload's N(0,1) logits do not
    sys.path.insert(0, ROOT)
    import bench
    from combine_moe_route_gb300 import workloads as wl
    ratios = {}
    for name in ("toy", "kimi_decode"):
        w = wl.WORKLOADS[name]
        inp = wl.generate(w, 0)
        idx, _ = oracle.route_topk(inp["logits"], w.K)
        d = oracle.dispatch(np.zeros((inp["T"], 8), np.uint16), idx, inp["B"], w.E)   # counts need no payload
        load = bench.routing_load(d["counts"], w.E, w.R)
        assert load["rows_per_expert"]["mean"] * w.E == inp["T"] * w.K
        ratios[name] = load["rows_per_expert"]["max_over_mean"]
    assert ratios["toy"] < 2.0 < 10.0 < ratios["kimi_decode"]


def test_gpu_arm_cpu_baseline_object(oracle):
    # the GPU arm's cpu_baseline leg runs only the oracle, so it can be checked here
    sys.path.insert(0, ROOT)
    import bench
    from combine_moe_route_gb300 import workloads as wl
    T = int(wl.draw_B(wl.WORKLOADS["toy"], 0).sum())
    cb = bench.cpu_baseline("toy", T)
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["unit"] == "us/layer" and cb["value"] > 0
    assert "toy" in cb["sample"] and f"of {T}" in cb["sample"]
    assert cb["host"]["nproc"] >= 1 and cb["host"]["model"]
    json.dumps(cb)


def test_profile_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    # the roofline's traffic comes from a committed ncu summary, and only while the
    # kernel source still has the hash recorded there
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    src_dir = tmp_path / "combine_moe_route_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src_dir / "k.cu").write_text("__global__ void k() {}\n")
    sha = hashlib.sha256((src_dir / "k.cu").read_bytes()).hexdigest()
    (tmp_path / "profiles" / "k.md").write_text(
        f"# k\n\n- dram_bytes_per_full_launch: 1234\n- kernel_source_sha256: {sha}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k.cu", "k.md") == 1234.0
    (src_dir / "k.cu").write_text("__global__ void k() { }\n")     # the kernel changed since the capture
    assert bench.profile_traffic("k.cu", "k.md") is None
    assert bench.profile_traffic("k.cu", "missing.md") is None


def test_clock_summary_reads_the_timed_window():
    # nvidia-smi rows (index, sm MHz, max sm MHz, power, hw_slowdown, hw_thermal,
    # sw_thermal, sw_power_cap), stamped by arrival; only rows inside the timed
    # region count, and a reason counts when it reads "Active"
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    rows = [(0.0, "0, 1200, 2070, 300.0, Not Active, Not Active, Not Active, Not Active"),    # warm-up
            (1.0, "0, 2070, 2070, 900.0, Not Active, Not Active, Not Active, Active"),
            (1.1, "0, 2055, 2070, 950.0, Not Active, Not Active, Not Active, Not Active"),
            (1.2, "0, 2040, 2070, 990.0, Not Active, Not Active, Not Active, Active"),
            (1.3, "[N/A], garbage"),
            (9.0, "0, 900, 2070, 200.0, Active, Not Active, Not Active, Not Active")]         # after
    c.lines = list(rows)
    c.t_start, c.t_stop = 0.95, 1.25
    got = c.summary()
    assert got["sm_mhz"] == 2055.0 and got["sm_max_mhz"] == 2070.0 and got["samples"] == 3
    assert got["reasons"] == ["sw_power_cap"] and got["window"] == "timed"
    # a timed region shorter than the sampling period falls back to every row
    c.t_start, c.t_stop = 5.0, 5.01
    got = c.summary()
    assert got["samples"] == 5 and "hw_slowdown" in got["reasons"] and got["window"].startswith("warmup")
    c.lines = []
    assert bench.ClockSampler(0).summary()["samples"] == 0
