"""The traced build (-DMOE_TRACE): same outputs as the default library, phases in order.

`combine_moe_route_gb300.trace` builds the library with %globaltimer stamps at the
phase boundaries of dispatch and combine.  The stamps must not change any output, and the
phases they report must come in the order the kernels run them."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def trace_mod(gpu):
    from combine_moe_route_gb300 import trace
    return trace


def _layer(b, inp, w, dev):
    x = inp["x"].to(dev)
    lg = torch.from_numpy(inp["logits"]).to(dev)
    idx, wts = b.route_topk(lg, w.K)
    d = b.dispatch(x, idx, inp["B"], w.E, fp8=w.fp8)
    y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, w.E)
    out = b.combine(y, d.tok2row, wts)
    torch.cuda.synchronize(dev)
    return [t.cpu() for t in (idx, wts, d.recv_x.view(torch.uint8), d.tok2row, d.row2src, d.counts, d.offsets, out)]


@pytest.mark.parametrize("three_kernel", [False, True])
def test_traced_build_matches_default(trace_mod, three_kernel, gpu):
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS["dsv3_decode"]
    inp = wl.generate(w, seed=0)
    ref = _layer(b, inp, w, gpu)
    with b.using_library(trace_mod.traced_library(three_kernel)):
        got = _layer(b, inp, w, gpu)
    for r, g in zip(ref, got):
        assert torch.equal(r, g)


def _in_order(phases, names):
    firsts = [phases[n][0] for n in names]
    assert firsts == sorted(firsts), dict(zip(names, firsts))
    for n in names:
        assert phases[n][0] <= phases[n][1]


def test_one_kernel_phases_in_order(trace_mod, gpu):
    res = trace_mod.timeline("dsv3_decode", three_kernel=False, reps=3, device=gpu)
    ph = res["dispatch"]["phases"]
    _in_order(ph, ["prep kernel starts", "block starts", "routing table staged", "counting done", "layout done",
                   "row stores issued", "warp done"])
    assert ph["warp done"][1] > 5.0                       # 132 MB do not move in 5 µs
    c = res["combine"]["phases"]
    _in_order(c, ["combine block starts", "combine block done"])


def test_three_kernel_phases_in_order(trace_mod, gpu):
    res = trace_mod.timeline("dsv3_decode", three_kernel=True, reps=3, device=gpu)
    ph = res["dispatch"]["phases"]
    _in_order(ph, ["histogram block starts", "histogram block done", "scan wait returned", "scan ticket taken",
                   "scan loads and local scan done", "scan lookback done", "scan block done",
                   "scatter wait returned", "scatter row stores issued", "scatter warp done"])
    # the scan waits for the whole histogram grid, the scatter for the whole scan grid
    assert ph["scan wait returned"][0] >= ph["histogram block done"][1]
    assert ph["scatter wait returned"][0] >= ph["scan block done"][1]
