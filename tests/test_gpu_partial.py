"""GPU parity of combine with sender-side partial accumulation
(moe_combine_partial_send / _recv) against the oracle on the same inputs:
the partial rows (one per token and expert rank) and the summed outputs,
bit for bit."""
import numpy as np
import pytest
import torch

from _compare import bits16, f32, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _check(gpu, oracle, inp, E, K, fp8):
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    B, T = inp["B"], inp["T"]
    R = len(B)
    x = inp["x"].to(gpu)
    o_idx, o_w = oracle.route_topk(inp["logits"], K)
    idx = torch.from_numpy(o_idx).to(gpu)
    wg = torch.from_numpy(o_w).to(gpu)
    d = b.dispatch(x, idx, B, E, fp8=fp8)
    y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E)
    part = b.combine_partial_send(y, d.tok2row, idx, wg, E, R)
    o16 = b.combine_partial_recv(part, idx, E, R)
    o32 = b.combine_partial_recv(part, idx, E, R, out_dtype=torch.float32)
    torch.cuda.synchronize()
    od = oracle.dispatch(wl.bf16_bits(inp["x"]), o_idx, B, E, fp8=fp8)
    oy = oracle.expert_scale(od["recv"], od["recv_scale"], od["expert_offsets"], E)
    ref32 = oracle.combine_partial(oy, od["tok2row"], o_idx, o_w, E, R, out="f32")
    ref16, ref_part = oracle.combine_partial(oy, od["tok2row"], o_idx, o_w, E, R, out="bf16", with_partial=True)
    assert np.array_equal(f32(o32).view(np.uint32), ref32.view(np.uint32))
    assert np.array_equal(bits16(o16), ref16)
    # the partial rows that would travel: slot of each (token, rank)'s first copy
    L = E // R
    ranks = o_idx // L
    first = np.ones_like(ranks, dtype=bool)
    for j in range(1, K):
        first[:, j] = ~np.any(ranks[:, :j] == ranks[:, j:j + 1], axis=1)
    slots = np.nonzero(first.reshape(-1))[0]
    sl = torch.from_numpy(slots.astype(np.int64)).to(gpu)
    assert np.array_equal(bits16(part.index_select(0, sl)), ref_part[slots])


@pytest.mark.parametrize("name", ["toy", "dsv3_decode", "dsv3_prefill", "wide_ep_decode"])
def test_partial_workloads(name, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    _check(gpu, oracle, wl.generate(w, seed=0), w.E, w.K, w.fp8)


@pytest.mark.parametrize("R,E,K,H,B", [
    (1, 8, 4, 256, [33]),                     # one rank: equals the receive-side combine
    (4, 32, 32, 128, [5, 0, 9, 1]),           # K = E: every rank gets a run of 8 copies
    (16, 64, 6, 512, [3] * 16),
])
def test_partial_small_shapes(R, E, K, H, B, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    _check(gpu, oracle, wl.random_shape_inputs(R, E, K, H, B, seed=E + K), E, K, False)
