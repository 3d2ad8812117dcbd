"""GPU parity of the low-latency (fixed-rectangle) layout: moe_dispatch_ll,
moe_combine_ll and the push-style return moe_combine_ll_push, against the
oracle on the same seeded inputs.  Bit-exact: counts, maps, payload bytes and
scales; the expert stand-in; both combine forms (same fma chain)."""
import numpy as np
import pytest
import torch

from _compare import bits16, bytes8, f32, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _check(gpu, oracle, inp, E, K, C, fp8):
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    B, T, H = inp["B"], inp["T"], inp["x"].shape[1]
    R = len(B)
    x = inp["x"].to(gpu)
    logits = torch.from_numpy(inp["logits"]).to(gpu)
    idx, w = b.route_topk(logits, K)
    d = b.dispatch_ll(x, idx, B, E, C, fp8=fp8)
    eo = torch.arange(E + 1, dtype=torch.int32, device=gpu) * (R * C)
    y = b.expert_scale(d.recv_x, d.recv_scale, eo, E)
    torch.cuda.synchronize()
    st, code = b.get_device_error(d.workspace)
    assert st == 0 and code == 0

    o_idx, o_w = oracle.route_topk(inp["logits"], K)
    assert np.array_equal(i32(idx), o_idx)
    x_bits = wl.bf16_bits(inp["x"])
    ll = oracle.dispatch_ll(x_bits, o_idx, B, E, C, fp8=fp8)
    t2r = i32(d.tok2row)
    assert np.array_equal(i32(d.counts), ll["counts"])
    assert np.array_equal(t2r, ll["tok2row"])
    assert np.array_equal(i32(d.row2src)[t2r], ll["row2src"][t2r])
    tr = torch.from_numpy(t2r.astype(np.int64)).to(gpu)
    if fp8:
        assert np.array_equal(bytes8(d.recv_x.view(torch.uint8).index_select(0, tr)), ll["recv"][t2r])
        assert np.array_equal(f32(d.recv_scale.index_select(0, tr)).view(np.uint32),
                              ll["recv_scale"][t2r].view(np.uint32))
    else:
        assert np.array_equal(bits16(d.recv_x.index_select(0, tr)), ll["recv"][t2r])
    # expert outputs of the filled rows equal the throughput layout's for the same copies
    rg = oracle.dispatch(x_bits, o_idx, B, E, fp8=fp8)
    yr = oracle.expert_scale(rg["recv"], rg["recv_scale"], rg["expert_offsets"], E)
    assert np.array_equal(bits16(y.index_select(0, tr)), yr[rg["tok2row"]])
    # combine: gather over the rectangle, and push + origin-side sum; both equal the oracle
    wg = torch.from_numpy(o_w).to(gpu)
    ref = oracle.combine(yr, rg["tok2row"], o_w, out="f32")
    g32 = b.combine_ll(y, E, R, C, d.tok2row, wg, out_dtype=torch.float32)
    ret = b.combine_ll_push(y, d, R, E, T, K)
    p32 = b.combine(ret, None, wg, out_dtype=torch.float32)
    g16 = b.combine_ll(y, E, R, C, d.tok2row, wg)
    torch.cuda.synchronize()
    assert np.array_equal(f32(g32).view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(f32(p32).view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(bits16(g16), oracle.bf16_from_f32(ref))


@pytest.mark.parametrize("name,C", [("dsv3_decode", 128), ("kimi_decode", 64), ("wide_ep_decode", 32)])
def test_ll_decode_workloads(name, C, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    assert int(inp["B"].max()) <= C
    _check(gpu, oracle, inp, w.E, w.K, C, fp8=False)


@pytest.mark.parametrize("R,E,K,H,B,C,fp8", [
    (8, 256, 8, 7168, [128] * 8, 128, True),            # DSv3 decode shape with the FP8 payload
    (4, 16, 4, 256, [300, 0, 257, 5], 300, False),      # ranks span several 2048-item tiles
    (3, 9, 3, 512, [700, 1, 699], 700, True),           # K = 3: tokens straddle tiles
    (2, 2, 2, 16, [3, 0], 4, False),
])
def test_ll_small_shapes(R, E, K, H, B, C, fp8, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    inp = wl.random_shape_inputs(R, E, K, H, B, seed=R + E + K)
    _check(gpu, oracle, inp, E, K, C, fp8)


def test_ll_rejects_overfull_ranks(gpu):
    from combine_moe_route_gb300 import binding as b
    x = torch.zeros((10, 16), dtype=torch.bfloat16, device=gpu)
    idx = torch.zeros((10, 1), dtype=torch.int32, device=gpu)
    with pytest.raises(b.MoeError):
        b.dispatch_ll(x, idx, [10], 2, 8)                 # 10 tokens on a rank, chunk cap 8


def _check_unordered(gpu, oracle, inp, E, K, C, fp8, calls=2):
    """moe_dispatch_ll_unordered: the order inside a region is free, everything else is fixed.
    Checked against the oracle's ordered low-latency layout: exact counts; every copy in its own
    region below the count; tok2row / row2src inverse; each copy's bytes (and scales) equal to
    the oracle's row for that copy; both combine forms bit-exact."""
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    B, T, H = inp["B"], inp["T"], inp["x"].shape[1]
    R = len(B)
    x = inp["x"].to(gpu)
    logits = torch.from_numpy(inp["logits"]).to(gpu)
    idx, w = b.route_topk(logits, K)
    o_idx, o_w = oracle.route_topk(inp["logits"], K)
    assert np.array_equal(i32(idx), o_idx)
    x_bits = wl.bf16_bits(inp["x"])
    ll = oracle.dispatch_ll(x_bits, o_idx, B, E, C, fp8=fp8)
    rank_of = np.repeat(np.arange(R), B)                      # source rank of every token
    region = (o_idx.astype(np.int64) * R + rank_of[:, None]).reshape(-1)
    d = None
    for _ in range(calls):                                    # the same buffers, called again
        d = b.dispatch_ll(x, idx, B, E, C, fp8=fp8, unordered=True, out=d)
        torch.cuda.synchronize()
        st, code = b.get_device_error(d.workspace)
        assert st == 0 and code == 0
        counts = i32(d.counts)
        assert np.array_equal(counts, ll["counts"])
        t2r = i32(d.tok2row).astype(np.int64)
        slot = t2r - region * C
        assert np.all((slot >= 0) & (slot < counts[region]))   # own region, below its count
        assert np.unique(t2r).size == t2r.size                  # distinct rows
        assert np.array_equal(i32(d.row2src)[t2r], np.arange(T * K))
        tr = torch.from_numpy(t2r).to(gpu)
        lt = ll["tok2row"]
        if fp8:
            assert np.array_equal(bytes8(d.recv_x.view(torch.uint8).index_select(0, tr)), ll["recv"][lt])
            assert np.array_equal(f32(d.recv_scale.index_select(0, tr)).view(np.uint32),
                                  ll["recv_scale"][lt].view(np.uint32))
        else:
            assert np.array_equal(bits16(d.recv_x.index_select(0, tr)), ll["recv"][lt])
    eo = torch.arange(E + 1, dtype=torch.int32, device=gpu) * (R * C)
    y = b.expert_scale(d.recv_x, d.recv_scale, eo, E)
    rg = oracle.dispatch(x_bits, o_idx, B, E, fp8=fp8)
    yr = oracle.expert_scale(rg["recv"], rg["recv_scale"], rg["expert_offsets"], E)
    wg = torch.from_numpy(o_w).to(gpu)
    ref = oracle.combine(yr, rg["tok2row"], o_w, out="f32")
    g32 = b.combine_ll(y, E, R, C, d.tok2row, wg, out_dtype=torch.float32)
    ret = b.combine_ll_push(y, d, R, E, T, K)
    p32 = b.combine(ret, None, wg, out_dtype=torch.float32)
    g16 = b.combine_ll(y, E, R, C, d.tok2row, wg)
    torch.cuda.synchronize()
    assert np.array_equal(f32(g32).view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(f32(p32).view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(bits16(g16), oracle.bf16_from_f32(ref))


@pytest.mark.parametrize("name,C", [("dsv3_decode", 128), ("kimi_decode", 64), ("wide_ep_decode", 32)])
def test_ll_unordered_decode_workloads(name, C, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    _check_unordered(gpu, oracle, inp, w.E, w.K, C, fp8=False)


@pytest.mark.parametrize("R,E,K,H,B,C,fp8", [
    (8, 256, 8, 7168, [128] * 8, 128, True),            # DSv3 decode shape with the FP8 payload
    (4, 16, 4, 256, [300, 0, 257, 5], 300, False),      # a region far larger than one warp's share
    (3, 9, 3, 512, [700, 1, 699], 700, True),
    (2, 2, 2, 16, [3, 0], 4, False),
    (1, 1, 1, 8, [5], 5, False),                        # one rank, one expert: a single region
])
def test_ll_unordered_small_shapes(R, E, K, H, B, C, fp8, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    inp = wl.random_shape_inputs(R, E, K, H, B, seed=R + E + K + 1)
    _check_unordered(gpu, oracle, inp, E, K, C, fp8)


def test_ll_unordered_empty_and_rejects(gpu):
    from combine_moe_route_gb300 import binding as b
    x = torch.zeros((0, 16), dtype=torch.bfloat16, device=gpu)
    idx = torch.zeros((0, 2), dtype=torch.int32, device=gpu)
    d = b.dispatch_ll(x, idx, [0, 0], 4, 2, unordered=True)
    torch.cuda.synchronize()
    assert np.array_equal(i32(d.counts), np.zeros(8, np.int32))
    x = torch.zeros((10, 16), dtype=torch.bfloat16, device=gpu)
    idx = torch.zeros((10, 1), dtype=torch.int32, device=gpu)
    with pytest.raises(b.MoeError):
        b.dispatch_ll(x, idx, [10], 2, 8, unordered=True)  # 10 tokens on a rank, chunk cap 8
