"""Split dispatch and combine (send half, receive half) on the GPU, through the
C ABI, against the CPU oracle on the same inputs.

The halves must give exactly what moe_dispatch and moe_combine give: counts,
offsets, maps, payload bytes and scales bit-exact against the oracle's
dispatch, and the weighted sums bit-exact against its combine (both sides run
the same fp32 fma chain).  The receive halves run on a second stream behind an
event recorded after their send halves (the ordering the header documents),
and the send half on a capped SM budget as well as on every SM.

The receive halves consume the send halves' signals, so a second receive with
no new send has nothing to wait for: its bounded wait runs out after about
2 s, it reports MOE_ERR_TIMEOUT through the workspace's error word, and the
next full layer is correct again.  That is failure detection without a fault:
a signal nothing sets."""
import time

import numpy as np
import pytest
import torch

from _compare import bits16, bytes8, f32, i32

pytestmark = pytest.mark.gpu

OK, TIMEOUT = 0, 5
RECV_TIMEOUT = 0x10


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _poisoned(T, H, E, R, K, fp8, dev):
    from combine_moe_route_gb300 import binding as b
    rows = T * K
    return b.DispatchResult(
        recv_x=(torch.full((rows, H), 0x7F, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn) if fp8
                else torch.full((rows, H), float("nan"), dtype=torch.bfloat16, device=dev)),
        recv_scale=torch.full((rows, H // 128), float("nan"), dtype=torch.float32, device=dev) if fp8 else None,
        counts=torch.full((E * R,), -7, dtype=torch.int32, device=dev),
        offsets=torch.full((E * R + 1,), -7, dtype=torch.int32, device=dev),
        expert_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        tok2row=torch.full((rows,), -7, dtype=torch.int32, device=dev),
        row2src=torch.full((rows,), -7, dtype=torch.int32, device=dev),
        workspace=torch.full((b.dispatch_workspace_bytes(R, E, K, T),), 0xEE, dtype=torch.uint8, device=dev))


def _split_layer(x, idx, wts, B, E, fp8, max_sms, dev):
    """send on one stream; receive on another behind an event; then the combine halves the
    same way.  Returns the dispatch result, the expert outputs and the fp32 and bf16 sums."""
    from combine_moe_route_gb300 import binding as b
    T, H = x.shape
    K = idx.shape[1]
    R = len(B)
    d = _poisoned(T, H, E, R, K, fp8, dev)
    s_send, s_recv = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_send.wait_stream(torch.cuda.current_stream(dev))
    s_recv.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s_send):
        b.dispatch_send(x, idx, B, E, fp8=fp8, max_sms=max_sms, out=d)
        sent = torch.cuda.Event()
        sent.record(s_send)
    with torch.cuda.stream(s_recv):
        s_recv.wait_event(sent)
        b.dispatch_recv(d, B, E, K)
        y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E)
        b.combine_send(d.workspace, R)
        published = torch.cuda.Event()
        published.record(s_recv)
    with torch.cuda.stream(s_send):
        s_send.wait_event(published)
        o32 = b.combine_recv(y, d.tok2row, wts, d.workspace, R, out_dtype=torch.float32)
        b.combine_send(d.workspace, R)                      # the flags are consumed by each receive
        o16 = b.combine_recv(y, d.tok2row, wts, d.workspace, R)
    torch.cuda.synchronize()
    return d, y, o32, o16


def _check_against_oracle(d, y, o32, o16, x_bits, o_idx, o_w, B, E, fp8, oracle):
    from combine_moe_route_gb300 import binding as b
    st, code = b.get_device_error(d.workspace)
    assert st == OK and code == 0, (st, code)
    od = oracle.dispatch(x_bits, o_idx, B, E, fp8=fp8)
    for key in ("counts", "offsets", "expert_offsets", "tok2row", "row2src"):
        assert np.array_equal(i32(getattr(d, key)), od[key]), key
    if fp8:
        assert np.array_equal(bytes8(d.recv_x), od["recv"])
        assert np.array_equal(f32(d.recv_scale).view(np.uint32), od["recv_scale"].view(np.uint32))
    else:
        assert np.array_equal(bits16(d.recv_x), od["recv"])
    oy = oracle.expert_scale(od["recv"], od["recv_scale"], od["expert_offsets"], E)
    assert np.array_equal(bits16(y), oy)
    ref32 = oracle.combine(oy, od["tok2row"], o_w, out="f32")
    g32 = f32(o32)
    assert np.all(np.abs(g32 - ref32) <= 1e-6 * np.abs(ref32))        # the stated gate
    assert np.array_equal(g32.view(np.uint32), ref32.view(np.uint32))  # same fma chain: exact
    assert np.array_equal(bits16(o16), oracle.bf16_from_f32(ref32))


@pytest.mark.parametrize("workload", ["toy", "dsv3_decode", "dsv3_prefill", "kimi_decode", "wide_ep_decode"])
def test_split_halves_on_the_workloads(workload, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    w = wl.WORKLOADS[workload]
    inp = wl.generate(w, seed=0)
    B = inp["B"]
    o_idx, o_w = oracle.route_topk(inp["logits"], w.K)
    x = inp["x"].to(gpu)
    idx = torch.from_numpy(o_idx).to(gpu)
    wts = torch.from_numpy(o_w).to(gpu)
    # every SM, then a capped budget that leaves SMs to other streams
    for max_sms in (0, 76):
        d, y, o32, o16 = _split_layer(x, idx, wts, B, w.E, w.fp8, max_sms, gpu)
        _check_against_oracle(d, y, o32, o16, wl.bf16_bits(inp["x"]), o_idx, o_w, B, w.E, w.fp8, oracle)
        del d, y, o32, o16
        torch.cuda.empty_cache()


@pytest.mark.parametrize("R,E,K,H,B,fp8", [
    (256, 256, 8, 256, [int(v) for v in np.random.default_rng(5).integers(0, 12, 256)], False),   # most ranks
    (256, 1024, 32, 128, [int(v) for v in np.random.default_rng(6).integers(0, 5, 256)], True),
    (1, 8, 2, 16384, [300], False),                                                             # largest H
    (8, 64, 8, 7168, [0, 0, 700, 0, 1, 0, 3000, 0], True),                                      # empty ranks, tiles
    (4, 16, 16, 520, [2049, 0, 5, 1], False),                                                   # K = E
])
def test_split_halves_edge_shapes(R, E, K, H, B, fp8, gpu, oracle):
    from combine_moe_route_gb300 import workloads as wl
    inp = wl.random_shape_inputs(R, E, K, H, B, seed=R + E + K + H, fp8=fp8)
    o_idx, o_w = oracle.route_topk(inp["logits"], K)
    x = inp["x"].to(gpu)
    d, y, o32, o16 = _split_layer(x, torch.from_numpy(o_idx).to(gpu), torch.from_numpy(o_w).to(gpu), inp["B"], E,
                                  fp8, 3, gpu)
    _check_against_oracle(d, y, o32, o16, wl.bf16_bits(inp["x"]), o_idx, o_w, inp["B"], E, fp8, oracle)


def test_split_halves_no_tokens(gpu):
    from combine_moe_route_gb300 import binding as b
    B = np.zeros(4, np.int32)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=gpu)
    idx = torch.empty((0, 2), dtype=torch.int32, device=gpu)
    d = _poisoned(0, 256, 16, 4, 2, False, gpu)
    b.dispatch_send(x, idx, B, 16, out=d)
    b.dispatch_recv(d, B, 16, 2)
    out = b.combine_recv(torch.empty((0, 256), dtype=torch.bfloat16, device=gpu), d.tok2row,
                         torch.empty((0, 2), dtype=torch.float32, device=gpu), d.workspace, 4)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)
    assert torch.all(d.counts == 0) and torch.all(d.offsets == 0) and torch.all(d.expert_offsets == 0)


def test_receive_without_a_new_send_times_out(gpu, oracle):
    """Each receive consumes what its send announced.  A second receive with no send in
    between waits for signals nothing will set: the wait ends after its limit with
    MOE_DEVERR_RECV_TIMEOUT, the call completes, and a full layer afterwards is correct."""
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    R, E, K, H = 4, 16, 2, 256
    inp = wl.random_shape_inputs(R, E, K, H, [40, 0, 17, 9], seed=3)
    o_idx, o_w = oracle.route_topk(inp["logits"], K)
    x = inp["x"].to(gpu)
    idx = torch.from_numpy(o_idx).to(gpu)
    wts = torch.from_numpy(o_w).to(gpu)
    B = inp["B"]
    d = b.dispatch_send(x, idx, B, E)
    b.dispatch_recv(d, B, E, K)
    torch.cuda.synchronize()
    assert b.get_device_error(d.workspace) == (OK, 0)
    counts = d.counts.clone()

    t0 = time.perf_counter()
    b.dispatch_recv(d, B, E, K)                               # nothing announced since
    st, code = b.get_device_error(d.workspace)
    dt = time.perf_counter() - t0
    assert st == TIMEOUT and (code & RECV_TIMEOUT), (st, code)
    assert 1.0 < dt < 60.0
    assert torch.equal(d.counts, counts)                      # the layout is still written, from the scan

    y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E)
    b.combine_send(d.workspace, R)
    b.combine_recv(y, d.tok2row, wts, d.workspace, R)
    t0 = time.perf_counter()
    b.combine_recv(y, d.tok2row, wts, d.workspace, R)        # flags consumed by the first receive
    st, code = b.get_device_error(d.workspace)
    dt = time.perf_counter() - t0
    assert st == TIMEOUT and (code & RECV_TIMEOUT), (st, code)
    assert 1.0 < dt < 60.0

    # the context is still usable, and the next layer (its send clears the error word) is exact
    d2, y2, o32, o16 = _split_layer(x, idx, wts, B, E, False, 0, gpu)
    _check_against_oracle(d2, y2, o32, o16, wl.bf16_bits(inp["x"]), o_idx, o_w, B, E, False, oracle)
