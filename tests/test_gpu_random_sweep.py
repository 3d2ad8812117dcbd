"""A seeded random sweep of small shapes through every dispatch form, against
the oracle on the same inputs.

Each case draws R, E (a multiple of R), K, H, a token count per rank (empty
ranks included), the payload type, the logits' character (random, rounded to
integers for many ties, or skewed by a Zipf bias) and an optional group
limit.  Then:
  * route (plain or group-limited): bit-exact indices, weights within the
    derived bound;
  * ragged dispatch: counts, offsets, maps, payload bytes and scales
    bit-exact; expert stand-in and combine (bf16 and fp32) bit-exact;
  * low-latency dispatch (C = the largest rank): bit-exact against the
    oracle's rectangle; the unordered form on what its contract fixes;
  * split dispatch and combine (send half, then receive half; the send half
    on a random SM budget): layout, payload and outputs bit-exact, device
    error word clear;
  * sender-side partial combine: outputs bit-exact.
The cases are small so that the oracle finishes each in well under a second."""
import numpy as np
import pytest
import torch

from _compare import bits16, bytes8, f32, i32, weight_tolerance

pytestmark = pytest.mark.gpu

N_CASES = 120


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _draw_case(i):
    rng = np.random.default_rng(1000 + i)
    R = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
    L = int(rng.integers(1, 9))                      # experts per rank
    E = R * L
    while E > 1024:
        L -= 1
        E = R * L
    K = int(rng.integers(1, min(E, 32) + 1))
    fp8 = bool(rng.integers(0, 2))
    H = int(rng.choice([128, 256, 384, 640])) if fp8 else int(rng.choice([8, 24, 136, 256, 520]))
    B = rng.integers(0, 200, size=R).astype(np.int32)
    if rng.random() < 0.3:
        B[rng.integers(0, R)] = 0                     # an empty rank
    if B.sum() == 0:
        B[0] = 1                                      # T = 0 has its own test
    kind = str(rng.choice(["random", "ties", "zipf"]))
    G = M = 1
    divisors = [g for g in range(2, min(E, 32) + 1) if E % g == 0]
    if divisors and rng.random() < 0.35:
        G = int(rng.choice(divisors))
        need = -(-K // (E // G))                      # groups needed to hold K experts
        M = int(rng.integers(need, G + 1))
    return dict(R=R, E=E, K=K, H=H, B=B, fp8=fp8, kind=kind, G=G, M=M, seed=2000 + i)


def _inputs(c):
    from combine_moe_route_gb300 import workloads as wl
    inp = wl.random_shape_inputs(c["R"], c["E"], c["K"], c["H"], c["B"], seed=c["seed"], fp8=c["fp8"],
                                 zipf_s=1.2 if c["kind"] == "zipf" else None)
    if c["kind"] == "ties":
        inp["logits"] = np.round(inp["logits"] * 2.0).astype(np.float32)
    return inp


def _poisoned(T, H, E, R, K, fp8, dev):
    """Dispatch outputs filled with values no call writes (NaN rows, e4m3 NaN bytes, -7 maps), so
    that a row or map entry left unwritten cannot match the oracle by chance."""
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
        workspace=torch.full((max(b.dispatch_workspace_bytes(R, E, K, T), 256),), 0xEE, dtype=torch.uint8,
                             device=dev))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i, gpu, oracle):
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    c = _draw_case(i)
    inp = _inputs(c)
    R, E, K, H, B, fp8 = c["R"], c["E"], c["K"], c["H"], inp["B"], c["fp8"]
    T = int(inp["T"])
    x = inp["x"].to(gpu)
    lg = torch.from_numpy(inp["logits"]).to(gpu)
    x_bits = wl.bf16_bits(inp["x"])

    # route
    if c["G"] > 1:
        idx, w = b.route_topk_grouped(lg, K, c["G"], c["M"])
        o_idx, o_w = oracle.route_topk_grouped(inp["logits"], K, c["G"], c["M"])
    else:
        idx, w = b.route_topk(lg, K)
        o_idx, o_w = oracle.route_topk(inp["logits"], K)
    torch.cuda.synchronize()
    assert np.array_equal(i32(idx), o_idx)
    if T:
        sel = np.take_along_axis(inp["logits"], o_idx, axis=1)
        assert np.all(np.abs(f32(w).astype(np.float64) - o_w) <= weight_tolerance(o_w, sel, K))
    wg = torch.from_numpy(o_w).to(gpu)                # both sides combine with the same weights

    # ragged dispatch, expert stand-in, combine
    d = b.dispatch(x, idx, B, E, fp8=fp8, out=_poisoned(T, H, E, R, K, fp8, gpu))
    y = b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E)
    o16 = b.combine(y, d.tok2row, wg)
    o32 = b.combine(y, d.tok2row, wg, out_dtype=torch.float32)
    torch.cuda.synchronize()
    st, code = b.get_device_error(d.workspace)
    assert st == 0 and code == 0
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
    assert np.array_equal(f32(o32).view(np.uint32), ref32.view(np.uint32))
    assert np.array_equal(bits16(o16), oracle.bf16_from_f32(ref32))

    # split halves: dispatch send (on a random SM budget) -> receive; combine send -> receive
    rng = np.random.default_rng(c["seed"])
    ds = b.dispatch_send(x, idx, B, E, fp8=fp8, max_sms=int(rng.choice([0, 1, 7, 38])),
                         out=_poisoned(T, H, E, R, K, fp8, gpu))
    b.dispatch_recv(ds, B, E, K)
    ys = b.expert_scale(ds.recv_x, ds.recv_scale, ds.expert_offsets, E)
    b.combine_send(ds.workspace, R)
    os32 = b.combine_recv(ys, ds.tok2row, wg, ds.workspace, R, out_dtype=torch.float32)
    torch.cuda.synchronize()
    st, code = b.get_device_error(ds.workspace)
    assert st == 0 and code == 0
    for key in ("counts", "offsets", "expert_offsets", "tok2row", "row2src"):
        assert np.array_equal(i32(getattr(ds, key)), od[key]), key
    if fp8:
        assert np.array_equal(bytes8(ds.recv_x), od["recv"])
        assert np.array_equal(f32(ds.recv_scale).view(np.uint32), od["recv_scale"].view(np.uint32))
    else:
        assert np.array_equal(bits16(ds.recv_x), od["recv"])
    assert np.array_equal(f32(os32).view(np.uint32), ref32.view(np.uint32))

    # low-latency layouts, chunk cap = the largest rank
    C = max(1, int(B.max()) if B.size else 1)
    dl = b.dispatch_ll(x, idx, B, E, C, fp8=fp8)
    du = b.dispatch_ll(x, idx, B, E, C, fp8=fp8, unordered=True)
    torch.cuda.synchronize()
    ll = oracle.dispatch_ll(x_bits, o_idx, B, E, C, fp8=fp8)
    assert np.array_equal(i32(dl.counts), ll["counts"])
    assert np.array_equal(i32(du.counts), ll["counts"])
    assert np.array_equal(i32(dl.tok2row), ll["tok2row"])
    if T:
        t2r = ll["tok2row"].astype(np.int64)
        tl = torch.from_numpy(t2r).to(gpu)
        assert np.array_equal(i32(dl.row2src)[t2r], ll["row2src"][t2r])
        payload = (lambda r: bytes8(r.view(torch.uint8))) if fp8 else bits16
        assert np.array_equal(payload(dl.recv_x.index_select(0, tl)), ll["recv"][t2r])
        tu = i32(du.tok2row).astype(np.int64)
        rank_of = np.repeat(np.arange(R), B)
        region = (o_idx.astype(np.int64) * R + rank_of[:, None]).reshape(-1)
        slot = tu - region * C
        assert np.all((slot >= 0) & (slot < ll["counts"][region]))
        assert np.array_equal(i32(du.row2src)[tu], np.arange(T * K))
        assert np.array_equal(payload(du.recv_x.index_select(0, torch.from_numpy(tu).to(gpu))), ll["recv"][t2r])

    # sender-side partial sums
    if T:
        part = b.combine_partial_send(y, d.tok2row, idx, wg, E, R)
        p32 = b.combine_partial_recv(part, idx, E, R, out_dtype=torch.float32)
        torch.cuda.synchronize()
        pref = oracle.combine_partial(oy, od["tok2row"], o_idx, o_w, E, R, out="f32")
        assert np.array_equal(f32(p32).view(np.uint32), pref.view(np.uint32))
