"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the
same seeded inputs.

Bar: routing ids, counts, offsets, maps and dispatched bf16 / e4m3 bytes and
scales bit-exact; the expert stand-in bit-exact; combine within 1e-6 relative
(fp32) or 1 bf16 ulp (bf16) -- and, since both sides run the same fp32 fma
chain in the same order, also bit-exact; router weights within the bound
derived in _compare.weight_tolerance.  Full-size runs use the launch
configuration the benchmark times (the library picks it from the shape)."""
import numpy as np
import pytest
import torch

from _compare import bf16_to_f32, bits16, bytes8, f32, i32, weight_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _wl():
    from combine_moe_route_gb300 import workloads
    return workloads


def _binding():
    from combine_moe_route_gb300 import binding
    return binding


# ---------------------------------------------------------------------------
# full-size workloads
# ---------------------------------------------------------------------------

WORKLOADS = ["toy", "dsv3_decode", "dsv3_prefill", "kimi_decode", "wide_ep_decode"]


@pytest.fixture(scope="module", params=WORKLOADS)
def case(request, gpu, oracle):
    """One full-size workload run on the GPU and through the oracle (once per workload;
    pytest groups the tests that use it by workload)."""
    wl, b = _wl(), _binding()
    w = wl.WORKLOADS[request.param]
    inp = wl.generate(w, seed=0)
    B, E, K = inp["B"], w.E, w.K
    x_bits = wl.bf16_bits(inp["x"])
    x = inp["x"].to(gpu)
    logits = torch.from_numpy(inp["logits"]).to(gpu)

    # every output poisoned first (and guard rows past the receive buffer), so that a row
    # or entry the kernels fail to write cannot pass by holding stale, equal values
    T = int(np.sum(B))
    rows = T * K
    idx = torch.full((T, K), -7, dtype=torch.int32, device=gpu)
    wts = torch.full((T, K), float("nan"), dtype=torch.float32, device=gpu)
    b.route_topk(logits, K, topk_idx=idx, topk_w=wts)
    guard = 64
    recv_all = torch.full(((rows + guard) * w.H * (1 if w.fp8 else 2),), 0xA5, dtype=torch.uint8, device=gpu)
    recv = recv_all[: rows * w.H * (1 if w.fp8 else 2)].view(torch.float8_e4m3fn if w.fp8 else torch.bfloat16)
    d = b.DispatchResult(
        recv_x=recv.view(rows, w.H),
        recv_scale=torch.full((rows, w.H // 128), float("nan"), dtype=torch.float32, device=gpu) if w.fp8 else None,
        counts=torch.full((E * len(B),), -7, dtype=torch.int32, device=gpu),
        offsets=torch.full((E * len(B) + 1,), -7, dtype=torch.int32, device=gpu),
        expert_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=gpu),
        tok2row=torch.full((rows,), -7, dtype=torch.int32, device=gpu),
        row2src=torch.full((rows,), -7, dtype=torch.int32, device=gpu),
        workspace=None)
    d = b.dispatch(x, idx, B, E, fp8=w.fp8, out=d)
    y = torch.full((rows, w.H), float("nan"), dtype=torch.bfloat16, device=gpu)
    b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E, out=y)
    out = torch.full((T, w.H), float("nan"), dtype=torch.bfloat16, device=gpu)
    b.combine(y, d.tok2row, wts, out=out)
    torch.cuda.synchronize()
    st, code = b.get_device_error(d.workspace)
    assert bool((recv_all[rows * w.H * (1 if w.fp8 else 2):] == 0xA5).all())   # guard rows untouched

    o_idx, o_w = oracle.route_topk(inp["logits"], K)
    od = oracle.dispatch(x_bits, o_idx, B, E, fp8=w.fp8)
    oy = oracle.expert_scale(od["recv"], od["recv_scale"], od["expert_offsets"], E)
    yield dict(w=w, inp=inp, B=B, idx=idx, wts=wts, d=d, y=y, out=out, st=st, code=code,
               o_idx=o_idx, o_w=o_w, od=od, oy=oy)
    torch.cuda.empty_cache()


def test_workload_route_dispatch_expert(case):
    r = case
    w, K = r["w"], r["w"].K
    assert r["st"] == 0 and r["code"] == 0

    # route: ids bit-exact, weights within the derived bound
    assert np.array_equal(i32(r["idx"]), r["o_idx"])
    sel = np.take_along_axis(r["inp"]["logits"], r["o_idx"], axis=1)
    tol = weight_tolerance(r["o_w"], sel, K)
    assert np.all(np.abs(f32(r["wts"]).astype(np.float64) - r["o_w"]) <= tol)

    # dispatch: layout and payload bit-exact
    d, od = r["d"], r["od"]
    for key in ("counts", "offsets", "expert_offsets", "tok2row", "row2src"):
        assert np.array_equal(i32(getattr(d, key)), od[key]), key
    if w.fp8:
        assert np.array_equal(bytes8(d.recv_x), od["recv"])
        assert np.array_equal(f32(d.recv_scale).view(np.uint32), od["recv_scale"].view(np.uint32))
    else:
        assert np.array_equal(bits16(d.recv_x), od["recv"])

    # expert stand-in: bit-exact
    assert np.array_equal(bits16(r["y"]), r["oy"])


def test_workload_combine(case, gpu, oracle):
    """Combine on identical inputs (the oracle's weights): fp32 and bf16 outputs."""
    b = _binding()
    r = case
    w_gpu = torch.from_numpy(r["o_w"]).to(gpu)
    o32 = b.combine(r["y"], r["d"].tok2row, w_gpu, out_dtype=torch.float32)
    o16 = b.combine(r["y"], r["d"].tok2row, w_gpu, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref32 = oracle.combine(r["oy"], r["od"]["tok2row"], r["o_w"], out="f32")
    g32 = f32(o32)
    assert np.all(np.abs(g32 - ref32) <= 1e-6 * np.abs(ref32))          # the stated gate
    assert np.array_equal(g32.view(np.uint32), ref32.view(np.uint32))    # same fma chain: exact
    ref16 = oracle.bf16_from_f32(ref32)
    g16 = bits16(o16)
    rf = bf16_to_f32(ref16)
    assert np.all(np.abs(bf16_to_f32(g16) - rf) <= np.abs(rf) * 2.0**-7)
    assert np.array_equal(g16, ref16)


def test_workload_end_to_end(case, oracle):
    """Each side with its own router weights: outputs agree to 1 bf16 ulp plus the weight error."""
    r = case
    ref = oracle.combine(r["oy"], r["od"]["tok2row"], r["o_w"], out="bf16")
    got = bf16_to_f32(bits16(r["out"])).astype(np.float64)
    want = bf16_to_f32(ref).astype(np.float64)
    # sum_j |w_j y_j| bounds how far the weight differences can move the fp32 sum
    T, K = r["o_w"].shape
    yabs = np.abs(bf16_to_f32(r["oy"]))
    mag = np.zeros_like(want)
    t2r = r["od"]["tok2row"].reshape(T, K)
    for j in range(K):
        mag += r["o_w"][:, j:j + 1].astype(np.float64) * yabs[t2r[:, j]]
    tol = np.abs(want) * 2.0**-7 + mag * 4e-6 + 1e-30
    assert np.all(np.abs(got - want) <= tol)


@pytest.mark.parametrize("E,K,G,M,T", [
    (256, 8, 8, 4, 32768),     # DeepSeek-V3-like grouping on the prefill layer's token count
    (256, 8, 1, 1, 4096),      # one group: plain routing
    (256, 8, 8, 8, 4096),      # every group kept: plain routing
    (384, 8, 32, 3, 2048),     # 32 groups of 12
    (64, 6, 16, 2, 1000),      # 16 groups of 4, K = 6 of the 8 kept experts
    (1024, 32, 32, 32, 256),   # limits
    # the 16-byte layout's group forms
    (512, 8, 2, 1, 4096),      # a group is two whole 128-expert blocks
    (256, 8, 2, 1, 4096),      # a group is one whole block
    (128, 4, 32, 8, 4096),     # groups of 4: one lane each
    (256, 8, 16, 8, 4096),     # groups of 16: four lanes
    (384, 8, 12, 4, 2048),     # groups of 32 over three blocks
])
def test_route_grouped(E, K, G, M, T, gpu, oracle):
    b = _binding()
    rng = np.random.default_rng(E + K + G + M)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[: T // 4] = np.round(logits[: T // 4])              # many exact ties in a quarter of the rows
    lg = torch.from_numpy(logits).to(gpu)
    idx, w = b.route_topk_grouped(lg, K, G, M)
    torch.cuda.synchronize()
    o_idx, o_w = oracle.route_topk_grouped(logits, K, G, M)
    assert np.array_equal(i32(idx), o_idx)
    sel = np.take_along_axis(logits, o_idx, axis=1)
    assert np.all(np.abs(f32(w).astype(np.float64) - o_w) <= weight_tolerance(o_w, sel, K))
    if G == 1 or M == G:
        p_idx, p_w = b.route_topk(lg, K)
        assert torch.equal(p_idx, idx) and torch.equal(p_w, w)


@pytest.mark.parametrize("E,K,T", [(1, 1, 70), (5, 3, 300), (31, 7, 500), (33, 8, 500), (100, 32, 400),
                                   (256, 8, 3000), (384, 8, 1200), (1000, 16, 300), (1024, 32, 256)])
def test_route_plain_shapes(E, K, T, gpu, oracle):
    """Plain top-K on rows of every kind: random; rounded (many exact ties, more candidates than
    the shared-memory ranking takes); constant; +0 and -0 mixed; and a row whose K-th and
    (K+1)-th keys tie across lanes."""
    b = _binding()
    rng = np.random.default_rng(E * 7 + K)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    q = T // 5
    logits[q:2 * q] = np.round(logits[q:2 * q])
    logits[2 * q:2 * q + 3] = 1.5
    logits[2 * q + 3] = np.where(rng.random(E) < 0.5, 0.0, -0.0).astype(np.float32)
    if E > K:
        row = rng.standard_normal(E).astype(np.float32)
        top = np.sort(row)[::-1]
        row[row == top[K]] = top[K - 1]                    # the K-th and (K+1)-th keys now tie
        logits[2 * q + 4] = row
    lg = torch.from_numpy(logits).to(gpu)
    idx, w = b.route_topk(lg, K)
    torch.cuda.synchronize()
    o_idx, o_w = oracle.route_topk(logits, K)
    assert np.array_equal(i32(idx), o_idx)
    sel = np.take_along_axis(logits, o_idx, axis=1)
    assert np.all(np.abs(f32(w).astype(np.float64) - o_w) <= weight_tolerance(o_w, sel, K))


# ---------------------------------------------------------------------------
# random small shapes, ragged tails, edge cases
# ---------------------------------------------------------------------------

def _small_case(gpu, oracle, R, E, K, H, B, fp8, seed, identity=False, zipf=None):
    wl, b = _wl(), _binding()
    inp = wl.random_shape_inputs(R, E, K, H, B, seed=seed, fp8=fp8, zipf_s=zipf)
    x_bits = wl.bf16_bits(inp["x"])
    x = inp["x"].to(gpu)
    logits = torch.from_numpy(inp["logits"]).to(gpu)
    r = b.moe_layer(x, logits, inp["B"], E, K, fp8=fp8, identity=identity)
    torch.cuda.synchronize()
    st, code = b.get_device_error(r["dispatch"].workspace)
    assert st == 0 and code == 0
    ref = oracle.layer(x_bits, inp["logits"], inp["B"], E, K, fp8=fp8, identity=identity)
    assert np.array_equal(i32(r["topk_idx"]), ref["topk_idx"])
    d = r["dispatch"]
    for key in ("counts", "offsets", "expert_offsets", "tok2row", "row2src"):
        assert np.array_equal(i32(getattr(d, key)), ref[key]), key
    if fp8:
        assert np.array_equal(bytes8(d.recv_x), ref["recv"])
        assert np.array_equal(f32(d.recv_scale).view(np.uint32), ref["recv_scale"].view(np.uint32))
    else:
        assert np.array_equal(bits16(d.recv_x), ref["recv"])
    assert np.array_equal(bits16(r["y"]), ref["y"])
    # combine on the oracle's weights: exact
    o = b.combine(r["y"], d.tok2row, torch.from_numpy(ref["topk_w"]).to(gpu))
    assert np.array_equal(bits16(o), ref["out"])
    return r, ref


SHAPES = [
    # R, E, K, H, B
    (1, 4, 1, 8, [1]),
    (1, 4, 4, 128, [37]),                      # K == E
    (2, 2, 2, 16, [3, 0]),                     # K == E == R, an empty rank
    (3, 9, 3, 256, [0, 700, 5]),               # K = 3: tokens straddle 2048-item tiles
    (3, 12, 2, 384, [1025, 1024, 1023]),       # odd number of 128-blocks (FP8)
    (2, 8, 2, 1280, [33, 20]),                 # 10 blocks: a full step of the in-place quantiser and a part
    (8, 16, 2, 256, [64, 1, 0, 33, 64, 2, 17, 5]),
    (8, 64, 8, 7168, [300, 0, 1, 257, 0, 0, 512, 3]),
    (4, 1024, 32, 128, [40, 0, 3, 9]),         # E and K at their limits
    (16, 32, 4, 1024, [0] * 15 + [900]),       # all tokens on the last rank
    (128, 256, 8, 512, list(range(0, 128))),   # many ranks, ragged
    (256, 256, 6, 128, [i % 5 for i in range(256)]),
    (8, 1024, 8, 128, [2100] * 8),             # 73728 histogram counts: the decoupled-lookback scan
    (1, 1, 1, 16384, [9]),                     # one expert, one rank, the largest hidden size
    (2, 4, 1, 2048, [0, 37]),                  # K = 1
]


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"R{s[0]}E{s[1]}K{s[2]}H{s[3]}" for s in SHAPES])
def test_small_shapes(shape, fp8, gpu, oracle):
    R, E, K, H, B = shape
    if fp8 and H % 128:
        pytest.skip("FP8 needs H % 128 == 0")
    _small_case(gpu, oracle, R, E, K, H, B, fp8, seed=sum(B) + K)


def test_identity_experts_return_input(gpu, oracle):
    r, ref = _small_case(gpu, oracle, 8, 32, 4, 1024, [17, 3, 0, 90, 2, 2, 40, 1], False, seed=3, identity=True)
    x = bf16_to_f32(bits16(r["dispatch"].recv_x))  # rows are exact copies of x
    out = bf16_to_f32(bits16(r["out"]))
    inp_rows = x[i32(r["dispatch"].tok2row).reshape(-1, 4)[:, 0]]
    assert np.all(np.abs(out - inp_rows) <= np.abs(inp_rows) * 2.0**-7)


def test_zipf_skewed_routing(gpu, oracle):
    _small_case(gpu, oracle, 32, 384, 8, 256, [i % 65 for i in range(32)], False, seed=5, zipf=1.2)


def test_empty_batch(gpu):
    b = _binding()
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=gpu)
    idx = torch.empty((0, 2), dtype=torch.int32, device=gpu)
    d = b.dispatch(x, idx, [0, 0, 0, 0], 16)
    torch.cuda.synchronize()
    assert int(d.counts.abs().sum()) == 0 and int(d.offsets.abs().sum()) == 0
    assert int(d.expert_offsets.abs().sum()) == 0
    o = b.combine(torch.empty((0, 256), dtype=torch.bfloat16, device=gpu), idx.view(-1),
                  torch.empty((0, 2), dtype=torch.float32, device=gpu))
    assert o.shape == (0, 256)


def test_reused_workspace_and_side_stream(gpu, oracle):
    """Back-to-back calls on one workspace (lookback flags re-armed) on a non-default stream."""
    wl, b = _wl(), _binding()
    inp = wl.random_shape_inputs(8, 64, 8, 1024, [200, 3, 0, 77, 512, 9, 1, 64], seed=9)
    x = inp["x"].to(gpu)
    logits = torch.from_numpy(inp["logits"]).to(gpu)
    s = torch.cuda.Stream(gpu)
    with torch.cuda.stream(s):
        idx, _ = b.route_topk(logits, 8)
        d1 = b.dispatch(x, idx, inp["B"], 64, fp8=True)
        snap = [t.clone() for t in (d1.recv_x.view(torch.uint8), d1.tok2row, d1.counts)]
        d2 = b.dispatch(x, idx, inp["B"], 64, fp8=True, out=d1)
    s.synchronize()
    for a, t in zip(snap, (d2.recv_x.view(torch.uint8), d2.tok2row, d2.counts)):
        assert torch.equal(a, t)
    ref = oracle.dispatch(wl.bf16_bits(inp["x"]), i32(idx), inp["B"], 64, fp8=True)
    assert np.array_equal(bytes8(d2.recv_x), ref["recv"])


def test_cuda_graph_replay_matches_eager(gpu):
    wl, b = _wl(), _binding()
    inp = wl.random_shape_inputs(8, 256, 8, 7168, [128] * 8, seed=11)
    x = inp["x"].to(gpu)
    logits = torch.from_numpy(inp["logits"]).to(gpu)
    eager = b.moe_layer(x, logits, inp["B"], 256, 8)
    torch.cuda.synchronize()
    ref_out = eager["out"].clone()
    # static buffers for capture
    idx = torch.empty((1024, 8), dtype=torch.int32, device=gpu)
    wts = torch.empty((1024, 8), dtype=torch.float32, device=gpu)
    d = b.dispatch(x, eager["topk_idx"], inp["B"], 256)      # allocates outputs + workspace
    y = torch.empty_like(eager["y"])
    out = torch.empty_like(ref_out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        b.route_topk(logits, 8, topk_idx=idx, topk_w=wts)
        b.dispatch(x, idx, inp["B"], 256, out=d)
        b.expert_scale(d.recv_x, None, d.expert_offsets, 256, out=y)
        b.combine(y, d.tok2row, wts, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)


# ---------------------------------------------------------------------------
# FP8 codec on the device, exhaustively over bf16 inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("amax", [448.0, 224.0, 3.0625, 1.0, 0.7734375, 2.0**-10, 0.0311279296875, 5.5625,
                                  17.875, 123.0, 300.0, 447.0,
                                  # at and below the 2^-119 amax floor: zero blocks, tiny blocks, subnormals
                                  0.0, 2.0**-70, 2.0**-100, 2.0**-119, float.fromhex("0x1.fep-120"), 2.0**-126,
                                  2.0**-133])
def test_fp8_codec_all_bf16_values(amax, gpu, oracle):
    """Every finite bf16 value v with |v| <= amax, quantised in blocks whose
    largest magnitude is amax (for amax = 448 the multiplier is exactly 1, so
    the device conversion of v itself is checked; for amax below 2^-119 the
    floor sets the scale, and subnormal scales and inputs are exercised)."""
    b = _binding()
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bf16_to_f32(h)
    keep = np.isfinite(v) & (np.abs(v) <= amax)
    vals = h[keep]
    per = 127
    nblk = -(-vals.size // per)
    pad = np.full(nblk * per - vals.size, 0, np.uint16)
    blocks = np.concatenate([vals, pad]).reshape(nblk, per)
    amax_bits = oracle.bf16_from_f32(np.array([amax], np.float32))[0]
    blocks = np.concatenate([blocks, np.full((nblk, 1), amax_bits, np.uint16)], axis=1)
    H = 128 * 8
    rows = -(-nblk // 8)
    xb = np.zeros((rows * 8, 128), np.uint16)
    xb[:nblk] = blocks
    xb = xb.reshape(rows, H)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(gpu)
    idx = torch.zeros((rows, 1), dtype=torch.int32, device=gpu)
    d = b.dispatch(x, idx, [rows], 1, fp8=True)
    torch.cuda.synchronize()
    q, s = oracle.quantize_rows_e4m3(xb)
    assert np.array_equal(bytes8(d.recv_x), q)
    assert np.array_equal(f32(d.recv_scale).view(np.uint32), s.view(np.uint32))


# ---------------------------------------------------------------------------
# device-side routing errors: reported, nothing written out of bounds
# ---------------------------------------------------------------------------

def test_bad_routing_is_reported(gpu):
    b = _binding()
    B = [6, 2]
    x = torch.randn(8, 256, device=gpu).to(torch.bfloat16)
    idx = torch.tensor([[0, 1]] * 8, dtype=torch.int32, device=gpu)
    idx[3, 1] = 9          # E = 8: out of range
    guard = torch.full((8 * 2 + 64, 256), 7, dtype=torch.bfloat16, device=gpu)
    recv = guard[:16]
    d0 = b.dispatch(x, torch.zeros_like(idx), B, 8)   # allocates maps/workspace
    d0.recv_x = recv
    d = b.dispatch(x, idx, B, 8, out=d0)
    st, code = b.get_device_error(d.workspace)
    assert st == 6 and (code & 1)
    assert torch.all(guard[16:] == 7)                 # nothing past the receive buffer
    idx2 = torch.tensor([[2, 2]] * 8, dtype=torch.int32, device=gpu)   # duplicate expert
    d = b.dispatch(x, idx2, B, 8, out=d0)
    st, code = b.get_device_error(d.workspace)
    assert st == 6 and (code & 2)
    d = b.dispatch(x, torch.tensor([[0, 1]] * 8, dtype=torch.int32, device=gpu), B, 8, out=d0)
    st, code = b.get_device_error(d.workspace)
    assert st == 0 and code == 0                      # the next good call clears the word
