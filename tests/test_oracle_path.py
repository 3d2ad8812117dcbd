"""Pins for the oracle's route, dispatch, expert stand-in and combine: library
routines, brute force on tiny inputs, invariants fixed by the sources, and the
counting examples the sources print.  CPU only."""
import itertools
import os

import numpy as np
import pytest
import scipy.special
import torch

from combine_moe_route_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# route
# --------------------------------------------------------------------------

def _tie_logits(T, E, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(-3, 4, size=(T, E)).astype(np.float32)   # many exact ties


def test_route_k1_is_argmax(oracle):
    for lg in (_tie_logits(200, 37, 0), np.random.default_rng(1).standard_normal((200, 64)).astype(np.float32)):
        idx, w = oracle.route_topk(lg, 1)
        assert np.array_equal(idx[:, 0], np.argmax(lg, axis=1))     # first max = lowest id
        assert np.all(w == 1.0)


def test_route_k_equals_e_is_stable_descending_sort(oracle):
    for lg in (_tie_logits(100, 12, 2), np.random.default_rng(3).standard_normal((100, 16)).astype(np.float32)):
        T, E = lg.shape
        idx, _ = oracle.route_topk(lg, E)
        for g in range(T):
            ref = np.lexsort((np.arange(E), -lg[g]))    # key: logit desc, then id asc
            assert np.array_equal(idx[g], ref)


def test_route_brute_force_tiny(oracle):
    rng = np.random.default_rng(4)
    for E in (2, 3, 4, 5, 6):
        for K in range(1, min(E, 3) + 1):
            lg = rng.integers(-2, 3, size=(30, E)).astype(np.float32)
            idx, _ = oracle.route_topk(lg, K)
            for g in range(30):
                best = max(itertools.permutations(range(E), K),
                           key=lambda tup: tuple(v for e in tup for v in (lg[g, e], -e)))
                assert tuple(idx[g]) == best


def test_route_weights_softmax(oracle):
    rng = np.random.default_rng(5)
    lg = (rng.standard_normal((500, 256)) * 2).astype(np.float32)
    for K in (2, 8):
        idx, w = oracle.route_topk(lg, K)
        sel = np.take_along_axis(lg, idx, axis=1).astype(np.float64)
        ref = scipy.special.softmax(sel, axis=1)
        assert np.all(np.abs(w - ref) <= 2.0**-24 * np.maximum(ref, 2.0**-126) * 2)
        assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= K * 2.0**-24)
        assert np.all(np.diff(w, axis=1) <= 0)          # descending like the logits
    # K = 2 closed form: w0 = 1 / (1 + exp(l1 - l0))
    idx, w = oracle.route_topk(lg, 2)
    sel = np.take_along_axis(lg, idx, axis=1).astype(np.float64)
    w0 = 1.0 / (1.0 + np.exp(sel[:, 1] - sel[:, 0]))
    assert np.all(np.abs(w[:, 0] - w0) <= 2.0**-24 * w0 * 2)


# --------------------------------------------------------------------------
# dispatch
# --------------------------------------------------------------------------

def _random_routing(T, E, K, rng):
    return np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32).reshape(T, K)


def _layout_by_library_sort(idx, B, E):
    """Reference layout from numpy's stable argsort (a library routine)."""
    T, K = idx.shape
    R = len(B)
    keys = idx.reshape(-1)
    row2src = np.argsort(keys, kind="stable").astype(np.int32)
    tok2row = np.empty_like(row2src)
    tok2row[row2src] = np.arange(T * K, dtype=np.int32)
    src_rank = np.repeat(np.arange(R), np.asarray(B) * K)
    counts = np.bincount(keys * R + src_rank, minlength=E * R).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return counts, offsets, tok2row, row2src


@pytest.mark.parametrize("R,E,K,H,B", [
    (8, 16, 2, 256, None),
    (1, 4, 4, 16, [5]),
    (3, 9, 3, 64, [0, 7, 2]),
    (4, 32, 8, 128, [1, 0, 33, 9]),
])
def test_dispatch_matches_library_stable_sort(oracle, R, E, K, H, B):
    rng = np.random.default_rng(7)
    if B is None:
        B = rng.integers(1, 65, size=R)
    B = np.asarray(B, np.int32)
    T = int(B.sum())
    idx = _random_routing(T, E, K, rng)
    x = oracle.bf16_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    d = oracle.dispatch(x, idx, B, E)
    counts, offsets, tok2row, row2src = _layout_by_library_sort(idx, B, E)
    assert np.array_equal(d["counts"], counts)
    assert np.array_equal(d["offsets"], offsets)
    assert np.array_equal(d["expert_offsets"], offsets[::R][: E + 1] if R > 0 else offsets)
    assert np.array_equal(d["tok2row"], tok2row)
    assert np.array_equal(d["row2src"], row2src)
    assert np.array_equal(d["recv"], x[row2src // K])


def _check_dispatch_invariants(d, idx, B, E, x):
    T, K = idx.shape
    R = len(B)
    counts, offsets, eo = d["counts"], d["offsets"], d["expert_offsets"]
    assert counts.sum() == T * K                                   # every token lands K times
    assert np.array_equal(counts.reshape(E, R).sum(0), np.asarray(B) * K)
    assert np.all(counts.reshape(E, R) <= np.asarray(B)[None, :])
    assert offsets[-1] == T * K and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(d["row2src"]), np.arange(T * K))   # a permutation
    assert np.array_equal(d["row2src"][d["tok2row"]], np.arange(T * K))
    e_of_row = idx.reshape(-1)[d["row2src"]]
    assert np.all(e_of_row[:-1] <= e_of_row[1:]) if T * K else True  # expert-contiguous
    for e in range(E):
        seg = d["row2src"][eo[e]:eo[e + 1]]
        assert np.all(idx.reshape(-1)[seg] == e)
        assert np.all(np.diff(seg // K) > 0)                        # ascending source token
    if x is not None and T:
        assert np.array_equal(d["recv"], x[d["row2src"] // K])


def test_dispatch_brute_force_all_routings(oracle):
    """Every routing of T tokens over ordered distinct K-tuples, tiny shapes."""
    cases = [(1, 3, 1, [3]), (2, 4, 2, [1, 2]), (3, 6, 2, [1, 0, 1]), (2, 6, 3, [1, 1]), (3, 3, 2, [0, 2, 1])]
    for R, E, K, B in cases:
        B = np.asarray(B, np.int32)
        T = int(B.sum())
        tuples = list(itertools.permutations(range(E), K))
        x = np.arange(T * 8, dtype=np.uint16).reshape(T, 8) + 0x3F00
        src_rank = np.repeat(np.arange(R), B)
        for routing in itertools.product(tuples, repeat=T):
            idx = np.array(routing, np.int32).reshape(T, K)
            d = oracle.dispatch(x, idx, B, E)
            # direct definition: row(g, j) = start of expert e + #earlier tokens routed to e
            flat = idx.reshape(-1)
            ecount = np.array([(flat == e).sum() for e in range(E)])
            estart = np.concatenate([[0], np.cumsum(ecount)])
            for g in range(T):
                for j in range(K):
                    e = idx[g, j]
                    before = sum(1 for g2 in range(g) if e in idx[g2])
                    assert d["tok2row"][g * K + j] == estart[e] + before
            cnt = np.zeros((E, R), np.int32)
            for g in range(T):
                for e in idx[g]:
                    cnt[e, src_rank[g]] += 1
            assert np.array_equal(d["counts"], cnt.reshape(-1))
            _check_dispatch_invariants(d, idx, B, E, x)


def test_dispatch_fp8_rows_are_quantised_source_rows(oracle):
    rng = np.random.default_rng(8)
    R, E, K, H = 4, 8, 3, 512
    B = np.array([3, 0, 5, 2], np.int32)
    T = int(B.sum())
    idx = _random_routing(T, E, K, rng)
    x = oracle.bf16_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    d = oracle.dispatch(x, idx, B, E, fp8=True)
    q, s = oracle.quantize_rows_e4m3(x)
    src = d["row2src"] // K
    assert np.array_equal(d["recv"], q[src])
    assert np.array_equal(d["recv_scale"].view(np.uint32), s[src].view(np.uint32))
    d16 = oracle.dispatch(x, idx, B, E, fp8=False)
    for key in ("counts", "offsets", "expert_offsets", "tok2row", "row2src"):
        assert np.array_equal(d[key], d16[key])


def test_dispatch_rejects_out_of_range_expert(oracle):
    x = np.zeros((2, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.dispatch(x, np.array([[0], [4]], np.int32), [1, 1], 4)


def test_dispatch_empty(oracle):
    d = oracle.dispatch(np.zeros((0, 8), np.uint16), np.zeros((0, 2), np.int32), [0, 0], 4)
    assert d["counts"].sum() == 0 and np.all(d["offsets"] == 0) and np.all(d["expert_offsets"] == 0)


def _golden_lines():
    with open(os.path.join(GOLDEN, "page_counting_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            name, *kv = lhs.split()
            yield name, {k: int(v) for k, v in (p.split("=") for p in kv)}, int(rhs)


def test_page_counting_examples(oracle):
    seen = set()
    for name, p, expect in _golden_lines():
        seen.add(name)
        T, K, E, R = p["T"], p["K"], p["E"], p["R"]
        B = np.full(R, T // R, np.int32)
        B[: T - int(B.sum())] += 1
        rng = np.random.default_rng(9)
        L = E // R
        if name in ("max_active_experts", "mean_active_experts_per_rank"):
            # two tokens routed to disjoint expert sets reach the printed maximum
            perm = rng.permutation(E)
            idx = perm[: T * K].reshape(T, K).astype(np.int32)
        elif name.startswith("worst_case_rows_per_rank"):
            # every token sends as many copies as it can to rank 0: all of its
            # experts there when K <= E/R, else all E/R of rank 0's and the rest
            # on the next rank
            loc = min(K, L)
            one = np.array(list(range(loc)) + list(range(L, L + K - loc)), np.int32)
            idx = np.tile(one, (T, 1))
        else:
            logits = wl.draw_logits(T, E, rng)
            idx, _ = oracle.route_topk(logits, K)
        d = oracle.dispatch(np.zeros((T, 8), np.uint16), idx, B, E)
        per_expert = d["counts"].reshape(E, R).sum(1)
        active = per_expert > 0
        if name.startswith("worst_case_rows_per_rank"):
            eo = d["expert_offsets"]
            got = int(eo[L] - eo[0])                      # rank 0's receive window
            assert got <= T * max(K, L)                   # the page's printed bound holds
            # and no routing gives any rank more: random routings of the same shape
            for seed in range(20):
                r_idx = np.stack([np.random.default_rng(seed * 1000 + g).permutation(E)[:K]
                                  for g in range(T)]).astype(np.int32)
                r_eo = oracle.dispatch(np.zeros((T, 8), np.uint16), r_idx, B, E)["expert_offsets"]
                assert np.all(r_eo[L::L] - r_eo[:-1:L] <= expect)
        elif name == "max_active_experts":
            got = int(active.sum())
            assert got <= T * K
        elif name in ("mean_active_experts_per_rank",):
            got = active.reshape(R, L).sum(1).mean()
        elif name == "active_experts_per_rank_large_batch":
            per_rank = active.reshape(R, L).sum(1)
            assert np.all(per_rank == per_rank[0])
            got = int(per_rank[0])
        elif name == "mean_tokens_per_expert":
            got = per_expert.mean()
        else:
            raise AssertionError(name)
        assert got == expect, (name, got, expect)
    assert seen == {"max_active_experts", "mean_active_experts_per_rank",
                    "active_experts_per_rank_large_batch", "mean_tokens_per_expert",
                    "worst_case_rows_per_rank", "worst_case_rows_per_rank_few_local_experts"}


# --------------------------------------------------------------------------
# expert stand-in
# --------------------------------------------------------------------------

def test_expert_scale_matches_library_ops(oracle):
    rng = np.random.default_rng(10)
    E, H = 6, 256
    eo = np.array([0, 3, 3, 7, 8, 12, 15], np.int32)
    xb = oracle.bf16_from_f32(rng.standard_normal((15, H)).astype(np.float32))
    e_of_row = np.repeat(np.arange(E), np.diff(eo))
    s = torch.tensor(1.0 + e_of_row / 256.0, dtype=torch.float32)[:, None]
    xt = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).float()
    ref = (xt * s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.expert_scale(xb, None, eo, E), ref)
    assert np.array_equal(oracle.expert_scale(xb, None, eo, E, identity=True), xb)
    # FP8 receive buffer: decode * scale, then * s_e
    q, sc = oracle.quantize_rows_e4m3(xb)
    qt = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).float()
    sct = torch.from_numpy(sc.copy()).repeat_interleave(128, dim=1)
    ref8 = ((qt * sct) * s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.expert_scale(q, sc, eo, E), ref8)


# --------------------------------------------------------------------------
# combine
# --------------------------------------------------------------------------

def _layer_inputs(oracle, R, E, K, H, B, seed):
    rng = np.random.default_rng(seed)
    T = int(np.sum(B))
    x = oracle.bf16_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    return x, logits


def test_combine_identity_experts_returns_input(oracle):
    x, logits = _layer_inputs(oracle, 4, 16, 4, 256, [9, 0, 17, 4], 11)
    d = oracle.layer(x, logits, [9, 0, 17, 4], 16, 4, identity=True)
    xf = oracle.f32_from_bf16(x)
    of = oracle.f32_from_bf16(d["out"])
    ulp = np.abs(xf) * 2.0**-7
    assert np.all(np.abs(of - xf) <= ulp)
    o32 = oracle.combine(d["y"], d["tok2row"], d["topk_w"], out="f32")
    assert np.all(np.abs(o32 - xf) <= np.abs(xf) * 4 * 2.0**-24)


def test_combine_identity_experts_fp8(oracle):
    B = [5, 3]
    x, logits = _layer_inputs(oracle, 2, 8, 2, 1024, B, 12)
    d = oracle.layer(x, logits, B, 8, 2, fp8=True, identity=True)
    q, s = oracle.quantize_rows_e4m3(x)
    dq = oracle.e4m3_decode(q).astype(np.float64) * np.repeat(s, 128, axis=1)
    o = oracle.f32_from_bf16(d["out"]).astype(np.float64)
    # out = bf16(dequant * sum(w)); sum(w) = 1 within a few ulp
    assert np.all(np.abs(o - dq) <= np.abs(dq) * (2.0**-8 + 1e-6) + 1e-30)


def test_combine_one_hot_weights_pick_the_row(oracle):
    rng = np.random.default_rng(13)
    T, K, H = 20, 4, 64
    y = oracle.bf16_from_f32(rng.standard_normal((T * K, H)).astype(np.float32))
    t2r = rng.permutation(T * K).astype(np.int32)
    for jj in range(K):
        w = np.zeros((T, K), np.float32)
        w[:, jj] = 1.0
        o = oracle.combine(y, t2r, w)
        assert np.array_equal(o, y[t2r.reshape(T, K)[:, jj]])


def test_combine_fp32_within_error_bound_of_exact(oracle):
    rng = np.random.default_rng(14)
    T, K, H = 64, 8, 512
    y = oracle.bf16_from_f32(rng.standard_normal((T * K, H)).astype(np.float32))
    t2r = rng.permutation(T * K).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    w[:, 3] = -w[:, 3]                                   # mixed signs: cancellation
    yf = oracle.f32_from_bf16(y).astype(np.float64)
    g = yf[t2r.reshape(T, K)]                            # [T, K, H]
    exact = np.einsum("tk,tkh->th", w.astype(np.float64), g)   # library contraction
    o64 = oracle.combine(y, t2r, w, out="f64")
    assert np.all(np.abs(o64 - exact) <= 1e-12 * np.einsum("tk,tkh->th", np.abs(w), np.abs(g)))
    o32 = oracle.combine(y, t2r, w, out="f32").astype(np.float64)
    u = 2.0**-24
    gamma = K * u / (1 - K * u)
    bound = gamma * np.einsum("tk,tkh->th", np.abs(w).astype(np.float64), np.abs(g))
    assert np.all(np.abs(o32 - exact) <= bound)
    ob = oracle.combine(y, t2r, w, out="bf16")
    assert np.array_equal(ob, oracle.bf16_from_f32(o32.astype(np.float32)))


def test_combine_fma_order_is_j_ascending(oracle):
    # a case where the order of the fused accumulation changes the fp32 result
    y = oracle.bf16_from_f32(np.array([[1.0], [2.0**-20], [-1.0]], np.float32).repeat(8, axis=1))
    t2r = np.array([0, 1, 2], np.int32)
    w = np.array([[1.0, 1.0, 1.0]], np.float32)
    o = oracle.combine(y, t2r, w, out="f32")
    acc = np.float32(0)
    for v in (1.0, 2.0**-20, -1.0):
        acc = np.float32(acc + np.float32(v))            # exact products; adds in j order
    assert np.all(o == acc)


def test_combine_linear_in_y(oracle):
    rng = np.random.default_rng(15)
    T, K, H = 16, 4, 64
    y = oracle.bf16_from_f32(rng.standard_normal((T * K, H)).astype(np.float32))
    y2 = oracle.bf16_from_f32(oracle.f32_from_bf16(y) * 2)      # exact doubling
    t2r = rng.permutation(T * K).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    a = oracle.combine(y, t2r, w, out="f32")
    b = oracle.combine(y2, t2r, w, out="f32")
    assert np.array_equal(b, a * 2)


def test_full_layer_invariants_workload_toy(oracle):
    inp = wl.generate("toy", seed=0)
    x = wl.bf16_bits(inp["x"])
    d = oracle.layer(x, inp["logits"], inp["B"], 16, 2)
    _check_dispatch_invariants(d, d["topk_idx"], inp["B"], 16, x)


# --------------------------------------------------------------------------
# group-limited route
# --------------------------------------------------------------------------

def test_grouped_route_one_group_or_all_groups_is_plain_route(oracle):
    # the MoE-router section: plain (Mixtral) routing is the case where the group
    # top-K covers every expert
    rng = np.random.default_rng(20)
    for lg in (_tie_logits(300, 64, 21), rng.standard_normal((300, 256)).astype(np.float32)):
        E = lg.shape[1]
        for K in (1, 2, 8):
            idx, w = oracle.route_topk(lg, K)
            for G, M in ((1, 1), (8, 8), (4, 4)):
                gi, gw = oracle.route_topk_grouped(lg, K, G, M)
                assert np.array_equal(gi, idx) and np.array_equal(gw, w)


def test_grouped_route_matches_library_sort(oracle):
    rng = np.random.default_rng(22)
    for lg in (_tie_logits(200, 32, 23), rng.standard_normal((200, 64)).astype(np.float32)):
        T, E = lg.shape
        for G, M, K in ((8, 4, 8), (4, 1, 2), (8, 3, 5), (2, 1, 1)):
            gs = E // G
            gi, gw = oracle.route_topk_grouped(lg, K, G, M)
            for g in range(T):
                gmax = lg[g].reshape(G, gs).max(axis=1)
                keep = np.lexsort((np.arange(G), -gmax))[:M]          # score desc, id asc
                allowed = np.isin(np.arange(E) // gs, keep)
                cand = np.nonzero(allowed)[0]
                order = cand[np.lexsort((cand, -lg[g, cand]))][:K]
                assert np.array_equal(gi[g], order)
                assert len(set(gi[g] // gs)) <= M
            sel = np.take_along_axis(lg, gi, axis=1).astype(np.float64)
            ref = scipy.special.softmax(sel, axis=1)
            assert np.all(np.abs(gw - ref) <= 2.0**-24 * np.maximum(ref, 2.0**-126) * 2)


# --------------------------------------------------------------------------
# low-latency (fixed-rectangle) layout
# --------------------------------------------------------------------------

@pytest.mark.parametrize("R,E,K,H,B,C,fp8", [
    (8, 16, 2, 256, [5, 0, 17, 3, 64, 1, 9, 2], 64, False),
    (4, 32, 8, 256, [7, 0, 3, 12], 12, True),
    (2, 8, 8, 128, [16, 16], 16, False),          # K == E: every expert gets every token
    (3, 9, 3, 64, [0, 0, 0], 4, False),           # empty
])
def test_ll_layout_is_the_ragged_layout_in_fixed_regions(oracle, R, E, K, H, B, C, fp8):
    rng = np.random.default_rng(30 + K)
    B = np.asarray(B, np.int32)
    T = int(B.sum())
    idx = _random_routing(T, E, K, rng) if T else np.zeros((0, K), np.int32)
    x = oracle.bf16_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    ll = oracle.dispatch_ll(x, idx, B, E, C, fp8=fp8)
    rg = oracle.dispatch(x, idx, B, E, fp8=fp8)
    assert np.array_equal(ll["counts"], rg["counts"])
    # copy j of token g: same (expert, rank) region, same slot as its place in the ragged segment
    ragged = rg["tok2row"]
    region = ll["tok2row"] // C
    slot = ll["tok2row"] % C
    flat = idx.reshape(-1)
    src_rank = np.repeat(np.arange(R), B * K)
    assert np.array_equal(region, flat * R + src_rank)
    assert np.array_equal(slot, ragged - rg["offsets"][flat * R + src_rank])
    assert np.all(slot < np.maximum(B[src_rank], 1))
    # payload and source tags of every filled row
    filled = ll["row2src"] >= 0
    assert filled.sum() == T * K
    assert np.array_equal(ll["recv"][ll["tok2row"]], rg["recv"][ragged])
    if fp8:
        assert np.array_equal(ll["recv_scale"][ll["tok2row"]], rg["recv_scale"][ragged])
    assert np.array_equal(ll["row2src"][ll["tok2row"]], np.arange(T * K))


def test_ll_rejects_more_tokens_than_the_chunk_cap(oracle):
    with pytest.raises(ValueError):
        oracle.dispatch_ll(np.zeros((5, 8), np.uint16), np.zeros((5, 1), np.int32), [5], 2, 4)


def test_ll_push_then_reduce_equals_gather(oracle):
    rng = np.random.default_rng(31)
    R, E, K, H, C = 4, 16, 4, 128, 20
    B = np.array([20, 3, 0, 11], np.int32)
    T = int(B.sum())
    idx = _random_routing(T, E, K, rng)
    x = oracle.bf16_from_f32(rng.standard_normal((T, H)).astype(np.float32))
    ll = oracle.dispatch_ll(x, idx, B, E, C)
    eo = np.arange(E + 1, dtype=np.int32) * (R * C)            # expert e owns rows [e*R*C, (e+1)*R*C)
    y = oracle.expert_scale(ll["recv"], None, eo, E)
    w = rng.random((T, K)).astype(np.float32)
    gather = oracle.combine(y, ll["tok2row"], w, out="f32")
    ret = oracle.combine_ll_push(y, ll["row2src"], ll["counts"], R, E, C, T, K)
    pushed = oracle.combine(ret, np.arange(T * K, dtype=np.int32), w, out="f32")
    assert np.array_equal(gather.view(np.uint32), pushed.view(np.uint32))
    # and both equal the throughput layout's combine
    rg = oracle.dispatch(x, idx, B, E)
    yr = oracle.expert_scale(rg["recv"], None, rg["expert_offsets"], E)
    assert np.array_equal(oracle.combine(yr, rg["tok2row"], w, out="f32").view(np.uint32), gather.view(np.uint32))


# --------------------------------------------------------------------------
# sender-side partial accumulation
# --------------------------------------------------------------------------

def _partial_case(oracle, R, E, K, H, T, seed):
    rng = np.random.default_rng(seed)
    idx = _random_routing(T, E, K, rng)
    y = oracle.bf16_from_f32(rng.standard_normal((T * K, H)).astype(np.float32))
    t2r = rng.permutation(T * K).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    return idx, y, t2r, w


def test_partial_with_one_rank_is_receive_side(oracle):
    # all experts on one rank: the single partial is the receive-side fp32 sum, rounded once
    idx, y, t2r, w = _partial_case(oracle, 1, 16, 4, 64, 40, 40)
    assert np.array_equal(oracle.combine_partial(y, t2r, idx, w, 16, 1), oracle.combine(y, t2r, w))
    f = oracle.combine_partial(y, t2r, idx, w, 16, 1, out="f32")
    assert np.array_equal(f, oracle.f32_from_bf16(oracle.combine(y, t2r, w)))


def test_partial_slots_and_error_bound(oracle):
    R, E, K, H, T = 8, 64, 8, 128, 60
    idx, y, t2r, w = _partial_case(oracle, R, E, K, H, T, 41)
    out, part = oracle.combine_partial(y, t2r, idx, w, E, R, out="f32", with_partial=True)
    L = E // R
    yf = oracle.f32_from_bf16(y).astype(np.float64)
    exact = np.zeros((T, H))
    bound = np.zeros((T, H))
    for g in range(T):
        ranks = idx[g] // L
        for r in np.unique(ranks):                            # numpy's own grouping of the K copies
            js = np.nonzero(ranks == r)[0]
            s = sum(float(w[g, j]) * yf[t2r[g * K + j]] for j in js)
            exact[g] += s
            # the partial travels in slot g*K + (first j of the rank)
            pr = oracle.f32_from_bf16(part[g * K + js[0]]).astype(np.float64)
            mag = sum(abs(float(w[g, j])) * np.abs(yf[t2r[g * K + j]]) for j in js)
            assert np.all(np.abs(pr - s) <= np.abs(s) * 2.0**-8 + mag * len(js) * 2.0**-23 + 1e-30)
            bound += np.abs(s) * 2.0**-8 + mag * len(js) * 2.0**-23
        # slots of non-first copies are not written
        firsts = {int(np.nonzero(ranks == r)[0][0]) for r in np.unique(ranks)}
        for j in range(K):
            if j not in firsts:
                assert np.all(part[g * K + j] == 0)
    n_ranks_max = K
    bound += np.abs(exact) * n_ranks_max * 2.0**-23
    assert np.all(np.abs(out - exact) <= bound + 1e-30)
