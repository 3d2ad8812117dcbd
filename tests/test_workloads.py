"""The seeded input generators follow their stated recipe (CPU only): the same seed gives the
same inputs, draws stay in their ranges, x is the bf16 rounding of a fp32 normal draw, and the
skewed-load workload's logits carry the Zipf bias over a permutation of the experts."""
import numpy as np
import pytest
import torch

from combine_moe_route_gb300 import workloads as wl


@pytest.mark.parametrize("name", ["toy", "kimi_decode", "wide_ep_decode"])
def test_same_seed_same_inputs_and_ranges(name):
    w = wl.WORKLOADS[name]
    a, b = wl.generate(w, seed=0), wl.generate(w, seed=0)
    assert np.array_equal(a["B"], b["B"]) and torch.equal(a["x"], b["x"])
    assert np.array_equal(a["logits"], b["logits"])
    c = wl.generate(w, seed=1)
    assert not np.array_equal(a["logits"][: min(a["T"], c["T"])].ravel()[:64],
                              c["logits"][: min(a["T"], c["T"])].ravel()[:64])
    B = a["B"]
    assert B.dtype == np.int32 and B.shape == (w.R,)
    assert np.all((B >= w.b_lo) & (B <= w.b_hi))
    assert a["T"] == int(B.sum())
    assert a["x"].dtype == torch.bfloat16 and tuple(a["x"].shape) == (a["T"], w.H)
    assert a["logits"].dtype == np.float32 and a["logits"].shape == (a["T"], w.E)
    assert np.array_equal(wl.draw_B(w, 0), B)


def test_x_is_the_bf16_rounding_of_a_normal_fp32_draw():
    # the same child stream, drawn directly in fp32, rounds to the generator's bf16 values
    w = wl.WORKLOADS["toy"]
    inp = wl.generate(w, seed=3)
    rx = [np.random.default_rng(s) for s in np.random.SeedSequence(3).spawn(4)][1]
    z = rx.standard_normal((inp["T"], w.H), dtype=np.float32)
    assert torch.equal(inp["x"], torch.from_numpy(z).to(torch.bfloat16))
    v = inp["x"].float().numpy().ravel()
    assert abs(v.mean()) < 0.05 and abs(v.std() - 1.0) < 0.05


def test_zipf_bias_over_a_permutation_of_the_experts():
    # Kimi-like layer: logits = N(0,1) + (-1.2 * ln(1 + pi(e))); with many tokens, the
    # per-expert column means recover the bias, and sorted they are the Zipf log weights
    w = wl.Workload("zipf_check", R=4, E=64, K=8, H=8, b_lo=2000, b_hi=2000, zipf_s=1.2)
    inp = wl.generate(w, seed=5)
    col = inp["logits"].astype(np.float64).mean(axis=0)
    want = -1.2 * np.log1p(np.arange(w.E))                     # pi(e) = 0..E-1 in some order
    assert np.all(np.abs(np.sort(col)[::-1] - want) < 5.0 / np.sqrt(inp["T"]) + 1e-3)
    rp = [np.random.default_rng(s) for s in np.random.SeedSequence(5).spawn(4)][3]
    pi = rp.permutation(w.E)
    assert np.all(np.abs(col - (-1.2 * np.log1p(pi))) < 5.0 / np.sqrt(inp["T"]))


def test_explicit_B_overrides_the_draw():
    inp = wl.random_shape_inputs(3, 9, 3, 16, [4, 0, 7], seed=2)
    assert np.array_equal(inp["B"], np.array([4, 0, 7], np.int32)) and inp["T"] == 11
    assert tuple(inp["x"].shape) == (11, 16) and inp["logits"].shape == (11, 9)
