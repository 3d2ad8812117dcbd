"""Seeded synthetic inputs for MoE route/dispatch/combine, shared by the tests,
the smoke check and the benchmark.

This module only draws random inputs; it holds none of the routing, dispatch
or combine arithmetic.  The shapes follow the layers the sources discuss:
DeepSeek-V3 (256 routed experts, top-8, hidden 7168; Perplexity, "Lower
latency and higher throughput with multi-node DeepSeek deployment", section
"Expert parallelism") and Kimi-K2 / DeepSeek-V3 dispatch at hidden size 7168
with FP8 block-scaled dispatch and bf16 combine (Perplexity, "Enabling
trillion-parameter models on AWS EFA", section "Evaluation"), plus the small
8-rank, 16-expert, top-2 problem of lehuy.net, "Decoding high-performance EP
kernels", section "Our task".

Recipe (all draws from ``numpy.random.SeedSequence(seed).spawn(4)``, one
child each for B, x, logits and the expert permutation):

* ``B[s]`` ~ discrete uniform on ``[b_lo, b_hi]`` inclusive, one per rank
  (empty ranks are legal);
* ``x`` = N(0, 1) drawn in fp32, rounded to bf16 (round to nearest even);
* ``logits`` = N(0, 1) in fp32, plus, for the skewed-load workload, a
  per-expert bias ``-s * ln(1 + pi(e))`` (the log of a Zipf(s) weight over a
  random permutation ``pi`` of the experts), computed in fp64 and added in fp32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    R: int            # logical EP ranks
    E: int            # routed experts (E/R per rank)
    K: int            # experts per token
    H: int            # hidden size
    b_lo: int         # tokens per rank ~ U{b_lo..b_hi}
    b_hi: int
    fp8: bool = False         # dispatch payload quantised to e4m3 + fp32 scales per 128 channels
    zipf_s: float | None = None
    note: str = field(default="", compare=False)

    @property
    def L(self) -> int:
        return self.E // self.R


WORKLOADS: dict[str, Workload] = {
    "toy": Workload("toy", R=8, E=16, K=2, H=256, b_lo=1, b_hi=64,
                    note="8 ranks, 16 experts (2 per rank), top-2, variable tokens per rank"),
    "dsv3_decode": Workload("dsv3_decode", R=8, E=256, K=8, H=7168, b_lo=128, b_hi=128,
                            note="DeepSeek-V3 decode layer, 128 tokens per rank, bf16"),
    "dsv3_prefill": Workload("dsv3_prefill", R=8, E=256, K=8, H=7168, b_lo=4096, b_hi=4096, fp8=True,
                             note="DeepSeek-V3 prefill layer, 4096 tokens per rank, FP8 dispatch, bf16 combine"),
    "kimi_decode": Workload("kimi_decode", R=32, E=384, K=8, H=7168, b_lo=0, b_hi=64, zipf_s=1.2,
                            note="Kimi-K2-style decode layer, Zipf(1.2) expert bias, bf16"),
    "wide_ep_decode": Workload("wide_ep_decode", R=128, E=256, K=8, H=7168, b_lo=0, b_hi=32,
                               note="Wide-EP decode layer, 128 ranks, 2 experts per rank, bf16"),
}


def _rngs(seed: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(4)]


def draw_B(w: Workload, seed: int = 0) -> np.ndarray:
    rb = _rngs(seed)[0]
    return rb.integers(w.b_lo, w.b_hi + 1, size=w.R, dtype=np.int64).astype(np.int32)


def draw_x(T: int, H: int, rng: np.random.Generator) -> torch.Tensor:
    """bf16 [T, H] on the CPU: N(0,1) in fp32 rounded to nearest-even bf16."""
    out = torch.empty((T, H), dtype=torch.bfloat16)
    rows = max(1, (1 << 24) // max(H, 1))          # bounded fp32 scratch per chunk
    for r0 in range(0, T, rows):
        r1 = min(T, r0 + rows)
        z = rng.standard_normal((r1 - r0, H), dtype=np.float32)
        out[r0:r1] = torch.from_numpy(z).to(torch.bfloat16)
    return out


def draw_logits(T: int, E: int, rng: np.random.Generator, zipf_s: float | None = None,
                perm_rng: np.random.Generator | None = None) -> np.ndarray:
    z = rng.standard_normal((T, E), dtype=np.float32)
    if zipf_s is not None:
        pi = perm_rng.permutation(E)
        bias = (-zipf_s * np.log1p(pi.astype(np.float64))).astype(np.float32)
        z += bias[None, :]
    return z


def generate(w: Workload | str, seed: int = 0, B=None) -> dict:
    """Inputs for one layer: B (int32 [R]), x (bf16 CPU tensor [T,H]), logits (fp32 [T,E])."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    rb, rx, rl, rp = _rngs(seed)
    if B is None:
        B = rb.integers(w.b_lo, w.b_hi + 1, size=w.R, dtype=np.int64).astype(np.int32)
    B = np.asarray(B, dtype=np.int32)
    assert B.size == w.R
    T = int(B.sum())
    x = draw_x(T, w.H, rx)
    logits = draw_logits(T, w.E, rl, w.zipf_s, rp)
    return dict(workload=w, B=B, T=T, x=x, logits=logits)


def random_shape_inputs(R: int, E: int, K: int, H: int, B, seed: int = 0, fp8: bool = False,
                        zipf_s: float | None = None) -> dict:
    """Inputs for an arbitrary small shape (parity sweeps over R, E, K, H and B)."""
    w = Workload(f"R{R}_E{E}_K{K}_H{H}", R=R, E=E, K=K, H=H, b_lo=0, b_hi=0, fp8=fp8, zipf_s=zipf_s)
    return generate(w, seed=seed, B=B)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a CPU bf16 tensor (a view, no arithmetic)."""
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)
