"""The bound behind the route kernel's candidate filter (CPU only).

The kernel keeps one warp per token; lane l holds the keys of experts l, l+32, ...
(or, with 16-byte loads when E is 32 * NPL and a multiple of 128, experts
128q + 4l .. 128q + 4l + 3); the bound holds for any split of the experts among the
lanes, and both splits are checked.
Its threshold tau is the upper 27 bits of the K-th largest of the 32 lane maxima, each
with its low 5 bits replaced by the tag 31 - l (a lane without keys contributes 0), and
every eligible key >= tau becomes a candidate.  The selection is exact only if the
candidates hold the whole top K (key descending, equal keys by smaller expert), which is
what these rows check: random, tie-heavy and denormal rows, and shapes where fewer than
K lanes hold keys.  The keys are the order-preserving image of fp32 (after adding +0).
The last test models how the 16-byte layout forms group maxima for group-limited routing."""
import numpy as np
import pytest


def _keys(f):
    u = (f.astype(np.float32) + np.float32(0.0)).view(np.uint32).astype(np.uint64)
    return np.where((u >> 31) == 1, (~u) & 0xFFFFFFFF, u | 0x80000000)


def _lane_of(e, E, vec):
    return (e % 128) // 4 if vec else e % 32


def _tagged_tau(k, K, vec=False):
    E = k.size
    lanes = np.zeros((32, -(-E // 32)), np.uint64)
    fill = np.zeros(32, np.int64)
    for e in range(E):
        l = _lane_of(e, E, vec)
        lanes[l, fill[l]] = k[e]
        fill[l] += 1
    lmax = lanes.max(axis=1)
    v = np.where(lmax > 0, (lmax & ~np.uint64(31)) | (31 - np.arange(32)).astype(np.uint64), 0)
    top = 0
    for _ in range(K):
        top = int(v.max())
        v[v == top] = 0          # the tags make the one lane holding top unique (top = 0: no change)
    return top & ~31


@pytest.mark.parametrize("E,K,vec", [(256, 8, False), (32, 32, False), (40, 33, False), (9, 3, False),
                                     (1024, 32, False), (384, 8, False), (64, 1, False),
                                     (256, 8, True), (128, 4, True), (384, 8, True), (1024, 32, True)])
@pytest.mark.parametrize("kind", ["normal", "ties", "denormal"])
def test_candidates_hold_the_top_k(E, K, vec, kind):
    rng = np.random.default_rng(E * 100 + K)
    for _ in range(150):
        if kind == "normal":
            f = rng.standard_normal(E)
        elif kind == "ties":
            f = np.round(rng.standard_normal(E) * 2.0)
        else:
            f = rng.integers(-3, 4, E) * np.float32(1e-45)
        k = _keys(np.asarray(f, np.float32))
        order = np.lexsort((np.arange(E), -k.astype(np.int64)))
        tau = _tagged_tau(k, K, vec)
        cand = np.flatnonzero((k != 0) & (k >= tau))
        assert set(order[:K].tolist()) <= set(cand.tolist())


def test_fewer_lanes_than_k_admits_every_key():
    # E = 40, K = 33: 32 lanes hold keys, so the 33rd round finds nothing and tau = 0
    k = _keys(np.random.default_rng(3).standard_normal(40).astype(np.float32))
    assert _tagged_tau(k, 33) == 0


def test_random_rows_admit_few_candidates():
    # DeepSeek-V3 router shape: about K plus one candidates per row on N(0, 1) logits
    rng = np.random.default_rng(11)
    for vec in (False, True):
        n = [int(((k := _keys(rng.standard_normal(256).astype(np.float32))) >= _tagged_tau(k, 8, vec)).sum())
             for _ in range(400)]
        assert 8 <= min(n) and np.mean(n) < 10 and max(n) <= 64


def _vec_group_maxima(keys, G):
    """The 16-byte layout's group maxima as the route kernel forms them: each lane's maximum
    over the four slots of a 128-expert block, a butterfly over the gs/4 lanes of a group
    (gs < 128) or a whole-warp maximum per block (gs >= 128), then lane q holding group q."""
    E = keys.size
    NPL, gs = E // 32, E // G
    slot = np.array([[keys[128 * (i // 4) + 4 * l + i % 4] for i in range(NPL)] for l in range(32)])
    vm = np.stack([slot[:, 4 * m:4 * m + 4].max(axis=1) for m in range(NPL // 4)], axis=1)
    gkey = np.zeros(32, np.uint64)
    if gs < 128:
        lpg, gpm = gs // 4, 128 // gs
        off = 1
        while off < lpg:
            vm = np.maximum(vm, vm[np.arange(32) ^ off])
            off <<= 1
        src = (np.arange(32) % gpm) * lpg
        for m in range(NPL // 4):
            t = vm[src, m]
            take = np.arange(32) // gpm == m
            gkey[take] = t[take]
        group_of = lambda l, i: (i // 4) * gpm + l // lpg
    else:
        bpg = gs // 128
        for m in range(NPL // 4):
            gkey[m // bpg] = max(gkey[m // bpg], vm[:, m].max())
        group_of = lambda l, i: (i // 4) // bpg
    return gkey[:G], group_of


@pytest.mark.parametrize("E,G", [(E, G) for E in (128, 256, 384, 512, 1024) for G in range(2, 33)
                                 if E % G == 0 and ((E // G < 128 and (E // G) % 4 == 0 and 128 % (E // G) == 0)
                                                    or (E // G) % 128 == 0)])
def test_vec_layout_group_maxima(E, G):
    """Group maxima and slot groups of the 16-byte layout equal the contiguous groups'."""
    rng = np.random.default_rng(E * 64 + G)
    keys = rng.integers(1, 2**32 - 1, size=E, dtype=np.uint64)
    gkey, group_of = _vec_group_maxima(keys, G)
    gs = E // G
    assert np.array_equal(gkey, keys.reshape(G, gs).max(axis=1))
    for l in range(32):
        for i in range(E // 32):
            assert group_of(l, i) == (128 * (i // 4) + 4 * l + i % 4) // gs
