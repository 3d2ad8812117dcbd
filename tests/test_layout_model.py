"""The dispatch kernels' row formula, modelled on the CPU and checked against the oracle.

The CUDA dispatch never sorts.  It cuts each source rank's (token, slot) items
into tiles of consecutive items, gives every item its stable rank among the
items of the same expert in its tile, counts each (expert, tile), and scans
those counts in expert-major, tile-minor order.  Because ranks hold
consecutive tokens and tiles never straddle two ranks, that order is the
order (expert, source rank, token), so

    row(g, j) = scan[e * ntiles + tile(g, j)] + rank_in_tile(g, j)

is the oracle's layout (a stable sort by expert, then global token).  The
low-latency layout replaces the scan by a fixed region per (expert, rank):

    row(g, j) = (e * R + s) * C + (items of rank s routed to e in earlier tiles)
                + rank_in_tile(g, j).

This file restates both formulas in plain numpy (no code shared with the
kernels) for several tile sizes, including the kernels' 2048, and checks them
against the oracle's dispatch.  It also checks the bound behind the
workspace size: the tiles a call needs never exceed ceil(T*K / tile) + R."""
import numpy as np
import pytest

KERNEL_TILE_ITEMS = 2048


def _tiles(B, K, tile):
    B = np.asarray(B, np.int64)
    per_rank = (B * K + tile - 1) // tile
    tile_off = np.concatenate([[0], np.cumsum(per_rank)])
    rank_off = np.concatenate([[0], np.cumsum(B)])
    return rank_off, tile_off


def _model(idx, B, E, tile, C=None):
    T, K = idx.shape
    R = len(B)
    rank_off, tile_off = _tiles(B, K, tile)
    ntiles = int(tile_off[-1])
    hist = np.zeros((E, max(ntiles, 1)), np.int64)
    tile_of = np.zeros(T * K, np.int64)
    rank_in_tile = np.zeros(T * K, np.int64)
    for s in range(R):
        for i in range(rank_off[s] * K, rank_off[s + 1] * K):
            t = tile_off[s] + (i - rank_off[s] * K) // tile
            e = idx.reshape(-1)[i]
            tile_of[i] = t
            rank_in_tile[i] = hist[e, t]          # earlier items of e in this tile
            hist[e, t] += 1
    e_of = idx.reshape(-1).astype(np.int64)
    if C is None:
        flat = hist[:, :ntiles].reshape(-1)
        scan = np.concatenate([[0], np.cumsum(flat)])
        rows = scan[e_of * ntiles + tile_of] + rank_in_tile
        counts = np.array([[scan[e * ntiles + tile_off[s + 1]] - scan[e * ntiles + tile_off[s]]
                            for s in range(R)] for e in range(E)]).reshape(-1)
        return rows, counts, scan
    rows = np.zeros(T * K, np.int64)
    s_of = np.searchsorted(rank_off, np.arange(T), side="right") - 1
    for i in range(T * K):
        e, s, t = e_of[i], s_of[i // K], tile_of[i]
        rows[i] = (e * R + s) * C + hist[e, tile_off[s]:t].sum() + rank_in_tile[i]
    counts = np.array([[hist[e, tile_off[s]:tile_off[s + 1]].sum() for s in range(R)] for e in range(E)]).reshape(-1)
    return rows, counts, None


def _routing(T, E, K, rng, skew):
    if skew:   # a few hot experts: many equal experts inside one tile
        p = 1.0 / np.arange(1, E + 1) ** 1.5
        return np.stack([rng.choice(E, K, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32).reshape(T, K)


CASES = [
    # R, E, K, B, tile, skew
    (1, 4, 2, [37], 8, False),
    (3, 6, 3, [5, 0, 11], 4, False),
    (4, 16, 4, [9, 1, 0, 30], 16, True),
    (8, 32, 8, [64, 3, 0, 17, 40, 1, 2, 90], 64, True),
    (2, 8, 1, [13, 13], 5, False),                 # a tile size that divides nothing
    (8, 256, 8, [300, 0, 257, 512, 1, 255, 256, 64], KERNEL_TILE_ITEMS, False),
    (4, 64, 8, [1000, 0, 1, 700], KERNEL_TILE_ITEMS, True),
]


@pytest.mark.parametrize("R,E,K,B,tile,skew", CASES)
def test_tile_scan_rows_are_the_oracle_layout(oracle, R, E, K, B, tile, skew):
    rng = np.random.default_rng(R * 1000 + E + tile)
    T = int(np.sum(B))
    idx = _routing(T, E, K, rng, skew)
    d = oracle.dispatch(np.zeros((T, 8), np.uint16), idx, B, E)
    rows, counts, scan = _model(idx, B, E, tile)
    assert np.array_equal(rows, d["tok2row"])
    assert np.array_equal(counts, d["counts"])
    assert scan[-1] == T * K == d["offsets"][-1]


@pytest.mark.parametrize("R,E,K,B,tile,skew", CASES[:5])
def test_low_latency_rows_are_the_oracle_regions(oracle, R, E, K, B, tile, skew):
    rng = np.random.default_rng(R * 1000 + E + tile + 1)
    T = int(np.sum(B))
    idx = _routing(T, E, K, rng, skew)
    C = max(B)
    d = oracle.dispatch_ll(np.zeros((T, 8), np.uint16), idx, B, E, C)
    rows, counts, _ = _model(idx, B, E, tile, C=C)
    assert np.array_equal(rows, d["tok2row"])
    assert np.array_equal(counts, d["counts"])


def test_workspace_tile_bound():
    # the workspace is sized for ceil(T*K / tile) + R tiles before the
    # per-rank split is known; the split never needs more
    rng = np.random.default_rng(5)
    for _ in range(2000):
        R = int(rng.integers(1, 257))
        K = int(rng.integers(1, 33))
        B = rng.integers(0, 5000, size=R) * (rng.random(R) < 0.8)
        _, tile_off = _tiles(B, K, KERNEL_TILE_ITEMS)
        T = int(B.sum())
        bound = (T * K + KERNEL_TILE_ITEMS - 1) // KERNEL_TILE_ITEMS + R
        assert tile_off[-1] <= bound


# ---------------------------------------------------------------------------
# the one-kernel path for small batches
# ---------------------------------------------------------------------------

def _one_kernel_model(idx, B, E, W, sms):
    """The small-batch kernel's arithmetic: blocks of W warps over contiguous token ranges
    [g0, g1) (tpb tokens each, at most `sms` blocks), each range taken in chunks of whole
    rounds of W tokens (at most 512 items); in each chunk
        row(i) = start(e) + pre(e) + #{earlier items of the chunk with expert e},
    start = exclusive scan of the per-expert totals, pre = the per-expert count of the items
    before the chunk; and block b writes source rank b's (then b + grid's ...) layout:
        offsets[e*R+s] = start(e) + (items of ranks below s routed to e),
        counts[e*R+s]  = items of rank s routed to e.
    Also checks every index the kernel forms against its buffer's size."""
    T, K = idx.shape
    R = len(B)
    flat = idx.reshape(-1).astype(np.int64)
    rank_off = np.concatenate([[0], np.cumsum(np.asarray(B, np.int64))])
    grid = min(sms, -(-T // W))
    tpb = -(-T // grid)
    grid = -(-T // tpb)
    tot = np.bincount(flat, minlength=E)
    start = np.concatenate([[0], np.cumsum(tot)])[:E]
    rows = np.full(T * K, -1, np.int64)
    offsets = np.full(E * R + 1, -1, np.int64)
    counts = np.full(E * R, -1, np.int64)
    for b in range(grid):
        g0, g1 = b * tpb, min(T, (b + 1) * tpb)
        assert g1 > g0                                     # every block has a token
        pre = np.bincount(flat[: g0 * K], minlength=E)
        ctok = W * max(1, 512 // K // W)                   # chunk: whole rounds of W tokens, <= 512 items
        assert ctok * K <= max(512, W * K) and ctok % W == 0
        for c0 in range(g0, g1, ctok):
            chunk = flat[c0 * K: min(g1, c0 + ctok) * K]
            for k, e in enumerate(chunk):
                rows[c0 * K + k] = start[e] + pre[e] + int(np.sum(chunk[:k] == e))
            pre = pre + np.bincount(chunk, minlength=E)
        for w in range(W):                                 # warp w's tokens g0 + w + it*W
            n = -(-(g1 - g0 - w) // W) if g1 - g0 > w else 0
            for it in range(n):
                assert g0 + w + it * W < g1
        # the kernel's first pass: one histogram per segment between the sorted
        # boundaries g0*K, rank_off[s]*K, rank_off[s+1]*K (s = b when b < R), and
        # the four counts as sums of leading segments
        mlo = rank_off[b] * K if b < R else 0
        mhi = rank_off[b + 1] * K if b < R else 0
        c = sorted([int(g0 * K), int(mlo), int(mhi)])
        seg = np.zeros((4, E), np.int64)
        for i, e in enumerate(flat):
            seg[(i >= c[0]) + (i >= c[1]) + (i >= c[2]), e] += 1
        run = np.cumsum(seg, axis=0)
        place = lambda v: c.index(int(v))
        assert np.array_equal(run[3], tot)
        assert np.array_equal(run[place(g0 * K)], np.bincount(flat[: g0 * K], minlength=E))
        if b < R:
            assert np.array_equal(run[place(mlo)], np.bincount(flat[:mlo], minlength=E))
            assert np.array_equal(run[place(mhi)] - run[place(mlo)], np.bincount(flat[mlo:mhi], minlength=E))
        for s in range(b, R, grid):
            bef = np.bincount(flat[: rank_off[s] * K], minlength=E)
            ins = np.bincount(flat[rank_off[s] * K: rank_off[s + 1] * K], minlength=E)
            for e in range(E):
                assert e * R + s < E * R
                offsets[e * R + s] = start[e] + bef[e]
                counts[e * R + s] = ins[e]
            if s == R - 1:
                offsets[E * R] = T * K
    return rows, counts, offsets, grid


ONE_KERNEL_CASES = [
    # R, E, K, B, W, sms, skew
    (8, 16, 2, [5, 0, 17, 3, 64, 1, 9, 2], 8, 152, False),
    (8, 256, 8, [128] * 8, 7, 152, False),                     # DeepSeek-V3 decode
    (32, 384, 8, list(np.random.default_rng(1).integers(0, 65, 32)), 7, 152, True),
    (128, 256, 8, list(np.random.default_rng(2).integers(0, 33, 128)), 7, 152, False),
    (256, 1024, 32, list(np.random.default_rng(3).integers(0, 5, 256)), 3, 7, False),   # ranks > blocks
    (4, 16, 16, [2049, 0, 5, 1], 8, 152, True),
    (1, 8, 1, [37], 2, 3, False),
    (8, 64, 8, [300, 0, 257, 512, 1, 255, 256, 64], 8, 1, True),   # one block: many chunks
    (4, 32, 3, [700, 5, 0, 900], 6, 2, False),                     # chunks of 6*28 tokens
]


@pytest.mark.parametrize("R,E,K,B,W,sms,skew", ONE_KERNEL_CASES)
def test_one_kernel_rows_are_the_oracle_layout(oracle, R, E, K, B, W, sms, skew):
    rng = np.random.default_rng(R + E + K + W)
    T = int(np.sum(B))
    idx = _routing(T, E, K, rng, skew)
    d = oracle.dispatch(np.zeros((T, 8), np.uint16), idx, B, E)
    rows, counts, offsets, _ = _one_kernel_model(idx, B, E, W, sms)
    assert np.array_equal(rows, d["tok2row"])
    assert np.array_equal(counts, d["counts"])
    assert np.array_equal(offsets, d["offsets"])
