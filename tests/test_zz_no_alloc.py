"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a plugin whose memory belongs to a host framework, or
a serving loop that must not allocate on its hot path).  It uses the library's
static device scratch instead of a workspace.

Called here through the C ABI with ctypes; every output must equal, bit for
bit, what moe_dispatch (with a caller workspace) produces for the same input
-- the same bar the other dispatch parity tests use -- on two calls in a row,
the second with different sizes, so that state left in the shared scratch by
the first call cannot leak into the second.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BF16, FP8 = 0, 1
OK, WORKSPACE = 0, 4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import binding, build
    build.build()
    lib = binding.load_library()
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.moe_dispatch_noalloc.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.moe_dispatch_noalloc.restype = i32
    return lib


def _outputs(T, K, H, E, R, fp8, dev):
    rows = T * K
    return dict(
        recv=torch.full((rows, H), 0x7F if fp8 else 0x55, dtype=torch.uint8 if fp8 else torch.int16, device=dev),
        scale=torch.full((rows, H // 128), -1.0, dtype=torch.float32, device=dev) if fp8 else None,
        counts=torch.full((E * R,), -7, dtype=torch.int32, device=dev),
        offsets=torch.full((E * R + 1,), -7, dtype=torch.int32, device=dev),
        expert_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        tok2row=torch.full((rows,), -7, dtype=torch.int32, device=dev),
        row2src=torch.full((rows,), -7, dtype=torch.int32, device=dev))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call(lib, noalloc, x, idx, B, E, fp8, o, stream):
    T, H = x.shape
    K = idx.shape[1]
    args = [_ptr(x), _ptr(idx), B.size, B.ctypes.data, E, K, H, FP8 if fp8 else BF16, _ptr(o["recv"]),
            _ptr(o["scale"]), _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["expert_offsets"]),
            _ptr(o["tok2row"]), _ptr(o["row2src"])]
    if noalloc:
        return lib.moe_dispatch_noalloc(*args, stream)
    R = B.size
    ws_bytes = lib.moe_dispatch_workspace_bytes(R, E, K, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    o["_ws"] = ws
    return lib.moe_dispatch(*args, ws.data_ptr(), ws_bytes, stream)


def _case(R, E, K, H, B, seed, dev):
    from combine_moe_route_gb300 import workloads as wl
    inp = wl.random_shape_inputs(R, E, K, H, B, seed=seed)
    x = inp["x"].to(dev)
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(inp["T"])]).astype(np.int32).reshape(inp["T"], K)
    return x, torch.from_numpy(idx).to(dev), np.asarray(inp["B"], np.int32)


def test_noalloc_matches_dispatch_two_calls_in_a_row(lib):
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    cases = [
        dict(R=8, E=256, K=8, H=7168, B=[128, 0, 77, 300, 5, 128, 64, 1], fp8=True, seed=21),
        dict(R=4, E=16, K=2, H=256, B=[9, 1, 0, 33], fp8=False, seed=22),
    ]
    for c in cases:   # two calls in a row on the shared scratch, different sizes and payloads
        x, idx, B = _case(c["R"], c["E"], c["K"], c["H"], c["B"], c["seed"], dev)
        T, K, H, E, R = x.shape[0], c["K"], c["H"], c["E"], c["R"]
        got = _outputs(T, K, H, E, R, c["fp8"], dev)
        ref = _outputs(T, K, H, E, R, c["fp8"], dev)
        assert _call(lib, True, x, idx, B, E, c["fp8"], got, stream) == OK
        assert _call(lib, False, x, idx, B, E, c["fp8"], ref, stream) == OK
        torch.cuda.synchronize()
        for key in ("recv", "scale", "counts", "offsets", "expert_offsets", "tok2row", "row2src"):
            if got[key] is None:
                continue
            a, b = got[key], ref[key]
            if a.dtype == torch.float32:
                a, b = a.view(torch.int32), b.view(torch.int32)
            assert torch.equal(a, b), key
        # the layout is a complete one: every routed copy placed exactly once
        assert int(got["offsets"][-1]) == T * K
        assert torch.equal(torch.sort(got["row2src"]).values, torch.arange(T * K, device=dev, dtype=torch.int32))


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # E = 1024 experts, K = 32, 8192 tokens on one rank: the workspace this
    # needs is larger than the static scratch; nothing may be enqueued
    B = np.array([8192], np.int32)
    assert lib.moe_dispatch_workspace_bytes(1, 1024, 32, 8192) > (1 << 20)
    fake = 0x100000   # rejected on the host before any pointer is used
    st = lib.moe_dispatch_noalloc(fake, fake, 1, B.ctypes.data, 1024, 32, 256, BF16, fake, None, fake, fake, fake,
                                  fake, fake, None)
    assert st == WORKSPACE
