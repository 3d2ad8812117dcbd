"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a plugin whose memory belongs to a host framework, or
a serving loop that must not allocate on its hot path).  It uses the library's
static device scratch instead of a workspace.

Called here through the C ABI with ctypes; every output must equal, bit for
bit, both the CPU oracle's dispatch and what moe_dispatch (with a caller
workspace) produces for the same input -- the same bar the other dispatch
parity tests use -- on two calls in a row, the second with different sizes, so
that state left in the shared scratch by the first call cannot leak into the
second.  One case needs a workspace within a few KB of the scratch's size, so
the end of the array (where the scan output lies) is used and compared; one
just past it is refused with MOE_ERR_WORKSPACE.  This file is collected last."""
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
    # K distinct experts per token: the K smallest of E uniform keys
    idx = np.argpartition(rng.random((inp["T"], E), dtype=np.float32), K - 1, axis=1)[:, :K]
    idx = np.ascontiguousarray(idx.astype(np.int32)).reshape(inp["T"], K)
    return x, torch.from_numpy(idx).to(dev), np.asarray(inp["B"], np.int32)


def _near_full_B():
    """8 ranks of 256*m + 1 tokens (one item past a whole number of 2048-item tiles, so the
    call's tile count is one short of the bound the workspace size is computed from), with
    E = 256 and K = 8: the workspace is within 3 KB of the 1 MiB scratch."""
    m = [63, 63, 63, 63, 63, 63, 62, 62]
    return [256 * v + 1 for v in m]


def _compare_with_oracle(got, x, idx, B, E, fp8):
    import oracle
    from combine_moe_route_gb300 import workloads as wl
    ref = oracle.dispatch(wl.bf16_bits(x.cpu()), idx.cpu().numpy(), B, E, fp8=fp8)
    for key in ("counts", "offsets", "expert_offsets", "tok2row", "row2src"):
        assert np.array_equal(got[key].cpu().numpy(), ref[key]), key
    if fp8:
        assert np.array_equal(got["recv"].cpu().numpy(), ref["recv"])
        assert np.array_equal(got["scale"].cpu().numpy().view(np.uint32), ref["recv_scale"].view(np.uint32))
    else:
        assert np.array_equal(got["recv"].cpu().numpy().view(np.uint16), ref["recv"])


def test_noalloc_matches_oracle_and_dispatch_on_calls_in_a_row(lib):
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    cases = [
        dict(R=8, E=256, K=8, H=7168, B=[128, 0, 77, 300, 5, 128, 64, 1], fp8=True, seed=21),
        dict(R=8, E=256, K=8, H=16, B=_near_full_B(), fp8=False, seed=23),
        dict(R=4, E=16, K=2, H=256, B=[9, 1, 0, 33], fp8=False, seed=22),
    ]
    near = lib.moe_dispatch_workspace_bytes(8, 256, 8, sum(_near_full_B()))
    assert (1 << 20) - 3 * 1024 <= near <= (1 << 20)
    for c in cases:   # calls in a row on the shared scratch, different sizes and payloads
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
        _compare_with_oracle(got, x, idx, B, E, c["fp8"])
        # the layout is a complete one: every routed copy placed exactly once
        assert int(got["offsets"][-1]) == T * K
        assert torch.equal(torch.sort(got["row2src"]).values, torch.arange(T * K, device=dev, dtype=torch.int32))
        del got, ref
        torch.cuda.empty_cache()


def test_noalloc_refuses_a_call_just_past_its_scratch(lib):
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    Bl = _near_full_B()
    Bl[0] += 256                          # one more tile: the bound passes 1 MiB
    assert lib.moe_dispatch_workspace_bytes(8, 256, 8, sum(Bl)) > (1 << 20)
    x, idx, B = _case(8, 256, 8, 16, Bl, 24, dev)
    got = _outputs(x.shape[0], 8, 16, 256, 8, False, dev)
    assert _call(lib, True, x, idx, B, 256, False, got, stream) == WORKSPACE
    torch.cuda.synchronize()
    assert bool((got["counts"] == -7).all()) and bool((got["tok2row"] == -7).all())   # nothing was enqueued


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # E = 1024 experts, K = 32, 8192 tokens on one rank: the workspace this
    # needs is larger than the static scratch; nothing may be enqueued
    B = np.array([8192], np.int32)
    assert lib.moe_dispatch_workspace_bytes(1, 1024, 32, 8192) > (1 << 20)
    fake = 0x100000   # rejected on the host before any pointer is used
    st = lib.moe_dispatch_noalloc(fake, fake, 1, B.ctypes.data, 1024, 32, 256, BF16, fake, None, fake, fake, fake,
                                  fake, fake, None)
    assert st == WORKSPACE
