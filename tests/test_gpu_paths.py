"""Both dispatch paths on the GPU against the oracle, whichever one a shape
would normally take.

A dispatch whose T*K items fit MOE_SMALL_DISPATCH_ITEMS runs as one kernel
(behind a header-clearing kernel); larger ones run the histogram, lookback
scan and scatter kernels.  The library is built twice more here, with the
threshold at 0 (every shape takes the three kernels) and at 2^30 (every shape
takes the one kernel), and the same shapes -- small ones that the default
build sends down the one-kernel path, and larger ones it sends down the
three-kernel path -- go through ragged dispatch and the split halves of both
builds.  Layout, payload bytes and scales must equal the oracle's bit for bit."""
import numpy as np
import pytest
import torch

from _compare import bits16, bytes8, f32, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module", params=["three_kernels", "one_kernel"])
def path_lib(request, gpu, tmp_path_factory):
    from combine_moe_route_gb300 import binding, build
    items = 0 if request.param == "three_kernels" else 1 << 30
    out = str(tmp_path_factory.mktemp(request.param))
    return binding.load_library(build.build(out_dir=out, defines=(f"MOE_SMALL_DISPATCH_ITEMS={items}",)))


SHAPES = [
    # R, E, K, H, B, fp8
    (8, 16, 2, 256, [5, 0, 17, 3, 64, 1, 9, 2], False),
    (8, 256, 8, 7168, [128] * 8, False),
    (8, 256, 8, 7168, [128, 0, 77, 300, 5, 128, 64, 1], True),
    (32, 384, 8, 512, [int(v) for v in np.random.default_rng(1).integers(0, 65, 32)], False),
    (256, 1024, 32, 128, [int(v) for v in np.random.default_rng(3).integers(0, 5, 256)], True),
    (4, 64, 8, 1280, [3000, 0, 1, 2100], True),                       # multi-tile ranks, 10 blocks of 128
    (2, 8, 1, 16384, [700, 555], False),
]


@pytest.mark.parametrize("R,E,K,H,B,fp8", SHAPES)
def test_dispatch_path_matches_oracle(path_lib, R, E, K, H, B, fp8, gpu, oracle, monkeypatch):
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    monkeypatch.setattr(b, "_lib", path_lib)
    inp = wl.random_shape_inputs(R, E, K, H, B, seed=R * 7 + K, fp8=fp8)
    o_idx, _ = oracle.route_topk(inp["logits"], K)
    x = inp["x"].to(gpu)
    idx = torch.from_numpy(o_idx).to(gpu)
    od = oracle.dispatch(wl.bf16_bits(inp["x"]), o_idx, inp["B"], E, fp8=fp8)
    d = b.dispatch(x, idx, inp["B"], E, fp8=fp8)
    ds = b.dispatch_send(x, idx, inp["B"], E, fp8=fp8, max_sms=5)
    b.dispatch_recv(ds, inp["B"], E, K)
    torch.cuda.synchronize()
    for r in (d, ds):
        st, code = b.get_device_error(r.workspace)
        assert st == 0 and code == 0
        for key in ("counts", "offsets", "expert_offsets", "tok2row", "row2src"):
            assert np.array_equal(i32(getattr(r, key)), od[key]), key
        if fp8:
            assert np.array_equal(bytes8(r.recv_x), od["recv"])
            assert np.array_equal(f32(r.recv_scale).view(np.uint32), od["recv_scale"].view(np.uint32))
        else:
            assert np.array_equal(bits16(r.recv_x), od["recv"])
