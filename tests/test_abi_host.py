"""The C ABI without a GPU: the library loads, exports every function the
public header declares, and its host-side validation rejects bad arguments
before anything reaches CUDA.

Every call below either fails validation or has nothing to do (T == 0), so
none of them touches device memory; the fake pointers are never used.  Keep
it that way: a call that passed validation with a fake pointer would launch a
kernel on a machine that has a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

OK, INVALID, UNSUPPORTED, CUDA, WORKSPACE = 0, 1, 2, 3, 4
BF16, FP8, FP32 = 0, 1, 2
FAKE = 0x100000          # a 16-byte aligned non-NULL address; never dereferenced by a rejected call
FAKE_MISALIGNED = 0x100008


def _declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            names += re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from combine_moe_route_gb300 import build, binding
    build.build()
    return binding.load_library()


def test_header_declares_the_abi():
    names = set(_declared_functions())
    assert {"moe_route_topk", "moe_dispatch", "moe_combine", "moe_dispatch_workspace_bytes",
            "moe_expert_scale", "moe_get_device_error", "moe_strerror", "moe_abi_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_library_exports_nothing_else(lib):
    import subprocess
    from combine_moe_route_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.library_path()], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    exported = {line.split()[-1] for line in out.stdout.splitlines() if line.strip()}
    assert exported == set(_declared_functions())


def test_version_and_strerror(lib):
    assert lib.moe_abi_version() == 1
    for s in range(7):
        assert len(lib.moe_strerror(s)) > 5
    assert b"unknown" in lib.moe_strerror(99)


def test_route_validation(lib):
    f = lib.moe_route_topk
    assert f(FAKE, -1, 16, 2, FAKE, FAKE, None) == INVALID
    assert f(FAKE, 4, 16, 0, FAKE, FAKE, None) == INVALID
    assert f(FAKE, 4, 16, 17, FAKE, FAKE, None) == INVALID
    assert f(FAKE, 4, 1025, 2, FAKE, FAKE, None) == INVALID
    assert f(FAKE, 4, 64, 33, FAKE, FAKE, None) == INVALID
    assert f(None, 4, 16, 2, FAKE, FAKE, None) == INVALID
    assert f(None, 0, 16, 2, None, None, None) == OK        # empty: nothing enqueued


def _B(*v):
    return np.array(v, dtype=np.int32)


def _dispatch(lib, B, E=16, K=2, H=256, dtype=BF16, x=FAKE, recv=FAKE, scale=FAKE, ws=FAKE, ws_bytes=1 << 30,
              idx=FAKE):
    return lib.moe_dispatch(x, idx, B.size, B.ctypes.data, E, K, H, dtype, recv, scale, FAKE, FAKE, FAKE,
                            FAKE, FAKE, ws, ws_bytes, None)


def test_dispatch_validation(lib):
    B = _B(3, 0, 5, 1)
    assert lib.moe_dispatch(FAKE, FAKE, 0, B.ctypes.data, 16, 2, 256, BF16, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                            FAKE, FAKE, 1 << 30, None) == INVALID                       # R = 0
    assert _dispatch(lib, _B(*([1] * 257)), E=257) == INVALID                         # R > 256
    assert _dispatch(lib, B, E=18) == INVALID                                         # E % R
    assert _dispatch(lib, B, H=12) == INVALID                                         # H % 8
    assert _dispatch(lib, B, H=16392) == INVALID                                      # H too large
    assert _dispatch(lib, B, H=264, dtype=FP8) == INVALID                             # FP8 needs H % 128
    assert _dispatch(lib, B, dtype=FP32) == INVALID                                   # no fp32 payload
    assert _dispatch(lib, _B(3, -1, 5, 1)) == INVALID                                 # negative B
    assert _dispatch(lib, _B(1 << 30, 1 << 30, 0, 0)) == INVALID                      # T*K overflows int32
    assert _dispatch(lib, B, K=17) == INVALID                                         # K > E
    assert _dispatch(lib, B, x=None) == INVALID
    assert _dispatch(lib, B, dtype=FP8, scale=None) == INVALID
    assert _dispatch(lib, B, ws=None) == WORKSPACE
    need = lib.moe_dispatch_workspace_bytes(4, 16, 2, 9)
    assert need > 256
    assert _dispatch(lib, B, ws_bytes=256) == WORKSPACE                                # header only
    assert _dispatch(lib, B, x=FAKE_MISALIGNED, ws_bytes=need) == UNSUPPORTED
    assert _dispatch(lib, B, recv=FAKE_MISALIGNED) == UNSUPPORTED
    assert _dispatch(lib, B, ws=FAKE_MISALIGNED) == UNSUPPORTED
    assert _dispatch(lib, B, dtype=FP8, scale=FAKE_MISALIGNED) == UNSUPPORTED


def test_dispatch_noalloc_size_validation(lib):
    # Only the rejections that come before the first CUDA call on every machine:
    # sizes that moe_dispatch rejects (passed through with its status) and
    # sizes whose workspace exceeds the static scratch.  Shapes that pass those
    # first look up the scratch's device address, so they are not called here.
    import ctypes
    f = lib.moe_dispatch_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    f.restype = i32

    def call(B, E=16, K=2, H=256, dtype=BF16, R=None):
        return f(FAKE, FAKE, B.size if R is None else R, B.ctypes.data, E, K, H, dtype, FAKE, FAKE, FAKE, FAKE, FAKE,
                 FAKE, FAKE, None)

    B = _B(3, 0, 5, 1)
    assert call(B, R=0) == INVALID                                  # R = 0
    assert call(_B(*([1] * 257)), E=257) == INVALID                 # R > 256
    assert call(B, E=18) == INVALID                                 # E % R
    assert call(B, K=17) == INVALID                                 # K > E
    assert call(B, K=0) == INVALID
    assert call(_B(3, -1, 5, 1)) == INVALID                         # negative B
    assert call(_B(1 << 30, 1 << 30, 0, 0)) == INVALID              # T*K overflows int32
    assert f(FAKE, FAKE, 4, None, 16, 2, 256, BF16, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == INVALID
    # beyond the 1 MiB static scratch: 1024 experts, top-32, 8192 tokens
    big = _B(8192)
    assert lib.moe_dispatch_workspace_bytes(1, 1024, 32, 8192) > (1 << 20)
    assert call(big, E=1024, K=32) == WORKSPACE
    assert call(_B(4096, 4096), E=1024, K=32) == WORKSPACE


def test_workspace_bytes(lib):
    f = lib.moe_dispatch_workspace_bytes
    assert f(0, 16, 2, 10) == 0 and f(4, 18, 2, 10) == 0 and f(4, 16, 0, 10) == 0 and f(4, 16, 2, -1) == 0
    assert f(4, 16, 2, 1 << 30) == 0
    sizes = [f(8, 256, 8, T) for T in (0, 1, 1000, 32768)]
    assert all(a <= b for a, b in zip(sizes, sizes[1:])) and sizes[0] > 0
    assert f(8, 256, 8, 32768) < 8 << 20        # small next to the payload


def test_combine_and_expert_validation(lib):
    c = lib.moe_combine
    assert c(FAKE, FAKE, FAKE, -1, 2, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, FAKE, FAKE, 4, 0, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, FAKE, FAKE, 4, 33, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, FAKE, FAKE, 4, 2, 250, BF16, FAKE, None) == INVALID
    assert c(FAKE, FAKE, FAKE, 4, 2, 256, FP8, FAKE, None) == INVALID
    assert c(None, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE_MISALIGNED, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == UNSUPPORTED
    assert c(FAKE, FAKE, FAKE, 4, 2, 256, FP32, FAKE_MISALIGNED, None) == UNSUPPORTED
    assert c(None, None, None, 0, 2, 256, BF16, None, None) == OK
    e = lib.moe_expert_scale
    assert e(FAKE, FAKE, BF16, FAKE, 0, 256, 8, 0, FAKE, None) == INVALID
    assert e(FAKE, FAKE, FP8, FAKE, 4, 200, 8, 0, FAKE, None) == INVALID
    assert e(FAKE, None, FP8, FAKE, 4, 256, 8, 0, FAKE, None) == INVALID
    assert e(FAKE_MISALIGNED, FAKE, BF16, FAKE, 4, 256, 8, 0, FAKE, None) == UNSUPPORTED
    assert e(None, None, BF16, None, 4, 256, 0, 0, None, None) == OK


def test_get_device_error_validation(lib):
    code = ctypes.c_int32(0)
    assert lib.moe_get_device_error(None, ctypes.byref(code), None) == INVALID
    assert lib.moe_get_device_error(FAKE, None, None) == INVALID


def test_binding_refuses_cpu_tensors(lib):
    import torch
    from combine_moe_route_gb300 import binding
    with pytest.raises(ValueError):
        binding.route_topk(torch.zeros(4, 16), 2)
    with pytest.raises(ValueError):
        binding.combine(torch.zeros(8, 16, dtype=torch.bfloat16), torch.zeros(8, dtype=torch.int32),
                        torch.zeros(4, 2))


def test_route_grouped_validation(lib):
    f = lib.moe_route_topk_grouped
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(FAKE, 4, 256, 8, 0, 1, FAKE, FAKE, None) == INVALID       # no groups
    assert f(FAKE, 4, 256, 8, 33, 1, FAKE, FAKE, None) == INVALID      # more than 32 groups
    assert f(FAKE, 4, 256, 8, 6, 1, FAKE, FAKE, None) == INVALID       # does not divide E
    assert f(FAKE, 4, 256, 8, 8, 0, FAKE, FAKE, None) == INVALID       # no kept group
    assert f(FAKE, 4, 256, 8, 8, 9, FAKE, FAKE, None) == INVALID       # more kept than groups
    assert f(FAKE, 4, 64, 9, 8, 1, FAKE, FAKE, None) == INVALID        # K > kept experts (8)
    assert f(None, 4, 256, 8, 8, 4, FAKE, FAKE, None) == INVALID
    assert f(None, 0, 256, 8, 8, 4, None, None, None) == OK


def _dispatch_ll(lib, unordered, B, E=16, K=2, H=256, C=8, dtype=BF16, x=FAKE, recv=FAKE, scale=FAKE, counts=FAKE,
                 ws=FAKE, ws_bytes=1 << 30):
    f = lib.moe_dispatch_ll_unordered if unordered else lib.moe_dispatch_ll
    return f(x, FAKE, B.size, B.ctypes.data, E, K, H, C, dtype, recv, scale, counts, FAKE, FAKE, ws, ws_bytes, None)


@pytest.mark.parametrize("unordered", [False, True])
def test_dispatch_ll_validation(lib, unordered):
    # T = 0 is left out on purpose: it zeroes counts, which here is a fake pointer
    B = _B(3, 0, 5, 1)
    assert _dispatch_ll(lib, unordered, _B()) == INVALID                                # R = 0
    assert _dispatch_ll(lib, unordered, B, E=18) == INVALID                             # E % R
    assert _dispatch_ll(lib, unordered, B, K=17) == INVALID                             # K > E
    assert _dispatch_ll(lib, unordered, B, H=12) == INVALID                             # H % 8
    assert _dispatch_ll(lib, unordered, B, H=264, dtype=FP8) == INVALID                 # FP8 needs H % 128
    assert _dispatch_ll(lib, unordered, B, dtype=FP32) == INVALID                       # no fp32 payload
    assert _dispatch_ll(lib, unordered, B, C=0) == INVALID                              # no slots
    assert _dispatch_ll(lib, unordered, B, E=1024, C=1 << 19) == INVALID                # E*R*C overflows int32
    assert _dispatch_ll(lib, unordered, B, C=4) == INVALID                              # B[2] = 5 > C
    assert _dispatch_ll(lib, unordered, _B(3, -1, 5, 1)) == INVALID                     # negative B
    assert _dispatch_ll(lib, unordered, B, counts=None) == INVALID
    assert _dispatch_ll(lib, unordered, B, x=None) == INVALID
    assert _dispatch_ll(lib, unordered, B, dtype=FP8, scale=None) == INVALID
    assert _dispatch_ll(lib, unordered, B, ws=None) == WORKSPACE
    assert _dispatch_ll(lib, unordered, B, ws_bytes=255) == WORKSPACE                   # less than the header
    # the ordered form needs the histogram workspace; the unordered one the 256-byte header only
    header_only = _dispatch_ll(lib, unordered, B, x=FAKE_MISALIGNED, ws_bytes=256)
    assert header_only == (UNSUPPORTED if unordered else WORKSPACE)
    assert _dispatch_ll(lib, unordered, B, recv=FAKE_MISALIGNED) == UNSUPPORTED
    assert _dispatch_ll(lib, unordered, B, ws=FAKE_MISALIGNED) == UNSUPPORTED
    assert _dispatch_ll(lib, unordered, B, dtype=FP8, scale=FAKE_MISALIGNED) == UNSUPPORTED


def test_combine_ll_validation(lib):
    c = lib.moe_combine_ll                  # (y, E, R, C, tok2row, w, T, K, H, out_dtype, out, stream)
    assert c(FAKE, 16, 4, 8, FAKE, FAKE, -1, 2, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, 16, 4, 8, FAKE, FAKE, 4, 0, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, 16, 4, 8, FAKE, FAKE, 4, 33, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, 0, 4, 8, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, 16, 0, 8, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, 16, 4, 0, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE, 1024, 256, 1 << 13, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == INVALID   # E*R*C = 2^31
    assert c(FAKE, 16, 4, 8, FAKE, FAKE, 4, 2, 250, BF16, FAKE, None) == INVALID
    assert c(FAKE, 16, 4, 8, FAKE, FAKE, 4, 2, 256, FP8, FAKE, None) == INVALID
    assert c(FAKE, 16, 4, 8, None, FAKE, 4, 2, 256, BF16, FAKE, None) == INVALID     # no identity map here
    assert c(None, 16, 4, 8, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == INVALID
    assert c(FAKE_MISALIGNED, 16, 4, 8, FAKE, FAKE, 4, 2, 256, BF16, FAKE, None) == UNSUPPORTED
    assert c(FAKE, 16, 4, 8, FAKE, FAKE, 4, 2, 256, FP32, FAKE_MISALIGNED, None) == UNSUPPORTED
    assert c(None, 16, 4, 8, None, None, 0, 2, 256, BF16, None, None) == OK
    p = lib.moe_combine_ll_push             # (y, row2src, counts, R, E, C, K, H, T, ret, stream)
    assert p(FAKE, FAKE, FAKE, 0, 16, 8, 2, 256, 4, FAKE, None) == INVALID
    assert p(FAKE, FAKE, FAKE, 4, 16, 8, 33, 256, 4, FAKE, None) == INVALID
    assert p(FAKE, FAKE, FAKE, 4, 16, 8, 2, 12, 4, FAKE, None) == INVALID
    assert p(FAKE, None, FAKE, 4, 16, 8, 2, 256, 4, FAKE, None) == INVALID
    assert p(FAKE, FAKE, None, 4, 16, 8, 2, 256, 4, FAKE, None) == INVALID
    assert p(FAKE, FAKE, FAKE, 4, 16, 8, 2, 256, 4, FAKE_MISALIGNED, None) == UNSUPPORTED
    assert p(None, None, None, 4, 16, 8, 2, 256, 0, None, None) == OK


def test_combine_partial_validation(lib):
    s = lib.moe_combine_partial_send        # (y, tok2row, idx, w, T, K, H, E, R, partial, stream)
    assert s(FAKE, FAKE, FAKE, FAKE, 4, 2, 256, 18, 4, FAKE, None) == INVALID        # E % R
    assert s(FAKE, FAKE, FAKE, FAKE, 4, 2, 256, 512, 512, FAKE, None) == INVALID     # R > 256
    assert s(FAKE, FAKE, FAKE, FAKE, 4, 17, 256, 16, 4, FAKE, None) == INVALID       # K > E
    assert s(FAKE, FAKE, FAKE, FAKE, 4, 2, 12, 16, 4, FAKE, None) == INVALID         # H % 8
    assert s(FAKE, FAKE, None, FAKE, 4, 2, 256, 16, 4, FAKE, None) == INVALID
    assert s(FAKE, FAKE, FAKE, FAKE, 4, 2, 256, 16, 4, FAKE_MISALIGNED, None) == UNSUPPORTED
    assert s(None, None, None, None, 0, 2, 256, 16, 4, None, None) == OK
    r = lib.moe_combine_partial_recv        # (partial, idx, T, K, H, E, R, out_dtype, out, stream)
    assert r(FAKE, FAKE, -1, 2, 256, 16, 4, BF16, FAKE, None) == INVALID
    assert r(FAKE, FAKE, 4, 2, 256, 18, 4, BF16, FAKE, None) == INVALID
    assert r(FAKE, FAKE, 4, 2, 256, 16, 4, FP8, FAKE, None) == INVALID
    assert r(FAKE, None, 4, 2, 256, 16, 4, BF16, FAKE, None) == INVALID
    assert r(FAKE_MISALIGNED, FAKE, 4, 2, 256, 16, 4, BF16, FAKE, None) == UNSUPPORTED
    assert r(None, None, 0, 2, 256, 16, 4, FP32, None, None) == OK


def test_plain_c_consumer_compiles_and_links(lib, tmp_path):
    """The C ABI needs nothing but its header and the CUDA runtime: a plain C11 program
    (tests/c_abi/roundtrip.c) compiles without warnings and links against the library."""
    import _c_abi
    from combine_moe_route_gb300 import build
    exe = _c_abi.compile_roundtrip(build.library_path(), str(tmp_path))
    assert os.path.exists(exe)


def test_split_halves_validation(lib):
    """moe_dispatch_send / _recv and moe_combine_send / _recv reject bad arguments on the host.
    (T == 0 is left out of the receive half: it zeroes counts, here a fake pointer.)"""
    B = _B(3, 0, 5, 1)

    def send(B, E=16, K=2, H=256, dtype=BF16, x=FAKE, recv=FAKE, scale=FAKE, max_sms=0, ws=FAKE, ws_bytes=1 << 30):
        return lib.moe_dispatch_send(x, FAKE, B.size, B.ctypes.data, E, K, H, dtype, recv, scale, FAKE, FAKE,
                                     max_sms, ws, ws_bytes, None)

    assert send(_B()) == INVALID                                        # R = 0
    assert send(B, E=18) == INVALID                                     # E % R
    assert send(B, K=17) == INVALID                                     # K > E
    assert send(B, H=264, dtype=FP8) == INVALID                         # FP8 needs H % 128
    assert send(_B(3, -1, 5, 1)) == INVALID                             # negative B
    assert send(B, x=None) == INVALID
    assert send(B, max_sms=-1) == INVALID
    assert send(B, ws=None) == WORKSPACE
    assert send(B, ws_bytes=256) == WORKSPACE                           # header only
    assert send(B, x=FAKE_MISALIGNED) == UNSUPPORTED
    assert send(B, ws=FAKE_MISALIGNED) == UNSUPPORTED
    assert send(_B(0, 0, 0, 0), x=None, recv=None) == OK                # T = 0: nothing to send

    def recv(B, E=16, K=2, counts=FAKE, ws=FAKE, ws_bytes=1 << 30):
        return lib.moe_dispatch_recv(B.size, B.ctypes.data, E, K, counts, FAKE, FAKE, ws, ws_bytes, None)

    assert recv(_B()) == INVALID
    assert recv(B, E=18) == INVALID
    assert recv(B, K=0) == INVALID
    assert recv(_B(3, -1, 5, 1)) == INVALID
    assert recv(B, counts=None) == INVALID
    assert recv(B, ws=None) == WORKSPACE
    assert recv(B, ws_bytes=256) == WORKSPACE                           # header only
    assert recv(B, ws=FAKE_MISALIGNED) == UNSUPPORTED

    cs = lib.moe_combine_send               # (R, ws, ws_bytes, stream)
    assert cs(0, FAKE, 1 << 20, None) == INVALID
    assert cs(257, FAKE, 1 << 20, None) == INVALID
    assert cs(4, None, 1 << 20, None) == WORKSPACE
    assert cs(4, FAKE, 256, None) == WORKSPACE                          # header only, no flags
    assert cs(4, FAKE_MISALIGNED, 1 << 20, None) == UNSUPPORTED
    cr = lib.moe_combine_recv               # (y, tok2row, w, T, K, H, out_dtype, out, R, ws, ws_bytes, stream)
    assert cr(FAKE, FAKE, FAKE, -1, 2, 256, BF16, FAKE, 4, FAKE, 1 << 20, None) == INVALID
    assert cr(FAKE, FAKE, FAKE, 4, 33, 256, BF16, FAKE, 4, FAKE, 1 << 20, None) == INVALID
    assert cr(FAKE, FAKE, FAKE, 4, 2, 250, BF16, FAKE, 4, FAKE, 1 << 20, None) == INVALID
    assert cr(FAKE, FAKE, FAKE, 4, 2, 256, FP8, FAKE, 4, FAKE, 1 << 20, None) == INVALID
    assert cr(FAKE, FAKE, FAKE, 4, 2, 256, BF16, FAKE, 0, FAKE, 1 << 20, None) == INVALID
    assert cr(FAKE, None, FAKE, 4, 2, 256, BF16, FAKE, 4, FAKE, 1 << 20, None) == INVALID
    assert cr(FAKE_MISALIGNED, FAKE, FAKE, 4, 2, 256, BF16, FAKE, 4, FAKE, 1 << 20, None) == UNSUPPORTED
    assert cr(FAKE, FAKE, FAKE, 4, 2, 256, BF16, FAKE, 4, None, 1 << 20, None) == WORKSPACE
    assert cr(FAKE, FAKE, FAKE, 4, 2, 256, BF16, FAKE, 4, FAKE, 256, None) == WORKSPACE
    assert cr(None, None, None, 0, 2, 256, BF16, None, 4, None, 0, None) == OK


def test_dispatch_noalloc_reports_argument_errors_before_its_size_limit(lib):
    """A call moe_dispatch rejects for its arguments gets moe_dispatch's status, even when its
    sizes are also beyond the static scratch; only an otherwise valid call gets
    MOE_ERR_WORKSPACE."""
    import ctypes
    f = lib.moe_dispatch_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    f.restype = i32
    big = _B(8192)                          # E = 1024, K = 32: beyond the scratch

    def call(H=256, dtype=BF16, x=FAKE, recv=FAKE, scale=FAKE, counts=FAKE):
        return f(x, FAKE, 1, big.ctypes.data, 1024, 32, H, dtype, recv, scale, counts, FAKE, FAKE, FAKE, FAKE, None)

    assert call() == WORKSPACE
    assert call(H=12) == INVALID                                        # H % 8
    assert call(H=264, dtype=FP8) == INVALID                            # FP8 needs H % 128
    assert call(dtype=FP32) == INVALID
    assert call(x=None) == INVALID
    assert call(counts=None) == INVALID
    assert call(dtype=FP8, scale=None) == INVALID
    assert call(x=FAKE_MISALIGNED) == UNSUPPORTED
    assert call(recv=FAKE_MISALIGNED) == UNSUPPORTED
    assert call(dtype=FP8, scale=FAKE_MISALIGNED) == UNSUPPORTED
