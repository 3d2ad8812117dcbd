"""Failure detection on the GPU without a fault: the library's bounded device
waits run out, report MOE_ERR_TIMEOUT through the workspace error word, keep
every write inside its buffer, and leave the CUDA context usable.

The waits are made to run out by test-only build switches (a flag or a bulk
copy that nothing ever provides); the product library is built without them.
  * MOE_TEST_WITHHOLD_SCAN_BLOCK=0: the first lookback-scan block never
    publishes its status, so the second block's lookback wait ends after its
    limit (about 2 s) with MOE_DEVERR_SCAN_TIMEOUT.
  * MOE_TEST_WITHHOLD_FIRST_LOAD: the warp that takes token 0 (in either dispatch path) arms
    that token's stage barrier but never issues the copy, so its wait ends
    after its limit with MOE_DEVERR_COPY_TIMEOUT.
  * MOE_TEST_WITHHOLD_IDS_COPY: the one-kernel dispatch arms the barrier of
    its routing-table copy into shared memory but never issues the copy; each
    block's wait ends after its limit, the block counts from global memory
    instead, and the dispatch is still exact, with MOE_DEVERR_COPY_TIMEOUT.
  * MOE_TEST_WITHHOLD_ARRIVAL_RANK=1 and MOE_TEST_WITHHOLD_READY_RANK=0 (one
    build): the dispatch send half never announces the copies it stored for
    rank 1, and the combine send half never publishes rank 0's outputs, so
    each receive half's wait ends after its limit with
    MOE_DEVERR_RECV_TIMEOUT; the data itself is in place, so the layout and
    the sums still equal the oracle's."""
import ctypes
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BF16 = 0
OK, TIMEOUT = 0, 5
SCAN_TIMEOUT, COPY_TIMEOUT, RECV_TIMEOUT = 0x4, 0x8, 0x10


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _hooked_library(tmp_path_factory, *defines):
    from combine_moe_route_gb300 import build
    out = str(tmp_path_factory.mktemp("hooks"))
    lib = ctypes.CDLL(build.build(out_dir=out, defines=defines))
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.moe_dispatch.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.moe_dispatch.restype = i32
    lib.moe_dispatch_workspace_bytes.argtypes = [i32, i32, i32, i64]
    lib.moe_dispatch_workspace_bytes.restype = sz
    lib.moe_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
    lib.moe_get_device_error.restype = i32
    lib.moe_dispatch_send.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, sz, vp]
    lib.moe_dispatch_send.restype = i32
    lib.moe_dispatch_recv.argtypes = [i32, vp, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.moe_dispatch_recv.restype = i32
    lib.moe_combine_send.argtypes = [i32, vp, sz, vp]
    lib.moe_combine_send.restype = i32
    lib.moe_combine_recv.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, i32, vp, sz, vp]
    lib.moe_combine_recv.restype = i32
    return lib


def _dispatch_with(lib, x, idx, B, E, dev):
    T, H = x.shape
    K = idx.shape[1]
    R = B.size
    rows = T * K
    o = dict(recv=torch.zeros((rows, H), dtype=torch.bfloat16, device=dev),
             counts=torch.zeros(E * R, dtype=torch.int32, device=dev),
             offsets=torch.zeros(E * R + 1, dtype=torch.int32, device=dev),
             eo=torch.zeros(E + 1, dtype=torch.int32, device=dev),
             tok2row=torch.zeros(rows, dtype=torch.int32, device=dev),
             row2src=torch.zeros(rows, dtype=torch.int32, device=dev))
    wsb = lib.moe_dispatch_workspace_bytes(R, E, K, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    t0 = time.perf_counter()
    st = lib.moe_dispatch(x.data_ptr(), idx.data_ptr(), R, B.ctypes.data, E, K, H, BF16, o["recv"].data_ptr(), None,
                          o["counts"].data_ptr(), o["offsets"].data_ptr(), o["eo"].data_ptr(),
                          o["tok2row"].data_ptr(), o["row2src"].data_ptr(), ws.data_ptr(), wsb, stream)
    assert st == OK                                   # launched fine; the failure is on the device
    code = ctypes.c_int32(0)
    dst = lib.moe_get_device_error(ws.data_ptr(), ctypes.byref(code), stream)   # synchronises
    return dst, code.value, time.perf_counter() - t0, o


def _inputs(R, E, K, H, tokens_per_rank, seed, dev):
    rng = np.random.default_rng(seed)
    B = np.full(R, tokens_per_rank, np.int32)
    T = int(B.sum())
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16).to(dev)
    return x, torch.from_numpy(idx).to(dev), B


def _context_still_works(x, idx, B, E, oracle):
    from combine_moe_route_gb300 import binding
    d = binding.dispatch(x, idx, B, E)
    st, code = binding.get_device_error(d.workspace)
    assert st == OK and code == 0
    ref = oracle.dispatch(x.cpu().view(torch.int16).numpy().view(np.uint16), idx.cpu().numpy(), B, E)
    assert np.array_equal(d.tok2row.cpu().numpy(), ref["tok2row"])
    assert np.array_equal(d.recv_x.cpu().view(torch.int16).numpy().view(np.uint16), ref["recv"])


def _indices_in_bounds(o, rows):
    t2r = o["tok2row"].cpu().numpy()
    r2s = o["row2src"].cpu().numpy()
    assert np.all((t2r >= -1) & (t2r < rows))
    assert np.all((r2s >= 0) & (r2s < rows))


def test_lookback_wait_runs_out_and_reports(gpu, oracle, tmp_path_factory):
    lib = _hooked_library(tmp_path_factory, "MOE_TEST_WITHHOLD_SCAN_BLOCK=0")
    # E = 1024 experts x 72 tiles = 73728 counts: larger than the histogram kernel scans
    # itself, so the decoupled-lookback scan runs (9 blocks)
    x, idx, B = _inputs(8, 1024, 8, 128, 2100, 1, gpu)
    st, code, dt, o = _dispatch_with(lib, x, idx, B, 1024, gpu)
    assert st == TIMEOUT and (code & SCAN_TIMEOUT), (st, code)
    assert 1.0 < dt < 60.0                            # the wait ran for its limit, then returned
    _indices_in_bounds(o, idx.numel())
    _context_still_works(x, idx, B, 1024, oracle)


def test_copy_wait_runs_out_and_reports(gpu, oracle, tmp_path_factory):
    lib = _hooked_library(tmp_path_factory, "MOE_TEST_WITHHOLD_FIRST_LOAD")
    x, idx, B = _inputs(2, 8, 2, 256, 40, 2, gpu)
    st, code, dt, o = _dispatch_with(lib, x, idx, B, 8, gpu)
    assert st == TIMEOUT and (code & COPY_TIMEOUT), (st, code)
    assert 1.0 < dt < 60.0
    t2r = o["tok2row"].cpu().numpy()
    assert np.all((t2r >= -1) & (t2r < idx.numel()))
    _context_still_works(x, idx, B, 8, oracle)


def test_receive_halves_run_out_when_a_send_half_withholds(gpu, oracle, tmp_path_factory):
    lib = _hooked_library(tmp_path_factory, "MOE_TEST_WITHHOLD_ARRIVAL_RANK=1", "MOE_TEST_WITHHOLD_READY_RANK=0")
    R, E, K, H = 4, 16, 2, 256
    x, idx, B = _inputs(R, E, K, H, 50, 4, gpu)
    T = x.shape[0]
    rows = T * K
    o = dict(recv=torch.zeros((rows, H), dtype=torch.bfloat16, device=gpu),
             counts=torch.zeros(E * R, dtype=torch.int32, device=gpu),
             offsets=torch.zeros(E * R + 1, dtype=torch.int32, device=gpu),
             eo=torch.zeros(E + 1, dtype=torch.int32, device=gpu),
             tok2row=torch.zeros(rows, dtype=torch.int32, device=gpu),
             row2src=torch.zeros(rows, dtype=torch.int32, device=gpu))
    wsb = lib.moe_dispatch_workspace_bytes(R, E, K, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=gpu)
    stream = torch.cuda.current_stream(gpu).cuda_stream
    code = ctypes.c_int32(0)

    t0 = time.perf_counter()
    assert lib.moe_dispatch_send(x.data_ptr(), idx.data_ptr(), R, B.ctypes.data, E, K, H, BF16,
                                 o["recv"].data_ptr(), None, o["tok2row"].data_ptr(), o["row2src"].data_ptr(), 0,
                                 ws.data_ptr(), wsb, stream) == OK
    assert lib.moe_dispatch_recv(R, B.ctypes.data, E, K, o["counts"].data_ptr(), o["offsets"].data_ptr(),
                                 o["eo"].data_ptr(), ws.data_ptr(), wsb, stream) == OK
    st = lib.moe_get_device_error(ws.data_ptr(), ctypes.byref(code), stream)   # synchronises
    dt = time.perf_counter() - t0
    assert st == TIMEOUT and (code.value & RECV_TIMEOUT), (st, code.value)
    assert 1.0 < dt < 60.0
    # the copies themselves were stored: the layout and the rows equal the oracle's
    ref = oracle.dispatch(x.cpu().view(torch.int16).numpy().view(np.uint16), idx.cpu().numpy(), B, E)
    assert np.array_equal(o["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(o["tok2row"].cpu().numpy(), ref["tok2row"])
    assert np.array_equal(o["recv"].cpu().view(torch.int16).numpy().view(np.uint16), ref["recv"])

    # combine: rank 0 never publishes
    w = torch.rand((T, K), generator=torch.Generator().manual_seed(4)).to(gpu)
    out = torch.zeros((T, H), dtype=torch.float32, device=gpu)
    y = o["recv"]
    t0 = time.perf_counter()
    assert lib.moe_combine_send(R, ws.data_ptr(), wsb, stream) == OK
    assert lib.moe_combine_recv(y.data_ptr(), o["tok2row"].data_ptr(), w.data_ptr(), T, K, H, 2, out.data_ptr(), R,
                                ws.data_ptr(), wsb, stream) == OK
    st = lib.moe_get_device_error(ws.data_ptr(), ctypes.byref(code), stream)
    dt = time.perf_counter() - t0
    assert st == TIMEOUT and (code.value & RECV_TIMEOUT), (st, code.value)
    assert 1.0 < dt < 60.0
    refc = oracle.combine(ref["recv"], ref["tok2row"], w.cpu().numpy(), out="f32")
    assert np.array_equal(out.cpu().numpy().view(np.uint32), refc.view(np.uint32))
    _context_still_works(x, idx, B, E, oracle)


def test_routing_table_copy_runs_out_and_the_dispatch_falls_back(gpu, oracle, tmp_path_factory):
    lib = _hooked_library(tmp_path_factory, "MOE_TEST_WITHHOLD_IDS_COPY")
    # 8 ranks x 128 tokens, top-8 of 256: the one-kernel path, table staged in shared memory
    x, idx, B = _inputs(8, 256, 8, 512, 128, 5, gpu)
    st, code, dt, o = _dispatch_with(lib, x, idx, B, 256, gpu)
    assert st == TIMEOUT and (code & COPY_TIMEOUT), (st, code)
    assert 1.0 < dt < 60.0
    ref = oracle.dispatch(x.cpu().view(torch.int16).numpy().view(np.uint16), idx.cpu().numpy(), B, 256)
    for key, name in (("counts", "counts"), ("offsets", "offsets"), ("eo", "expert_offsets"),
                      ("tok2row", "tok2row"), ("row2src", "row2src")):
        assert np.array_equal(o[key].cpu().numpy(), ref[name]), key
    assert np.array_equal(o["recv"].cpu().view(torch.int16).numpy().view(np.uint16), ref["recv"])
    _context_still_works(x, idx, B, 256, oracle)
