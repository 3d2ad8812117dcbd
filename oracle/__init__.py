"""CPU oracle for MoE route -> dispatch -> expert stand-in -> combine.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package.  The product
(the CUDA library and its Python binding) never imports, links or executes
anything here, and this package never imports the product.

The arithmetic lives in ``moe_oracle.c`` (plain single-threaded C, every step
written out as the definition); this module only marshals numpy arrays in and
out of it with ctypes.  Sources cited in that file:

* Perplexity, "Lower latency and higher throughput with multi-node DeepSeek
  deployment" -- "Expert parallelism", "Quantization", "MoE router".
* Perplexity, "Enabling trillion-parameter models on AWS EFA" -- "Send and
  receive buffers", "Dispatch and combine".
* lehuy.net, "Decoding high-performance EP kernels" -- "Our task",
  "Optimising for throughput" > "Dispatch" / "Combine".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

GCC_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into _build/liboracle.so with gcc; return its path."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_vp = ctypes.c_void_p


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
            lib.oracle_bf16_from_f32.restype = ctypes.c_uint16
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = ctypes.c_float
            lib.oracle_bf16_from_f32_array.argtypes = [_f32p, ctypes.c_int64, _u16p]
            lib.oracle_e4m3_encode_array.argtypes = [_f32p, ctypes.c_int64, _u8p]
            lib.oracle_e4m3_decode_array.argtypes = [_u8p, ctypes.c_int64, _f32p]
            lib.oracle_quantize_rows_e4m3.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, _u8p, _f32p]
            lib.oracle_route_topk.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _f32p]
            lib.oracle_route_topk_grouped.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int, _i32p, _f32p]
            lib.oracle_dispatch.argtypes = [
                _u16p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, _vp, _f32p, _i32p, _i32p, _i32p, _i32p, _i32p]
            lib.oracle_dispatch.restype = ctypes.c_int
            lib.oracle_dispatch_ll.argtypes = [
                _u16p, _i32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, _vp, _f32p, _i32p, _i32p, _i32p]
            lib.oracle_dispatch_ll.restype = ctypes.c_int
            lib.oracle_combine_ll_push.argtypes = [_u16p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, _u16p]
            lib.oracle_expert_scale.argtypes = [
                _vp, _f32p, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p]
            lib.oracle_combine.argtypes = [
                _u16p, _i32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p, _f32p]
            lib.oracle_combine_partial.argtypes = [
                _u16p, _i32p, _i32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _u16p, _u16p, _f32p]
            lib.oracle_combine_f64.argtypes = [
                _u16p, _i32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctype)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def bf16_from_f32(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_bf16_from_f32_array(_ptr(x.reshape(-1), _f32p), x.size, _ptr(out.reshape(-1), _u16p))
    return out


def f32_from_bf16(h) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 (exact)."""
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def e4m3_encode(x) -> np.ndarray:
    """fp32 -> OCP E4M3 codes (uint8), round to nearest even, saturating at 448."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x.reshape(-1), _f32p), x.size, _ptr(out.reshape(-1), _u8p))
    return out


def e4m3_decode(c) -> np.ndarray:
    """OCP E4M3 codes (uint8) -> fp32 (exact)."""
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float32)
    _load().oracle_e4m3_decode_array(_ptr(c.reshape(-1), _u8p), c.size, _ptr(out.reshape(-1), _f32p))
    return out


def quantize_rows_e4m3(x_bf16: np.ndarray):
    """Per-128-channel FP8 quantisation of bf16 rows [n, H] -> (q uint8 [n,H], scale f32 [n,H/128])."""
    x = _c(x_bf16, np.uint16)
    n, H = x.shape
    assert H % 128 == 0
    q = np.empty((n, H), np.uint8)
    s = np.empty((n, H // 128), np.float32)
    _load().oracle_quantize_rows_e4m3(_ptr(x, _u16p), n, H, _ptr(q, _u8p), _ptr(s, _f32p))
    return q, s


# --------------------------------------------------------------------------
# the path
# --------------------------------------------------------------------------

def route_topk(logits: np.ndarray, K: int):
    """Top-K expert ids (descending logit, ties -> lower id) and softmax weights over them."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    assert 1 <= K <= E
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    _load().oracle_route_topk(_ptr(logits, _f32p), T, E, K, _ptr(idx, _i32p), _ptr(w, _f32p))
    return idx, w


def route_topk_grouped(logits: np.ndarray, K: int, n_groups: int, topk_groups: int):
    """Group-limited top-K: best ``topk_groups`` of ``n_groups`` groups by their largest logit,
    then top-K among their experts; weights as in ``route_topk``."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    assert E % n_groups == 0 and 1 <= topk_groups <= n_groups and 1 <= K <= topk_groups * (E // n_groups)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    _load().oracle_route_topk_grouped(_ptr(logits, _f32p), T, E, K, n_groups, topk_groups, _ptr(idx, _i32p),
                                      _ptr(w, _f32p))
    return idx, w


def dispatch(x_bf16: np.ndarray, topk_idx: np.ndarray, B, E: int, fp8: bool = False) -> dict:
    """Count, prefix-sum and scatter tokens into the expert-contiguous receive buffer.

    ``x_bf16`` is uint16 bf16 bits [T, H]; ``topk_idx`` int32 [T, K]; ``B`` the
    per-rank token counts (R of them).  Returns a dict with recv (uint16 [T*K,H]
    or uint8 [T*K,H]), recv_scale (fp32 [T*K,H/128] or None), counts [E*R],
    offsets [E*R+1], expert_offsets [E+1], tok2row [T*K], row2src [T*K].
    """
    x = _c(x_bf16, np.uint16)
    idx = _c(topk_idx, np.int32)
    B = _c(B, np.int32)
    R = B.size
    T, H = x.shape
    K = idx.shape[1] if idx.ndim == 2 else (idx.size // T if T else 0)
    assert int(B.sum()) == T
    rows = T * K
    if fp8:
        assert H % 128 == 0
        recv = np.empty((rows, H), np.uint8)
        recv_scale = np.empty((rows, H // 128), np.float32)
    else:
        recv = np.empty((rows, H), np.uint16)
        recv_scale = None
    counts = np.empty(E * R, np.int32)
    offsets = np.empty(E * R + 1, np.int32)
    expert_offsets = np.empty(E + 1, np.int32)
    tok2row = np.empty(rows, np.int32)
    row2src = np.empty(rows, np.int32)
    rc = _load().oracle_dispatch(
        _ptr(x, _u16p), _ptr(idx.reshape(-1), _i32p), R, _ptr(B, _i32p), E, K, H, int(bool(fp8)),
        recv.ctypes.data_as(_vp), _ptr(recv_scale, _f32p), _ptr(counts, _i32p), _ptr(offsets, _i32p),
        _ptr(expert_offsets, _i32p), _ptr(tok2row, _i32p), _ptr(row2src, _i32p))
    if rc != 0:
        raise ValueError("oracle_dispatch: expert index out of range")
    return dict(recv=recv, recv_scale=recv_scale, counts=counts, offsets=offsets,
                expert_offsets=expert_offsets, tok2row=tok2row, row2src=row2src)


def dispatch_ll(x_bf16: np.ndarray, topk_idx: np.ndarray, B, E: int, C: int, fp8: bool = False) -> dict:
    """Low-latency layout: copy j of token g of rank s goes to row (e*R + s)*C + slot of an
    [E*R*C, H] rectangle.  Rows past counts[e*R+s] in a region stay zero here.  Returns recv,
    recv_scale, counts [E*R], tok2row [T*K], row2src [E*R*C] (-1 where unfilled)."""
    x = _c(x_bf16, np.uint16)
    idx = _c(topk_idx, np.int32)
    B = _c(B, np.int32)
    R = B.size
    T, H = x.shape
    K = idx.shape[1] if idx.ndim == 2 else (idx.size // T if T else 0)
    rows = E * R * C
    if fp8:
        recv = np.zeros((rows, H), np.uint8)
        recv_scale = np.zeros((rows, H // 128), np.float32)
    else:
        recv = np.zeros((rows, H), np.uint16)
        recv_scale = None
    counts = np.empty(E * R, np.int32)
    tok2row = np.empty(T * K, np.int32)
    row2src = np.full(rows, -1, np.int32)
    rc = _load().oracle_dispatch_ll(
        _ptr(x, _u16p), _ptr(idx.reshape(-1), _i32p), R, _ptr(B, _i32p), E, K, H, C, int(bool(fp8)),
        recv.ctypes.data_as(_vp), _ptr(recv_scale, _f32p), _ptr(counts, _i32p), _ptr(tok2row, _i32p),
        _ptr(row2src, _i32p))
    if rc == -1:
        raise ValueError("oracle_dispatch_ll: expert index out of range")
    if rc == -2:
        raise ValueError("oracle_dispatch_ll: a rank holds more tokens than the chunk cap C")
    return dict(recv=recv, recv_scale=recv_scale, counts=counts, tok2row=tok2row, row2src=row2src)


def combine_ll_push(y_bf16: np.ndarray, row2src: np.ndarray, counts: np.ndarray, R: int, E: int, C: int,
                    T: int, K: int) -> np.ndarray:
    """Push each filled rectangle row to its origin slot: ret [T*K, H] (bf16 bits)."""
    y = _c(y_bf16, np.uint16)
    H = y.shape[1]
    ret = np.zeros((T * K, H), np.uint16)
    _load().oracle_combine_ll_push(_ptr(y, _u16p), _ptr(_c(row2src, np.int32), _i32p),
                                   _ptr(_c(counts, np.int32), _i32p), R, E, C, H, _ptr(ret, _u16p))
    return ret


def expert_scale(recv: np.ndarray, recv_scale, expert_offsets: np.ndarray, E: int,
                 identity: bool = False) -> np.ndarray:
    """Expert stand-in: y = bf16(xhat * (1 + e/256)) per row of expert e (or * 1 if identity)."""
    fp8 = recv.dtype == np.uint8
    recv = np.ascontiguousarray(recv)
    rows, H = recv.shape
    eo = _c(expert_offsets, np.int32)
    y = np.empty((rows, H), np.uint16)
    sc = None if recv_scale is None else _c(recv_scale, np.float32)
    _load().oracle_expert_scale(recv.ctypes.data_as(_vp), _ptr(sc, _f32p), int(fp8), _ptr(eo, _i32p),
                                E, H, int(bool(identity)), _ptr(y, _u16p))
    return y


def combine(y_bf16: np.ndarray, tok2row: np.ndarray, topk_w: np.ndarray, out: str = "bf16"):
    """out[g] = sum_j w[g,j] * y[tok2row[g*K+j]] (fp32 fma chain, j ascending).

    ``out`` is "bf16" (uint16 bits), "f32", or "f64" (the same sum in double).
    """
    y = _c(y_bf16, np.uint16)
    t2r = _c(tok2row, np.int32).reshape(-1)
    w = _c(topk_w, np.float32)
    T, K = w.shape
    H = y.shape[1]
    lib = _load()
    if out == "f64":
        o = np.empty((T, H), np.float64)
        lib.oracle_combine_f64(_ptr(y, _u16p), _ptr(t2r, _i32p), _ptr(w, _f32p), T, K, H, _ptr(o, _f64p))
        return o
    if out == "f32":
        o = np.empty((T, H), np.float32)
        lib.oracle_combine(_ptr(y, _u16p), _ptr(t2r, _i32p), _ptr(w, _f32p), T, K, H, None, _ptr(o, _f32p))
        return o
    if out == "bf16":
        o = np.empty((T, H), np.uint16)
        lib.oracle_combine(_ptr(y, _u16p), _ptr(t2r, _i32p), _ptr(w, _f32p), T, K, H, _ptr(o, _u16p), None)
        return o
    raise ValueError(out)


def combine_partial(y_bf16: np.ndarray, tok2row: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray,
                    E: int, R: int, out: str = "bf16", with_partial: bool = False):
    """Sender-side partial accumulation: bf16 partial per (token, expert rank), summed on the origin.

    Returns out (bf16 bits or fp32), and with ``with_partial`` also the [T*K, H] partial rows
    (bf16 bits; only slot g*K + j0 of each (token, rank) is meaningful, the rest stays 0)."""
    y = _c(y_bf16, np.uint16)
    t2r = _c(tok2row, np.int32).reshape(-1)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_w, np.float32)
    T, K = w.shape
    H = y.shape[1]
    part = np.zeros((T * K, H), np.uint16) if with_partial else None
    ob = np.empty((T, H), np.uint16) if out == "bf16" else None
    of = np.empty((T, H), np.float32) if out == "f32" else None
    _load().oracle_combine_partial(_ptr(y, _u16p), _ptr(t2r, _i32p), _ptr(idx.reshape(-1), _i32p), _ptr(w, _f32p),
                                   T, K, H, E, R, _ptr(part, _u16p), _ptr(ob, _u16p), _ptr(of, _f32p))
    o = ob if out == "bf16" else of
    return (o, part) if with_partial else o


def layer(x_bf16, logits, B, E: int, K: int, fp8: bool = False, identity: bool = False,
          out: str = "bf16") -> dict:
    """The whole path on the CPU: route, dispatch, expert stand-in, combine."""
    idx, w = route_topk(logits, K)
    d = dispatch(x_bf16, idx, B, E, fp8=fp8)
    y = expert_scale(d["recv"], d["recv_scale"], d["expert_offsets"], E, identity=identity)
    o = combine(y, d["tok2row"], w, out=out)
    d.update(topk_idx=idx, topk_w=w, y=y, out=o)
    return d
