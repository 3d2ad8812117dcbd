"""ctypes binding over libmoeroute's C ABI (include/moe_route.h).

Argument marshalling only: every step of route, dispatch, expert stand-in and
combine runs in the library's CUDA kernels.  torch supplies device memory and
streams.  Functions keep the C names without the ``moe_`` prefix; each checks
shapes, dtypes and devices, allocates outputs that were not passed in (with
torch, on the input's device), and calls the matching C entry point on the
current torch stream (or the one given).  A non-OK status raises ``MoeError``.

There is no CPU fallback: if the library is missing, loading raises
``ImportError``; if the tensors are not on a CUDA device, ``ValueError``.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np
import torch

from . import build as _build

MOE_OK = 0
_DTYPE_BF16, _DTYPE_FP8, _DTYPE_FP32 = 0, 1, 2

_lock = threading.Lock()
_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status})")


def library_path() -> str:
    return _build.library_path()


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libmoeroute.so (raises ImportError if it has not been built).

    ``path`` loads another build of the library (one built with other tuning
    defines, say) and returns it with its signatures declared, without making it
    the one the functions below call."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        default = path is None
        path = path or library_path()
        if not os.path.exists(path):
            raise ImportError(
                f"libmoeroute.so not found at {path}; build it with "
                "`python -m combine_moe_route_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.moe_abi_version.argtypes = []
        lib.moe_abi_version.restype = i32
        lib.moe_strerror.argtypes = [i32]
        lib.moe_strerror.restype = ctypes.c_char_p
        lib.moe_route_topk.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        lib.moe_route_topk.restype = i32
        lib.moe_route_topk_grouped.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp]
        lib.moe_route_topk_grouped.restype = i32
        lib.moe_dispatch_workspace_bytes.argtypes = [i32, i32, i32, i64]
        lib.moe_dispatch_workspace_bytes.restype = sz
        lib.moe_dispatch.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.moe_dispatch.restype = i32
        lib.moe_expert_scale.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp]
        lib.moe_expert_scale.restype = i32
        lib.moe_combine.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
        lib.moe_combine.restype = i32
        lib.moe_dispatch_ll.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.moe_dispatch_ll.restype = i32
        lib.moe_dispatch_ll_unordered.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                                  sz, vp]
        lib.moe_dispatch_ll_unordered.restype = i32
        lib.moe_combine_ll.argtypes = [vp, i32, i32, i32, vp, vp, i32, i32, i32, i32, vp, vp]
        lib.moe_combine_ll.restype = i32
        lib.moe_combine_ll_push.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.moe_combine_ll_push.restype = i32
        lib.moe_combine_partial_send.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
        lib.moe_combine_partial_send.restype = i32
        lib.moe_combine_partial_recv.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.moe_combine_partial_recv.restype = i32
        lib.moe_dispatch_send.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, sz, vp]
        lib.moe_dispatch_send.restype = i32
        lib.moe_dispatch_recv.argtypes = [i32, vp, i32, i32, vp, vp, vp, vp, sz, vp]
        lib.moe_dispatch_recv.restype = i32
        lib.moe_combine_send.argtypes = [i32, vp, sz, vp]
        lib.moe_combine_send.restype = i32
        lib.moe_combine_recv.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, i32, vp, sz, vp]
        lib.moe_combine_recv.restype = i32
        lib.moe_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
        lib.moe_get_device_error.restype = i32
        lib.moe_dispatch_noalloc.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.moe_dispatch_noalloc.restype = i32
        for reader in ("moe_trace_dispatch", "moe_trace_combine"):   # builds with -DMOE_TRACE only
            try:
                fn = getattr(lib, reader)
            except AttributeError:
                continue
            fn.argtypes = [i32, vp]
            fn.restype = i32
        if default:
            _lib = lib
        return lib


@contextlib.contextmanager
def using_library(lib: ctypes.CDLL):
    """Route the functions below through ``lib`` (another build, from ``load_library(path)``)
    inside the ``with`` block; the previous library is restored afterwards."""
    global _lib
    with _lock:
        prev = _lib
        _lib = lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = prev


def abi_version() -> int:
    return load_library().moe_abi_version()


def strerror(status: int) -> str:
    return load_library().moe_strerror(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, what)


def _stream_handle(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> torch.Tensor:
    # on every call's path: attribute checks only (no device objects or tuple copies)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); there is no CPU path")
    if dtype is not None:
        if (t.dtype not in dtype) if type(dtype) is tuple else (t.dtype is not dtype):
            raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and t.shape != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else int(t.data_ptr())


# ---------------------------------------------------------------------------
# route
# ---------------------------------------------------------------------------

def route_topk(logits: torch.Tensor, K: int, *, topk_idx: torch.Tensor | None = None,
               topk_w: torch.Tensor | None = None, stream=None):
    """Top-K experts per token and their softmax weights: (int32 [T,K], fp32 [T,K])."""
    _dev(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    dev = logits.device
    if topk_idx is None:
        topk_idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, K), dtype=torch.float32, device=dev)
    _dev(topk_idx, "topk_idx", torch.int32, (T, K))
    _dev(topk_w, "topk_w", torch.float32, (T, K))
    with torch.cuda.device(dev):
        _check(load_library().moe_route_topk(_ptr(logits), T, E, K, _ptr(topk_idx), _ptr(topk_w),
                                             _stream_handle(stream, dev)), "moe_route_topk")
    return topk_idx, topk_w


def route_topk_grouped(logits: torch.Tensor, K: int, n_groups: int, topk_groups: int, *,
                       topk_idx: torch.Tensor | None = None, topk_w: torch.Tensor | None = None, stream=None):
    """Group-limited top-K: keep the ``topk_groups`` best of ``n_groups`` contiguous expert
    groups (by their largest logit), then top-K among their experts."""
    _dev(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    dev = logits.device
    if topk_idx is None:
        topk_idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, K), dtype=torch.float32, device=dev)
    _dev(topk_idx, "topk_idx", torch.int32, (T, K))
    _dev(topk_w, "topk_w", torch.float32, (T, K))
    with torch.cuda.device(dev):
        _check(load_library().moe_route_topk_grouped(_ptr(logits), T, E, K, n_groups, topk_groups, _ptr(topk_idx),
                                                     _ptr(topk_w), _stream_handle(stream, dev)),
               "moe_route_topk_grouped")
    return topk_idx, topk_w


# ---------------------------------------------------------------------------
# dispatch
# ---------------------------------------------------------------------------

def dispatch_workspace_bytes(R: int, E: int, K: int, T: int) -> int:
    return int(load_library().moe_dispatch_workspace_bytes(R, E, K, T))


@dataclass
class DispatchResult:
    recv_x: torch.Tensor            # [T*K, H] bf16 or float8_e4m3fn
    recv_scale: torch.Tensor | None  # [T*K, H/128] fp32 (FP8 only)
    counts: torch.Tensor            # [E*R] int32, e-major
    offsets: torch.Tensor           # [E*R+1] int32
    expert_offsets: torch.Tensor    # [E+1] int32
    tok2row: torch.Tensor           # [T*K] int32
    row2src: torch.Tensor           # [T*K] int32
    workspace: torch.Tensor         # uint8, holds the device error word


def _host_B(B) -> np.ndarray:
    if isinstance(B, torch.Tensor):
        if B.device.type != "cpu":
            raise ValueError("B (tokens per rank) is read on the host: pass a CPU tensor, list or array")
        B = B.numpy()
    return np.ascontiguousarray(np.asarray(B, dtype=np.int32))


def dispatch(x: torch.Tensor, topk_idx: torch.Tensor, B, E: int, *, fp8: bool = False,
             out: DispatchResult | None = None, workspace: torch.Tensor | None = None,
             stream=None) -> DispatchResult:
    """Count, scan and scatter x [T,H] bf16 into expert-contiguous rows (optionally FP8)."""
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be [T, H]")
    T, H = x.shape
    _dev(topk_idx, "topk_idx", torch.int32)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, K]")
    K = topk_idx.shape[1]
    Bh = _host_B(B)
    R = Bh.size
    if int(Bh.astype(np.int64).sum()) != T:
        raise ValueError(f"sum(B) = {int(Bh.sum())} does not match x.shape[0] = {T}")
    dev = x.device
    rows = T * K
    if out is None:
        recv_x = torch.empty((rows, H), dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16, device=dev)
        recv_scale = torch.empty((rows, H // 128), dtype=torch.float32, device=dev) if fp8 else None
        out = DispatchResult(
            recv_x=recv_x, recv_scale=recv_scale,
            counts=torch.empty(E * R, dtype=torch.int32, device=dev),
            offsets=torch.empty(E * R + 1, dtype=torch.int32, device=dev),
            expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            tok2row=torch.empty(rows, dtype=torch.int32, device=dev),
            row2src=torch.empty(rows, dtype=torch.int32, device=dev),
            workspace=None)
    need = dispatch_workspace_bytes(R, E, K, T)
    if workspace is None:
        workspace = out.workspace
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    out.workspace = workspace
    _dev(out.recv_x, "recv_x", (torch.float8_e4m3fn, torch.uint8) if fp8 else torch.bfloat16, (rows, H))
    if fp8:
        _dev(out.recv_scale, "recv_scale", torch.float32, (rows, H // 128))
    for name, n in (("counts", E * R), ("offsets", E * R + 1), ("expert_offsets", E + 1),
                    ("tok2row", rows), ("row2src", rows)):
        _dev(getattr(out, name), name, torch.int32, (n,))
    _dev(workspace, "workspace", torch.uint8)
    with torch.cuda.device(dev):
        _check(load_library().moe_dispatch(
            _ptr(x), _ptr(topk_idx), R, Bh.ctypes.data, E, K, H, _DTYPE_FP8 if fp8 else _DTYPE_BF16,
            _ptr(out.recv_x), _ptr(out.recv_scale) if fp8 else None, _ptr(out.counts), _ptr(out.offsets),
            _ptr(out.expert_offsets), _ptr(out.tok2row), _ptr(out.row2src), _ptr(workspace),
            workspace.numel(), _stream_handle(stream, dev)), "moe_dispatch")
    return out


def get_device_error(workspace: torch.Tensor, stream=None) -> tuple[int, int]:
    """Synchronise the stream and read the dispatch error word: (status, raw bits)."""
    _dev(workspace, "workspace", torch.uint8)
    code = ctypes.c_int32(0)
    with torch.cuda.device(workspace.device):
        st = load_library().moe_get_device_error(_ptr(workspace), ctypes.byref(code),
                                                 _stream_handle(stream, workspace.device))
    return int(st), int(code.value)


# ---------------------------------------------------------------------------
# expert stand-in and combine
# ---------------------------------------------------------------------------

def expert_scale(recv_x: torch.Tensor, recv_scale: torch.Tensor | None, expert_offsets: torch.Tensor,
                 E: int, *, identity: bool = False, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = bf16(xhat * (1 + e/256)) per row of expert e (the grouped-GEMM stand-in)."""
    fp8 = recv_x.dtype in (torch.float8_e4m3fn, torch.uint8)
    _dev(recv_x, "recv_x")
    rows, H = recv_x.shape
    _dev(expert_offsets, "expert_offsets", torch.int32, (E + 1,))
    if fp8:
        _dev(recv_scale, "recv_scale", torch.float32, (rows, H // 128))
    if out is None:
        out = torch.empty((rows, H), dtype=torch.bfloat16, device=recv_x.device)
    _dev(out, "y", torch.bfloat16, (rows, H))
    with torch.cuda.device(recv_x.device):
        _check(load_library().moe_expert_scale(
            _ptr(recv_x), _ptr(recv_scale) if fp8 else None, _DTYPE_FP8 if fp8 else _DTYPE_BF16,
            _ptr(expert_offsets), E, H, rows, int(bool(identity)), _ptr(out),
            _stream_handle(stream, recv_x.device)), "moe_expert_scale")
    return out


def combine(y: torch.Tensor, tok2row: torch.Tensor, topk_w: torch.Tensor, *,
            out_dtype: torch.dtype = torch.bfloat16, out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """out[g] = sum_j topk_w[g,j] * y[tok2row[g*K+j]] (fp32 fma, j ascending) -> [T, H]."""
    _dev(y, "y", torch.bfloat16)
    _dev(topk_w, "topk_w", torch.float32)
    if topk_w.dim() != 2:
        raise ValueError("topk_w must be [T, K]")
    T, K = topk_w.shape
    H = y.shape[1]
    if tok2row is not None:       # None: the identity map (rows g*K + j)
        _dev(tok2row, "tok2row", torch.int32)
        if tok2row.numel() != T * K:
            raise ValueError("tok2row must have T*K entries")
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be bfloat16 or float32")
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=y.device)
    _dev(out, "out", out_dtype, (T, H))
    with torch.cuda.device(y.device):
        _check(load_library().moe_combine(
            _ptr(y), _ptr(tok2row), _ptr(topk_w), T, K, H,
            _DTYPE_FP32 if out_dtype == torch.float32 else _DTYPE_BF16, _ptr(out),
            _stream_handle(stream, y.device)), "moe_combine")
    return out


# ---------------------------------------------------------------------------
# low-latency (fixed-rectangle) layout
# ---------------------------------------------------------------------------

@dataclass
class DispatchLLResult:
    recv_x: torch.Tensor             # [E*R*C, H] bf16 or float8_e4m3fn
    recv_scale: torch.Tensor | None  # [E*R*C, H/128] fp32 (FP8 only)
    counts: torch.Tensor             # [E*R] int32: filled rows per (expert, source rank) region
    tok2row: torch.Tensor            # [T*K] int32
    row2src: torch.Tensor            # [E*R*C] int32 (meaningful on filled rows only)
    workspace: torch.Tensor
    C: int


def dispatch_ll(x: torch.Tensor, topk_idx: torch.Tensor, B, E: int, C: int, *, fp8: bool = False,
                unordered: bool = False, out: DispatchLLResult | None = None, stream=None) -> DispatchLLResult:
    """Low-latency dispatch into a fixed [E*R*C, H] rectangle (C rows per (expert, rank) region).

    unordered=True: each copy takes its slot in its region by an atomic increment
    (moe_dispatch_ll_unordered): no histogram pass, and the order of the rows inside
    a region is unspecified."""
    _dev(x, "x", torch.bfloat16)
    T, H = x.shape
    _dev(topk_idx, "topk_idx", torch.int32)
    K = topk_idx.shape[1]
    Bh = _host_B(B)
    R = Bh.size
    if int(Bh.astype(np.int64).sum()) != T:
        raise ValueError(f"sum(B) = {int(Bh.sum())} does not match x.shape[0] = {T}")
    dev = x.device
    rows = E * R * C
    if out is None:
        out = DispatchLLResult(
            recv_x=torch.empty((rows, H), dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16, device=dev),
            recv_scale=torch.empty((rows, H // 128), dtype=torch.float32, device=dev) if fp8 else None,
            counts=torch.empty(E * R, dtype=torch.int32, device=dev),
            tok2row=torch.empty(T * K, dtype=torch.int32, device=dev),
            row2src=torch.empty(rows, dtype=torch.int32, device=dev),
            workspace=torch.empty(max(dispatch_workspace_bytes(R, E, K, T), 256), dtype=torch.uint8, device=dev),
            C=C)
    lib = load_library()
    fn, name = ((lib.moe_dispatch_ll_unordered, "moe_dispatch_ll_unordered") if unordered
                else (lib.moe_dispatch_ll, "moe_dispatch_ll"))
    with torch.cuda.device(dev):
        _check(fn(
            _ptr(x), _ptr(topk_idx), R, Bh.ctypes.data, E, K, H, C, _DTYPE_FP8 if fp8 else _DTYPE_BF16,
            _ptr(out.recv_x), _ptr(out.recv_scale) if fp8 else None, _ptr(out.counts), _ptr(out.tok2row),
            _ptr(out.row2src), _ptr(out.workspace), out.workspace.numel(), _stream_handle(stream, dev)), name)
    return out


def combine_ll(y: torch.Tensor, E: int, R: int, C: int, tok2row: torch.Tensor, topk_w: torch.Tensor, *,
               out_dtype: torch.dtype = torch.bfloat16, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Weighted sum gathered from the low-latency rectangle y [E*R*C, H]."""
    _dev(y, "y", torch.bfloat16)
    _dev(tok2row, "tok2row", torch.int32)
    _dev(topk_w, "topk_w", torch.float32)
    T, K = topk_w.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=y.device)
    _dev(out, "out", out_dtype, (T, H))
    with torch.cuda.device(y.device):
        _check(load_library().moe_combine_ll(
            _ptr(y), E, R, C, _ptr(tok2row), _ptr(topk_w), T, K, H,
            _DTYPE_FP32 if out_dtype == torch.float32 else _DTYPE_BF16, _ptr(out), _stream_handle(stream, y.device)),
            "moe_combine_ll")
    return out


def combine_ll_push(y: torch.Tensor, d: DispatchLLResult, R: int, E: int, T: int, K: int, *,
                    out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Push each filled rectangle row to its origin slot g*K + j: ret [T*K, H] bf16."""
    _dev(y, "y", torch.bfloat16)
    H = y.shape[1]
    if out is None:
        out = torch.empty((T * K, H), dtype=torch.bfloat16, device=y.device)
    _dev(out, "ret", torch.bfloat16, (T * K, H))
    with torch.cuda.device(y.device):
        _check(load_library().moe_combine_ll_push(
            _ptr(y), _ptr(d.row2src), _ptr(d.counts), R, E, d.C, K, H, T, _ptr(out),
            _stream_handle(stream, y.device)), "moe_combine_ll_push")
    return out


# ---------------------------------------------------------------------------
# sender-side partial accumulation
# ---------------------------------------------------------------------------

def combine_partial_send(y: torch.Tensor, tok2row: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                         E: int, R: int, *, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One bf16 partial per (token, expert rank) in slot g*K + (first copy on that rank): [T*K, H]."""
    _dev(y, "y", torch.bfloat16)
    _dev(tok2row, "tok2row", torch.int32)
    _dev(topk_idx, "topk_idx", torch.int32)
    _dev(topk_w, "topk_w", torch.float32)
    T, K = topk_w.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty((T * K, H), dtype=torch.bfloat16, device=y.device)
    _dev(out, "partial", torch.bfloat16, (T * K, H))
    with torch.cuda.device(y.device):
        _check(load_library().moe_combine_partial_send(
            _ptr(y), _ptr(tok2row), _ptr(topk_idx), _ptr(topk_w), T, K, H, E, R, _ptr(out),
            _stream_handle(stream, y.device)), "moe_combine_partial_send")
    return out


def combine_partial_recv(partial: torch.Tensor, topk_idx: torch.Tensor, E: int, R: int, *,
                         out_dtype: torch.dtype = torch.bfloat16, out: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Sum of each token's partials in ascending rank order (fp32) -> [T, H]."""
    _dev(partial, "partial", torch.bfloat16)
    _dev(topk_idx, "topk_idx", torch.int32)
    T, K = topk_idx.shape
    H = partial.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=partial.device)
    _dev(out, "out", out_dtype, (T, H))
    with torch.cuda.device(partial.device):
        _check(load_library().moe_combine_partial_recv(
            _ptr(partial), _ptr(topk_idx), T, K, H, E, R, _DTYPE_FP32 if out_dtype == torch.float32 else _DTYPE_BF16,
            _ptr(out), _stream_handle(stream, partial.device)), "moe_combine_partial_recv")
    return out


def moe_layer(x: torch.Tensor, logits: torch.Tensor, B, E: int, K: int, *, fp8: bool = False,
              identity: bool = False, out_dtype: torch.dtype = torch.bfloat16, stream=None) -> dict:
    """One layer on the GPU: route, dispatch, expert stand-in, combine (all enqueued, no sync)."""
    idx, w = route_topk(logits, K, stream=stream)
    d = dispatch(x, idx, B, E, fp8=fp8, stream=stream)
    y = expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E, identity=identity, stream=stream)
    o = combine(y, d.tok2row, w, out_dtype=out_dtype, stream=stream)
    return dict(topk_idx=idx, topk_w=w, dispatch=d, y=y, out=o)


class BoundLayer:
    """One layer's four calls (route, dispatch, expert stand-in, combine) with every tensor
    checked and every argument marshalled once, for loops that run the same shapes again and
    again (a decode step run eagerly).  A call then costs one ctypes call per step, with none
    of the per-call checks.

    The layer reads ``x`` [T, H] bf16 and ``logits`` [T, E] fp32 in place and writes into
    buffers it owns (``topk_idx``, ``topk_w``, ``dispatch``, ``y``, ``out``).  Refill the
    inputs in place between calls; do not resize or replace them.  Calls are enqueued on the
    stream given (default: the current stream at bind time) and on the inputs' device."""

    def __init__(self, x: torch.Tensor, logits: torch.Tensor, B, E: int, K: int, *, fp8: bool = False,
                 identity: bool = False, out_dtype: torch.dtype = torch.bfloat16, stream=None):
        dev = x.device
        self.x, self.logits = x, logits
        # the regular entry points check every tensor once and allocate the outputs
        self.topk_idx, self.topk_w = route_topk(logits, K, stream=stream)
        self.dispatch = dispatch(x, self.topk_idx, B, E, fp8=fp8, stream=stream)
        d = self.dispatch
        self.y = expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, E, identity=identity, stream=stream)
        self.out = combine(self.y, d.tok2row, self.topk_w, out_dtype=out_dtype, stream=stream)
        self._B = _host_B(B)                          # kept alive: the dispatch reads it on each call
        self._device = dev.index if dev.index is not None else torch.cuda.current_device()
        T, H = x.shape
        R = self._B.size
        st = _stream_handle(stream, dev)
        lib = load_library()
        self._calls = (
            (lib.moe_route_topk, (_ptr(logits), T, E, K, _ptr(self.topk_idx), _ptr(self.topk_w), st),
             "moe_route_topk"),
            (lib.moe_dispatch, (_ptr(x), _ptr(self.topk_idx), R, self._B.ctypes.data, E, K, H,
                                _DTYPE_FP8 if fp8 else _DTYPE_BF16, _ptr(d.recv_x),
                                _ptr(d.recv_scale) if fp8 else None, _ptr(d.counts), _ptr(d.offsets),
                                _ptr(d.expert_offsets), _ptr(d.tok2row), _ptr(d.row2src), _ptr(d.workspace),
                                d.workspace.numel(), st), "moe_dispatch"),
            (lib.moe_expert_scale, (_ptr(d.recv_x), _ptr(d.recv_scale) if fp8 else None,
                                    _DTYPE_FP8 if fp8 else _DTYPE_BF16, _ptr(d.expert_offsets), E, H, T * K,
                                    int(bool(identity)), _ptr(self.y), st), "moe_expert_scale"),
            (lib.moe_combine, (_ptr(self.y), _ptr(d.tok2row), _ptr(self.topk_w), T, K, H,
                               _DTYPE_FP32 if out_dtype == torch.float32 else _DTYPE_BF16, _ptr(self.out), st),
             "moe_combine"),
        )

    def _run(self, i: int) -> None:
        fn, args, name = self._calls[i]
        if torch.cuda.current_device() == self._device:
            _check(fn(*args), name)
        else:
            with torch.cuda.device(self._device):
                _check(fn(*args), name)

    def route(self) -> None:
        self._run(0)

    def dispatch_call(self) -> None:
        self._run(1)

    def expert(self) -> None:
        self._run(2)

    def combine_call(self) -> None:
        self._run(3)

    def __call__(self) -> torch.Tensor:
        """Enqueue the whole layer; returns ``out`` (valid once the stream reaches it)."""
        for i in range(4):
            self._run(i)
        return self.out


# ---------------------------------------------------------------------------
# split dispatch and combine (send and receive halves)
# ---------------------------------------------------------------------------

def _dispatch_buffers(T: int, H: int, E: int, R: int, K: int, fp8: bool, dev) -> DispatchResult:
    rows = T * K
    return DispatchResult(
        recv_x=torch.empty((rows, H), dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16, device=dev),
        recv_scale=torch.empty((rows, H // 128), dtype=torch.float32, device=dev) if fp8 else None,
        counts=torch.empty(E * R, dtype=torch.int32, device=dev),
        offsets=torch.empty(E * R + 1, dtype=torch.int32, device=dev),
        expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
        tok2row=torch.empty(rows, dtype=torch.int32, device=dev),
        row2src=torch.empty(rows, dtype=torch.int32, device=dev),
        workspace=torch.empty(max(dispatch_workspace_bytes(R, E, K, T), 256), dtype=torch.uint8, device=dev))


def dispatch_send(x: torch.Tensor, topk_idx: torch.Tensor, B, E: int, *, fp8: bool = False, max_sms: int = 0,
                  out: DispatchResult | None = None, stream=None) -> DispatchResult:
    """Send half of the split dispatch: the rows, tok2row and row2src of ``dispatch``, each copy
    announced to its destination rank.  ``counts``, ``offsets`` and ``expert_offsets`` of the
    result are written by ``dispatch_recv``.  ``max_sms`` > 0 keeps the copy kernel on at most
    that many SMs."""
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be [T, H]")
    T, H = x.shape
    _dev(topk_idx, "topk_idx", torch.int32)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, K]")
    K = topk_idx.shape[1]
    Bh = _host_B(B)
    R = Bh.size
    if int(Bh.astype(np.int64).sum()) != T:
        raise ValueError(f"sum(B) = {int(Bh.sum())} does not match x.shape[0] = {T}")
    dev = x.device
    rows = T * K
    if out is None:
        out = _dispatch_buffers(T, H, E, R, K, fp8, dev)
    _dev(out.recv_x, "recv_x", (torch.float8_e4m3fn, torch.uint8) if fp8 else torch.bfloat16, (rows, H))
    if fp8:
        _dev(out.recv_scale, "recv_scale", torch.float32, (rows, H // 128))
    for name in ("tok2row", "row2src"):
        _dev(getattr(out, name), name, torch.int32, (rows,))
    _dev(out.workspace, "workspace", torch.uint8)
    with torch.cuda.device(dev):
        _check(load_library().moe_dispatch_send(
            _ptr(x), _ptr(topk_idx), R, Bh.ctypes.data, E, K, H, _DTYPE_FP8 if fp8 else _DTYPE_BF16,
            _ptr(out.recv_x), _ptr(out.recv_scale) if fp8 else None, _ptr(out.tok2row), _ptr(out.row2src),
            int(max_sms), _ptr(out.workspace), out.workspace.numel(), _stream_handle(stream, dev)),
            "moe_dispatch_send")
    return out


def dispatch_recv(d: DispatchResult, B, E: int, K: int, *, stream=None) -> DispatchResult:
    """Receive half of the split dispatch: waits until the send half's copies have landed and
    writes ``d.counts``, ``d.offsets`` and ``d.expert_offsets``."""
    Bh = _host_B(B)
    R = Bh.size
    for name, n in (("counts", E * R), ("offsets", E * R + 1), ("expert_offsets", E + 1)):
        _dev(getattr(d, name), name, torch.int32, (n,))
    _dev(d.workspace, "workspace", torch.uint8)
    dev = d.workspace.device
    with torch.cuda.device(dev):
        _check(load_library().moe_dispatch_recv(
            R, Bh.ctypes.data, E, K, _ptr(d.counts), _ptr(d.offsets), _ptr(d.expert_offsets), _ptr(d.workspace),
            d.workspace.numel(), _stream_handle(stream, dev)), "moe_dispatch_recv")
    return d


def combine_send(workspace: torch.Tensor, R: int, *, stream=None) -> None:
    """Send half of the split combine: the expert ranks publish their outputs (enqueue it after
    the work that wrote them)."""
    _dev(workspace, "workspace", torch.uint8)
    with torch.cuda.device(workspace.device):
        _check(load_library().moe_combine_send(R, _ptr(workspace), workspace.numel(),
                                               _stream_handle(stream, workspace.device)), "moe_combine_send")


def combine_recv(y: torch.Tensor, tok2row: torch.Tensor, topk_w: torch.Tensor, workspace: torch.Tensor, R: int, *,
                 out_dtype: torch.dtype = torch.bfloat16, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Receive half of the split combine: waits for every expert rank's outputs, then the
    weighted sum of ``combine`` -> [T, H]."""
    _dev(y, "y", torch.bfloat16)
    _dev(topk_w, "topk_w", torch.float32)
    _dev(tok2row, "tok2row", torch.int32)
    _dev(workspace, "workspace", torch.uint8)
    if topk_w.dim() != 2:
        raise ValueError("topk_w must be [T, K]")
    T, K = topk_w.shape
    H = y.shape[1]
    if tok2row.numel() != T * K:
        raise ValueError("tok2row must have T*K entries")
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be bfloat16 or float32")
    if out is None:
        out = torch.empty((T, H), dtype=out_dtype, device=y.device)
    _dev(out, "out", out_dtype, (T, H))
    with torch.cuda.device(y.device):
        _check(load_library().moe_combine_recv(
            _ptr(y), _ptr(tok2row), _ptr(topk_w), T, K, H,
            _DTYPE_FP32 if out_dtype == torch.float32 else _DTYPE_BF16, _ptr(out), R, _ptr(workspace),
            workspace.numel(), _stream_handle(stream, y.device)), "moe_combine_recv")
    return out


# ---------------------------------------------------------------------------
# dispatch without a caller-supplied workspace
# ---------------------------------------------------------------------------

def dispatch_noalloc(x: torch.Tensor, topk_idx: torch.Tensor, B, E: int, *, fp8: bool = False,
                     out: DispatchResult, stream=None) -> DispatchResult:
    """moe_dispatch_noalloc: like ``dispatch`` but with the library's static
    device scratch as workspace, for callers that cannot allocate device memory.
    Every output buffer must be passed in ``out`` (its ``workspace`` is ignored);
    nothing is allocated here.  The first call on a device must come before any
    stream capture; calls that overlap on the GPU race on the shared scratch."""
    fn = load_library().moe_dispatch_noalloc
    _dev(x, "x", torch.bfloat16)
    T, H = x.shape
    _dev(topk_idx, "topk_idx", torch.int32)
    K = topk_idx.shape[1]
    Bh = _host_B(B)
    R = Bh.size
    if int(Bh.astype(np.int64).sum()) != T:
        raise ValueError(f"sum(B) = {int(Bh.sum())} does not match x.shape[0] = {T}")
    rows = T * K
    _dev(out.recv_x, "recv_x", (torch.float8_e4m3fn, torch.uint8) if fp8 else torch.bfloat16, (rows, H))
    if fp8:
        _dev(out.recv_scale, "recv_scale", torch.float32, (rows, H // 128))
    for name, n in (("counts", E * R), ("offsets", E * R + 1), ("expert_offsets", E + 1),
                    ("tok2row", rows), ("row2src", rows)):
        _dev(getattr(out, name), name, torch.int32, (n,))
    with torch.cuda.device(x.device):
        _check(fn(_ptr(x), _ptr(topk_idx), R, Bh.ctypes.data, E, K, H, _DTYPE_FP8 if fp8 else _DTYPE_BF16,
                  _ptr(out.recv_x), _ptr(out.recv_scale) if fp8 else None, _ptr(out.counts), _ptr(out.offsets),
                  _ptr(out.expert_offsets), _ptr(out.tok2row), _ptr(out.row2src),
                  _stream_handle(stream, x.device)), "moe_dispatch_noalloc")
    return out
