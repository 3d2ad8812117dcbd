"""Layers whose inputs and outputs live in (pinned) host memory, with the
copies of one layer overlapped with the compute of its neighbours.

Every layer still makes the full trip: its tokens and router logits go host ->
device, the route, dispatch, expert stand-in and combine run through the C
ABI, and its output goes device -> host.  ``HostLayerPipeline`` keeps
``depth`` sets of device buffers and three streams (host->device, compute,
device->host) ordered by events, so the input copy of layer i+1 and the output
copy of layer i-1 run while layer i computes -- the overlap of transfers and
compute that the sources build their schedules around (Perplexity, "Lower
latency and higher throughput with multi-node DeepSeek deployment",
"Computation and communication overlap").  Nothing here computes: it only
orders copies and calls.
"""
from __future__ import annotations

import torch

from . import binding as b


class HostLayerPipeline:
    """Overlapped host-in / host-out layers of one fixed shape (T tokens over R ranks)."""

    def __init__(self, B, E: int, K: int, H: int, *, fp8: bool = False, identity: bool = False,
                 out_dtype: torch.dtype = torch.bfloat16, device=None, depth: int = 2):
        self.B = list(int(v) for v in B)
        self.T = sum(self.B)
        self.E, self.K, self.H = E, K, H
        self.fp8, self.identity, self.out_dtype = fp8, identity, out_dtype
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.depth = depth
        T, dev = self.T, self.device
        self.h2d = torch.cuda.Stream(dev)
        self.compute = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.slots = []
        for _ in range(depth):
            slot = dict(
                x=torch.empty((T, H), dtype=torch.bfloat16, device=dev),
                logits=torch.empty((T, E), dtype=torch.float32, device=dev),
                idx=torch.empty((T, K), dtype=torch.int32, device=dev),
                w=torch.empty((T, K), dtype=torch.float32, device=dev),
                out=torch.empty((T, H), dtype=out_dtype, device=dev),
                loaded=torch.cuda.Event(), computed=torch.cuda.Event(), stored=torch.cuda.Event(),
                used=False)
            R, rows = len(self.B), T * K
            slot["dispatch"] = b.DispatchResult(
                recv_x=torch.empty((rows, H), dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16, device=dev),
                recv_scale=torch.empty((rows, H // 128), dtype=torch.float32, device=dev) if fp8 else None,
                counts=torch.empty(E * R, dtype=torch.int32, device=dev),
                offsets=torch.empty(E * R + 1, dtype=torch.int32, device=dev),
                expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                tok2row=torch.empty(rows, dtype=torch.int32, device=dev),
                row2src=torch.empty(rows, dtype=torch.int32, device=dev),
                workspace=torch.empty(max(b.dispatch_workspace_bytes(R, E, K, T), 256), dtype=torch.uint8,
                                      device=dev))
            slot["y"] = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
            self.slots.append(slot)
        torch.cuda.synchronize(dev)
        self._next = 0

    def submit(self, x_host: torch.Tensor, logits_host: torch.Tensor, out_host: torch.Tensor) -> None:
        """Enqueue one layer.  ``x_host`` [T, H] bf16 and ``logits_host`` [T, E] fp32 must stay
        unchanged, and ``out_host`` [T, H] unread, until the layer has finished
        (``synchronize``).  Host tensors should be pinned for the copies to be asynchronous."""
        s = self.slots[self._next]
        self._next = (self._next + 1) % self.depth
        if s["used"]:
            self.h2d.wait_event(s["computed"])      # the slot's inputs have been consumed
            self.compute.wait_event(s["stored"])    # the slot's output has been read back
        s["used"] = True
        with torch.cuda.stream(self.h2d):
            s["x"].copy_(x_host, non_blocking=True)
            s["logits"].copy_(logits_host, non_blocking=True)
            s["loaded"].record(self.h2d)
        self.compute.wait_event(s["loaded"])
        with torch.cuda.stream(self.compute):
            b.route_topk(s["logits"], self.K, topk_idx=s["idx"], topk_w=s["w"])
            d = b.dispatch(s["x"], s["idx"], self.B, self.E, fp8=self.fp8, out=s["dispatch"])
            b.expert_scale(d.recv_x, d.recv_scale, d.expert_offsets, self.E, identity=self.identity, out=s["y"])
            b.combine(s["y"], d.tok2row, s["w"], out_dtype=self.out_dtype, out=s["out"])
            s["computed"].record(self.compute)
        self.d2h.wait_event(s["computed"])
        with torch.cuda.stream(self.d2h):
            out_host.copy_(s["out"], non_blocking=True)
            s["stored"].record(self.d2h)

    def synchronize(self) -> None:
        for st in (self.h2d, self.compute, self.d2h):
            st.synchronize()
