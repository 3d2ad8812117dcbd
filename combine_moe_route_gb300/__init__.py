"""MoE expert-parallel route -> dispatch -> combine on one GB300 (sm_103a).

The compute runs in the CUDA library ``libmoeroute.so`` (sources in
``csrc/``, C ABI in ``include/moe_route.h``); ``binding`` is a thin ctypes
layer over it that takes torch tensors.  Importing the package does not load
the library; the first use of an operation does, and raises ``ImportError``
if the library has not been built -- there is no fallback.

``workloads`` draws the seeded synthetic inputs.
"""
from importlib import import_module

_API = {
    "route_topk", "dispatch", "combine", "expert_scale", "dispatch_workspace_bytes",
    "get_device_error", "abi_version", "strerror", "MoeError", "DispatchResult",
    "moe_layer", "library_path", "load_library", "MOE_OK", "dispatch_noalloc",
    "route_topk_grouped", "dispatch_ll", "combine_ll", "combine_ll_push", "DispatchLLResult",
    "combine_partial_send", "combine_partial_recv", "BoundLayer",
}

__all__ = sorted(_API) + ["workloads", "HostLayerPipeline"]


def __getattr__(name):
    if name in _API:
        return getattr(import_module(".binding", __name__), name)
    if name == "workloads":
        return import_module(".workloads", __name__)
    if name == "HostLayerPipeline":
        return import_module(".pipeline", __name__).HostLayerPipeline
    raise AttributeError(name)
