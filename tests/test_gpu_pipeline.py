"""HostLayerPipeline: layers from pinned host memory with copies overlapped
across layers give, layer by layer, exactly the outputs of the plain
device-resident calls."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_pipelined_host_layers_equal_plain_layers():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    build.build()
    from combine_moe_route_gb300 import HostLayerPipeline
    from combine_moe_route_gb300 import binding as b
    from combine_moe_route_gb300 import workloads as wl
    dev = torch.device("cuda:0")
    B, E, K, H = [40, 0, 17, 63, 5, 128, 9, 30], 64, 8, 1024
    layers = [wl.random_shape_inputs(8, E, K, H, B, seed=s, fp8=True) for s in range(5)]
    pipe = HostLayerPipeline(B, E, K, H, fp8=True, device=dev, depth=2)
    hosts = [(l["x"].pin_memory(), torch.from_numpy(l["logits"]).pin_memory(),
              torch.empty((l["T"], H), dtype=torch.bfloat16).pin_memory()) for l in layers]
    for x_h, lg_h, out_h in hosts:
        pipe.submit(x_h, lg_h, out_h)
    pipe.synchronize()
    for (x_h, lg_h, out_h), l in zip(hosts, layers):
        r = b.moe_layer(l["x"].to(dev), torch.from_numpy(l["logits"]).to(dev), B, E, K, fp8=True)
        torch.cuda.synchronize()
        assert torch.equal(out_h, r["out"].cpu())
