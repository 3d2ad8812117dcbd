"""Run the plain C consumer of the library (tests/c_abi/roundtrip.c) on the GPU: route,
dispatch, identity expert stand-in and combine through the C ABI alone, with its own checks
of the counts, the maps, the dispatched rows and the combined output."""
import subprocess

import pytest
import torch

import _c_abi

pytestmark = pytest.mark.gpu


def test_plain_c_roundtrip(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_moe_route_gb300 import build
    exe = _c_abi.compile_roundtrip(build.build(), str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi roundtrip ok" in r.stdout
