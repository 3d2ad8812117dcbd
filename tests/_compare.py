"""Helpers for the GPU parity tests: move results to numpy, tolerances."""
import numpy as np
import torch


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bytes8(t: torch.Tensor) -> np.ndarray:
    """fp8 / uint8 tensor -> uint8."""
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def weight_tolerance(w_ref: np.ndarray, sel_logits: np.ndarray, K: int) -> np.ndarray:
    """Allowed |w_gpu - w_oracle| for the router weights.

    The GPU computes t_j = l_j - l_0 in fp32 (error <= u|d_j|, u = 2^-24), exp
    in fp32 (CUDA documents at most 2 ulp), a K-term fp32 sum and one IEEE
    division; the oracle evaluates in fp64 and rounds once.  The relative
    difference is below u * (|d_j| + 2K + 10) on every term; the bound used is
    2u * (|d_j| + K + 5), which covers that with margin.
    """
    d = np.abs(sel_logits.astype(np.float64) - sel_logits[:, :1].astype(np.float64))
    return w_ref.astype(np.float64) * 2.0**-23 * (d + K + 5) + 2.0**-140
