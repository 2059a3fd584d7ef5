"""Shared helpers for the GPU parity tests: device transfer and the tolerance check.

Tolerance (stated for the attention forward): O within max abs error 1e-2 and mean abs error
1e-3 of the float64 oracle, LSE within 1e-3 absolute.  O is a bf16 output, and a correctly
rounded bf16 value can sit up to half a bf16 spacing from the exact result (0.0156 for |O| in
[4, 8)); the max-abs bound is therefore applied to the kernel's error on top of that unavoidable
output rounding: |O_gpu - O_ref| <= 1e-2 + half_ulp_bf16(O_ref).
"""
import numpy as np
import torch

from io_aware_attention_attn_gb300 import accounting as acc

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_ABS = 1e-3


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def check(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
          what: str = "") -> dict:
    """Element-wise comparison; raises AssertionError with a summary on failure."""
    assert o_gpu.shape == o_ref.shape and lse_gpu.shape == lse_ref.shape, what
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    assert np.isfinite(lse_gpu).all(), f"{what}: non-finite LSE"
    err = np.abs(o_gpu - o_ref)
    tol = O_MAX_ABS + acc.bf16_half_ulp(o_ref)
    bad = err > tol
    lerr = np.abs(lse_gpu - lse_ref)
    stats = {"o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
             "o_over_1e-2": int((err > O_MAX_ABS).sum()), "lse_max_abs": float(lerr.max()),
             "n": int(err.size)}
    assert not bad.any(), f"{what}: {int(bad.sum())} O values over tolerance; {stats}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean abs error {err.mean()}; {stats}"
    assert lerr.max() <= LSE_ABS, f"{what}: LSE error {lerr.max()}; {stats}"
    return stats
