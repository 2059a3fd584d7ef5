"""FLOP, byte and roofline accounting for the attention forward and its unfused comparison.

Pure host arithmetic used by the bench and the tests.  The formulas follow the pages' own
accounting: a matmul of an [m x k] by a [k x n] matrix costs 2mkn FLOPs (one multiply and one
add per term), bytes are what must cross HBM at least once, arithmetic intensity is FLOPs per
byte and the roofline is ``min(peak, bandwidth * AI)`` (CS336 Lecture 5 notes, sections 2.1
and 2.2; "GPU Lesson 09", the matrix-multiplication worked example).
"""
from __future__ import annotations

import math

BF16 = 2
FP32 = 4


def matmul_flops(m: int, n: int, k: int) -> int:
    """FLOPs of C[m,n] = A[m,k] B[k,n]: 2 per multiply-add."""
    return 2 * m * n * k


def matmul_bytes(m: int, n: int, k: int, elem: int) -> int:
    """Read A and B once, write C once."""
    return elem * (m * k + k * n + m * n)


def ridge_point(peak_flops: float, bandwidth_bytes: float) -> float:
    """Arithmetic intensity where the bandwidth slope meets the compute roof."""
    return peak_flops / bandwidth_bytes


def roofline(peak_flops: float, bandwidth_bytes: float, ai: float) -> float:
    """Attainable FLOP/s at arithmetic intensity ``ai``."""
    return min(peak_flops, bandwidth_bytes * ai)


def visible_pairs(L: int, causal: bool) -> int:
    """Number of (query, key) pairs a length-L sequence scores (causal keeps j <= i)."""
    return L * (L + 1) // 2 if causal else L * L


def attention_flops(heads: int, lengths, d: int, causal: bool) -> float:
    """Headline FLOP count: two L x L x d matmuls per head (QK^T and PV), 4 L^2 d, halved
    for causal masking.  ``lengths``: per-sequence lengths (dense: B copies of N)."""
    total = 0.0
    for L in lengths:
        f = 4.0 * heads * L * L * d
        total += f / 2.0 if causal else f
    return total


def attention_bwd_flops(heads: int, lengths, d: int, causal: bool) -> float:
    """Backward FLOP count: five L x L x d matmuls per head (S recomputed, dP = dO V^T,
    dV = P^T dO, dQ = dS K, dK = dS^T Q), i.e. 2.5x the forward count, halved for causal."""
    return 2.5 * attention_flops(heads, lengths, d, causal)


def attention_bwd_ideal_bytes(heads: int, total_tokens: int, d: int) -> int:
    """Backward minimum: read Q, K, V, O, dO once and write dQ, dK, dV once (bf16), read the
    lse (fp32)."""
    return heads * total_tokens * (8 * d * 2 + 4)


def attention_exact_flops(heads: int, lengths, d: int, causal: bool) -> float:
    """4 d FLOPs per visible (query, key) pair (the causal diagonal counted exactly)."""
    return float(sum(4 * heads * visible_pairs(int(L), causal) * d for L in lengths))


def attention_ideal_bytes(heads: int, total_tokens: int, d: int) -> int:
    """Fused forward minimum: read Q, K, V once and write O once (bf16), write LSE (fp32)."""
    return heads * total_tokens * (4 * d * BF16 + FP32)


def score_matrix_bytes(n: int, elem: int) -> int:
    """One head's materialised N x N score or probability matrix."""
    return n * n * elem


def unfused_bytes(batch: int, heads: int, n: int, d: int) -> int:
    """Three-kernel path through HBM: S (fp32) written then read, P (bf16) written then read,
    plus the fused minimum (Q, K, V read, O and LSE written)."""
    bh = batch * heads
    return bh * (2 * score_matrix_bytes(n, FP32) + 2 * score_matrix_bytes(n, BF16)) + \
        attention_ideal_bytes(heads, batch * n, d)


def tflops(flops: float, seconds: float) -> float:
    return flops / seconds / 1e12


def gbs(nbytes: float, seconds: float) -> float:
    return nbytes / seconds / 1e9


def bf16_half_ulp(x):
    """Half the bf16 spacing at |x| (the largest error of a correctly rounded bf16 output).

    bf16 keeps 8 significant bits, so values in [2^e, 2^(e+1)) are spaced 2^(e-7) apart.
    Works elementwise on numpy arrays or on a float.
    """
    try:
        import numpy as np
    except ImportError:  # pragma: no cover
        np = None
    if np is not None and hasattr(x, "shape"):
        ax = np.maximum(np.abs(x), 2.0 ** -126)
        e = np.floor(np.log2(ax))
        return 2.0 ** (e - 8)
    ax = max(abs(x), 2.0 ** -126)
    return 2.0 ** (math.floor(math.log2(ax)) - 8)
