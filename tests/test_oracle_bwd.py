"""Pins for the float64 backward oracle (CPU only).

The pages print no gradient values, so the backward oracle is pinned by things that do not
depend on it: central finite differences of the (separately pinned) forward oracle, invariants
of the definition, and special cases with closed forms.  Planted mistakes in copies of the
backward must each fail at least one pin.
"""
import math

import numpy as np
import pytest

from gen import inputs
from oracle import attention as orc
from oracle import backward as bwd


def grads(q, k, v, do, causal, scale):
    dq, dk, dv, _, _ = bwd.attention_bwd_head(q, k, v, do, causal, scale)
    return dq, dk, dv


def loss(q, k, v, do, causal, scale):
    """sum(dO * O) with O from the forward oracle: its gradient is the backward's output."""
    o, _ = orc.attention_head_rows(q, k, v, np.arange(q.shape[0]), causal, scale)
    return float(np.sum(do * o))


def _small(seed, L, d, amp=1.2):
    rng = np.random.default_rng(seed)
    return [rng.uniform(-amp, amp, size=(L, d)) for _ in range(4)]


def pin_failures(fn):
    """Run every pin against ``fn(q, k, v, do, causal, scale) -> (dq, dk, dv)``; returns the
    names of the failing pins."""
    fails = []

    def check(name, ok):
        if not ok:
            fails.append(name)

    # 1. every gradient entry against a central finite difference of the forward oracle
    eps = 1e-6
    for seed, (L, d) in enumerate([(1, 2), (3, 2), (5, 3), (6, 4)]):
        q, k, v, do = _small(100 + seed, L, d)
        for causal in (False, True):
            for scale in (1.0, 0.43):
                g = fn(q, k, v, do, causal, scale)
                ok = True
                for t, x in enumerate((q, k, v)):
                    for idx in np.ndindex(x.shape):
                        args = [q.copy(), k.copy(), v.copy()]
                        args[t][idx] += eps
                        lp = loss(*args, do, causal, scale)
                        args[t][idx] -= 2 * eps
                        lm = loss(*args, do, causal, scale)
                        fd = (lp - lm) / (2 * eps)
                        ok &= abs(fd - g[t][idx]) <= 1e-7 * (1 + abs(fd))
                check(f"finite difference L{L} d{d} c{causal} s{scale}", ok)

    L, d = 29, 8
    q = orc.bf16_bits_to_f64(inputs.bf16_normal(31, (L, d), 1.5))
    k = orc.bf16_bits_to_f64(inputs.bf16_normal(32, (L, d), 1.5))
    v = orc.bf16_bits_to_f64(inputs.bf16_normal(33, (L, d)))
    do = orc.bf16_bits_to_f64(inputs.bf16_normal(34, (L, d)))
    sc = 1.0 / math.sqrt(d)
    for causal in (False, True):
        dq, dk, dv = fn(q, k, v, do, causal, sc)
        # 2. shifting every key by the same vector leaves P unchanged: the rows of dK sum to 0
        check(f"sum dK c{causal}", np.allclose(dk.sum(0), 0.0, atol=1e-12))
        # 3. rows of P sum to one: the rows of dV sum to the rows of dO
        check(f"sum dV c{causal}", np.allclose(dv.sum(0), do.sum(0), atol=1e-12))
        # 4. equal V rows make O constant: no gradient reaches Q or K
        cst = np.broadcast_to(v[4], v.shape).copy()
        dq0, dk0, dv0 = fn(q, k, cst, do, causal, sc)
        check(f"const V c{causal}", np.allclose(dq0, 0, atol=1e-12) and
              np.allclose(dk0, 0, atol=1e-12))
        # 5. Q = 0: uniform P, dV_j = sum over the queries that see j of dO_i / (keys they see)
        _, _, dvz = fn(np.zeros_like(q), k, v, do, causal, sc)
        cnt = np.arange(1, L + 1) if causal else np.full(L, L)
        w = do / cnt[:, None]
        ref = np.cumsum(w[::-1], axis=0)[::-1] if causal else np.broadcast_to(w.sum(0), w.shape)
        check(f"q0 dV c{causal}", np.allclose(dvz, ref, atol=1e-12))
    # 6. a single key: O = V[0] whatever Q and K are
    dq1, dk1, dv1 = fn(q[:1], k[:1], v[:1], do[:1], False, sc)
    check("single key", np.allclose(dv1, do[:1], atol=1e-15) and
          np.allclose(dq1, 0, atol=1e-15) and np.allclose(dk1, 0, atol=1e-15))
    # 7. causal: a gradient on row r reaches only Q_r and keys/values 0..r
    r = 11
    dor = np.zeros_like(do); dor[r] = do[r]
    dq, dk, dv = fn(q, k, v, dor, True, sc)
    check("causal reach", np.all(dq[np.arange(L) != r] == 0) and np.all(dk[r + 1:] == 0) and
          np.all(dv[r + 1:] == 0) and np.any(dk[:r + 1] != 0))
    return fails


def test_backward_oracle_passes_all_pins():
    assert pin_failures(grads) == []


def test_blocked_recomputation_equals_definition():
    L, d = 203, 16
    q = inputs.bf16_normal(41, (L, d), 2.0)
    k = inputs.bf16_normal(42, (L, d), 2.0)
    v = inputs.bf16_normal(43, (L, d))
    do = inputs.bf16_normal(44, (L, d))
    for causal in (False, True):
        dq, dk, dv, o, lse = bwd.attention_bwd_head(q, k, v, do, causal, 0.25)
        for bq, bk in ((64, 64), (50, 33), (203, 7)):
            r = bwd.blocked_backward_head(q, k, v, o, lse, do, causal, 0.25, bq, bk)
            for a, b in zip(r, (dq, dk, dv)):
                assert np.max(np.abs(a - b)) < 1e-11


def test_dense_batch_matches_per_head():
    B, H, N, d = 2, 3, 40, 8
    q = inputs.bf16_normal(51, (B, H, N, d))
    k = inputs.bf16_normal(52, (B, H, N, d))
    v = inputs.bf16_normal(53, (B, H, N, d))
    do = inputs.bf16_normal(54, (B, H, N, d))
    res = bwd.attention_bwd_dense(q, k, v, do, True, 0.3)
    one = bwd.attention_bwd_head(q[1, 2], k[1, 2], v[1, 2], do[1, 2], True, 0.3)
    for a, b in zip(res, one):
        assert np.array_equal(a[1, 2], b)
    o, lse = orc.attention_dense(q, k, v, True, 0.3)
    assert np.allclose(res[3], o, atol=1e-14) and np.allclose(res[4], lse, atol=1e-14)


# ----------------------------------------------------------- planted mistakes (mutants)
def _parts(q, k, v, do, c, s):
    q, k, v, do = (np.asarray(x, float) for x in (q, k, v, do))
    p = orc.probabilities(q, k, c, s)
    return q, k, v, do, p


def _mut_no_d(q, k, v, do, c, s):  # softmax gradient without the D_i term
    q, k, v, do, p = _parts(q, k, v, do, c, s)
    ds = p * (do @ v.T)
    return s * ds @ k, s * ds.T @ q, p.T @ do


def _mut_sign(q, k, v, do, c, s):  # dS = P (D - dP)
    q, k, v, do, p = _parts(q, k, v, do, c, s)
    ds = p * (np.sum(do * (p @ v), 1, keepdims=True) - do @ v.T)
    return s * ds @ k, s * ds.T @ q, p.T @ do


def _mut_dk_unscaled(q, k, v, do, c, s):
    dq, dk, dv = grads(q, k, v, do, c, s)
    return dq, dk / s, dv


def _mut_dv_untransposed(q, k, v, do, c, s):  # dV = P dO
    dq, dk, _ = grads(q, k, v, do, c, s)
    _, _, _, do_, p = _parts(q, k, v, do, c, s)
    return dq, dk, p @ do_


def _mut_dq_transposed(q, k, v, do, c, s):  # dQ = scale dS^T K
    q, k, v, do, p = _parts(q, k, v, do, c, s)
    ds = p * (do @ v.T - np.sum(do * (p @ v), 1, keepdims=True))
    return s * ds.T @ k, s * ds.T @ q, p.T @ do


def _mut_d_from_dp(q, k, v, do, c, s):  # D_i = rowsum(dP) instead of rowsum(P * dP)
    q, k, v, do, p = _parts(q, k, v, do, c, s)
    dp = do @ v.T
    if c:
        dp = np.tril(dp)
    ds = p * (dp - dp.sum(1, keepdims=True) / max(1, dp.shape[1]))
    return s * ds @ k, s * ds.T @ q, p.T @ do


def _mut_unmasked_dv(q, k, v, do, c, s):  # P rebuilt without the causal mask for dV
    dq, dk, _ = grads(q, k, v, do, c, s)
    _, _, _, do_, p = _parts(q, k, v, do, False, s)
    return dq, dk, p.T @ do_


@pytest.mark.parametrize("mutant", [_mut_no_d, _mut_sign, _mut_dk_unscaled, _mut_dv_untransposed,
                                    _mut_dq_transposed, _mut_d_from_dp, _mut_unmasked_dv])
def test_pins_catch_planted_mistake(mutant):
    assert pin_failures(mutant), f"{mutant.__name__} slipped through every pin"


# ----------------------------------------------------------------- grouped-query backward
def _gqa_loss(q, k, v, do, causal, scale):
    o, _ = orc.attention_gqa_dense(q, k, v, causal, scale)
    return float(np.sum(do * o))


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_backward_finite_differences(causal):
    rng = np.random.default_rng(77)
    B, H, H_kv, N, d = 1, 4, 2, 5, 3
    q = rng.uniform(-1, 1, (B, H, N, d))
    k = rng.uniform(-1, 1, (B, H_kv, N, d))
    v = rng.uniform(-1, 1, (B, H_kv, N, d))
    do = rng.uniform(-1, 1, (B, H, N, d))
    dq, dk, dv, _, _ = bwd.attention_gqa_bwd_dense(q, k, v, do, causal, 0.6)
    eps = 1e-6
    for t, x, g in ((0, q, dq), (1, k, dk), (2, v, dv)):
        for idx in np.ndindex(x.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[t][idx] += eps
            lp = _gqa_loss(*args, do, causal, 0.6)
            args[t][idx] -= 2 * eps
            lm = _gqa_loss(*args, do, causal, 0.6)
            assert abs((lp - lm) / (2 * eps) - g[idx]) <= 1e-7 * (1 + abs(g[idx]))


def test_gqa_backward_with_all_heads_is_multi_head():
    q = inputs.bf16_normal(81, (2, 3, 40, 8))
    k = inputs.bf16_normal(82, (2, 3, 40, 8))
    v = inputs.bf16_normal(83, (2, 3, 40, 8))
    do = inputs.bf16_normal(84, (2, 3, 40, 8))
    a = bwd.attention_gqa_bwd_dense(q, k, v, do, True, 0.3)
    b = bwd.attention_bwd_dense(q, k, v, do, True, 0.3)
    for x, y in zip(a, b):
        assert np.allclose(x, y, atol=1e-13)
