"""Pins for the float64 oracle: brute force, closed forms and invariants (CPU only).

No numeric attention example is printed on the pages, so the oracle is pinned by things
that do not depend on it: a separate brute-force triple loop (no max subtraction,
``math.fsum``), closed forms of special inputs, and invariants of the definition.  The last
test plants plausible mistakes in copies of the oracle and checks that each one is caught.
"""
import math

import numpy as np
import pytest

from gen import configs, inputs
from oracle import attention as orc


def head_fn(q, k, v, causal, scale):
    """The oracle on one head of one sequence, all rows."""
    return orc.attention_head_rows(q, k, v, np.arange(q.shape[0]), causal, scale)


# --------------------------------------------------------------------------- brute force
def brute_force(q, k, v, causal, scale):
    """Textbook softmax(scale q k^T) v with pure-Python loops, exp without max subtraction,
    exactly rounded sums (math.fsum); LSE = log(sum exp(s))."""
    L, d = len(q), len(q[0])
    O, LSE = [], []
    for i in range(L):
        keys = [j for j in range(L) if (not causal or j <= i)]
        s = [scale * math.fsum(q[i][c] * k[j][c] for c in range(d)) for j in keys]
        e = [math.exp(x) for x in s]
        z = math.fsum(e)
        O.append([math.fsum(e[t] * v[j][c] for t, j in enumerate(keys)) / z for c in range(d)])
        LSE.append(math.log(z))
    return np.array(O), np.array(LSE)


def _small(seed, L, d, amp=1.5):
    rng = np.random.default_rng(seed)
    return [rng.uniform(-amp, amp, size=(L, d)) for _ in range(3)]


# --------------------------------------------------------------------------- pin suite
def pin_failures(fn):
    """Run every pin against a one-head attention function ``fn(q,k,v,causal,scale)``.
    Returns the names of the pins that fail (empty for a correct implementation)."""
    fails = []

    def check(name, ok):
        if not ok:
            fails.append(name)

    # 1. brute force on tiny inputs
    for seed, (L, d) in enumerate([(1, 1), (2, 3), (5, 4), (8, 2), (7, 4)]):
        q, k, v = _small(seed, L, d)
        for causal in (False, True):
            for scale in (1.0, 0.37):
                o, lse = fn(q, k, v, causal, scale)
                ob, lb = brute_force(q.tolist(), k.tolist(), v.tolist(), causal, scale)
                check(f"brute L{L} d{d} c{causal} s{scale}",
                      np.allclose(o, ob, atol=1e-12, rtol=0) and
                      np.allclose(lse, lb, atol=1e-12, rtol=0))
    # inputs with bf16 values from the generator for the closed forms
    L, d = 37, 16
    q = orc.bf16_bits_to_f64(inputs.bf16_normal(11, (L, d)))
    k = orc.bf16_bits_to_f64(inputs.bf16_normal(12, (L, d)))
    v = orc.bf16_bits_to_f64(inputs.bf16_normal(13, (L, d)))
    sc = 1.0 / math.sqrt(d)
    # 2. Q = 0: uniform probabilities over the visible keys
    for causal in (False, True):
        o, lse = fn(np.zeros_like(q), k, v, causal, sc)
        cnt = np.arange(1, L + 1) if causal else np.full(L, L)
        mean = np.cumsum(v, axis=0) / cnt[:, None] if causal else np.broadcast_to(v.mean(0), v.shape)
        check(f"q0 mean c{causal}", np.allclose(o, mean, atol=1e-13, rtol=0))
        check(f"q0 lse c{causal}", np.allclose(lse, np.log(cnt), atol=1e-13, rtol=0))
    # 3. a single key: O = V[0], LSE = s00
    o, lse = fn(q[:1], k[:1], v[:1], False, sc)
    check("single key O", np.array_equal(o[0], v[0]))
    check("single key LSE", abs(lse[0] - sc * float(q[0] @ k[0])) < 1e-14)
    # 4. causal row 0 sees only key 0
    o, lse = fn(q, k, v, True, sc)
    check("causal row0 O", np.array_equal(o[0], v[0]))
    check("causal row0 LSE", abs(lse[0] - sc * float(q[0] @ k[0])) < 1e-14)
    # 5. constant V rows give that constant
    cst = np.broadcast_to(v[3], v.shape).copy()
    for causal in (False, True):
        o, _ = fn(q, k, cst, causal, sc)
        check(f"const V c{causal}", np.allclose(o, cst, atol=1e-13, rtol=0))
    # 6. non-causal: permuting keys and values together changes nothing
    perm = np.random.default_rng(5).permutation(L)
    o1, l1 = fn(q, k, v, False, sc)
    o2, l2 = fn(q, k[perm], v[perm], False, sc)
    check("kv permutation", np.allclose(o1, o2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13))
    # 7. causal row i equals non-causal attention over the prefix 0..i
    oc, lc = fn(q, k, v, True, sc)
    ok = True
    for i in (1, 5, 17, L - 1):
        op, lp = fn(q[: i + 1], k[: i + 1], v[: i + 1], False, sc)
        ok &= np.allclose(oc[i], op[i], atol=1e-13) and abs(lc[i] - lp[i]) < 1e-13
    check("causal prefix", ok)
    # 8. shift invariance: K + w adds scale*q_i.w to every score of row i
    w = np.linspace(-0.7, 0.9, d)
    for causal in (False, True):
        o1, l1 = fn(q, k, v, causal, sc)
        o2, l2 = fn(q, k + w, v, causal, sc)
        check(f"shift c{causal}", np.allclose(o1, o2, atol=1e-12) and
              np.allclose(l2 - l1, sc * (q @ w), atol=1e-12))
    # 9. one dominant key: O -> that key's value row
    qd = np.zeros((4, d)); qd[:, 0] = 1.0
    kd = np.zeros((4, d)); kd[2, 0] = 200.0
    vd = np.arange(4 * d, dtype=float).reshape(4, d)
    o, lse = fn(qd, kd, vd, False, 1.0)
    check("dominant key", np.allclose(o, np.broadcast_to(vd[2], o.shape), atol=1e-12) and
          np.allclose(lse, 200.0 + np.log1p(3 * np.exp(-200.0)), atol=1e-12))
    # 10. rows of P sum to one and O = P V
    P = orc.probabilities(q, k, True, sc)
    check("P rows", np.allclose(P.sum(1), 1.0, atol=1e-14) and np.all(np.triu(P, 1) == 0))
    check("O = PV", np.allclose(fn(q, k, v, True, sc)[0], P @ v, atol=1e-13))
    return fails


def test_oracle_passes_all_pins():
    assert pin_failures(head_fn) == []


# ----------------------------------------------------------- planted mistakes (mutants)
def _mut_no_scale(q, k, v, c, s):
    return head_fn(q, k, v, c, 1.0)


def _mut_transposed(q, k, v, c, s):  # scores k_i . q_j instead of q_i . k_j
    return head_fn(k, q, v, c, s)


def _mut_mask_strict(q, k, v, c, s):  # causal keeps j < i (drops the diagonal)
    L = q.shape[0]
    if not c:
        return head_fn(q, k, v, c, s)
    o = np.zeros_like(q[:, :v.shape[1]]); lse = np.zeros(L)
    for i in range(L):
        if i == 0:
            o[0], lse[0] = v[0], 0.0
            continue
        oo, ll = orc.attention_head_rows(q[: i + 1], k[:i], v[:i], [i], False, s)
        o[i], lse[i] = oo[0], ll[0]
    return o, lse


def _mut_lse_no_max(q, k, v, c, s):  # LSE = ln l only
    o, lse = head_fn(q, k, v, c, s)
    sc = s * (np.asarray(q, float) @ np.asarray(k, float).T)
    if c:
        sc = np.where(np.tril(np.ones_like(sc)) > 0, sc, -np.inf)
    return o, lse - sc.max(1)


def _mut_lse_log2(q, k, v, c, s):
    o, lse = head_fn(q, k, v, c, s)
    return o, lse / math.log(2.0)


def _mut_column_softmax(q, k, v, c, s):  # normalise over queries instead of keys
    q, k, v = (np.asarray(x, float) for x in (q, k, v))
    sc = s * (q @ k.T)
    if c:
        sc = np.where(np.tril(np.ones_like(sc)) > 0, sc, -np.inf)
    m = sc.max(0, keepdims=True)
    e = np.exp(sc - m)
    p = e / e.sum(0, keepdims=True)
    return p @ v, (m + np.log(e.sum(0, keepdims=True)))[0]


def _mut_v_reversed(q, k, v, c, s):
    return head_fn(q, k, np.asarray(v)[::-1], c, s)


def _mut_dropped_rescale(q, k, v, c, s):  # online softmax that never rescales the accumulator
    q, k, v = (np.asarray(x, float) for x in (q, k, v))
    L = q.shape[0]
    o = np.empty((L, v.shape[1])); lse = np.empty(L)
    for i in range(L):
        m = -np.inf; ell = 0.0; acc = np.zeros(v.shape[1])
        for j in range(L if not c else i + 1):
            x = s * float(q[i] @ k[j]); mn = max(m, x)
            ell = ell * math.exp(m - mn) + math.exp(x - mn)
            acc = acc + math.exp(x - mn) * v[j]          # missing acc * exp(m - mn)
            m = mn
        o[i], lse[i] = acc / ell, m + math.log(ell)
    return o, lse


@pytest.mark.parametrize("mutant", [_mut_no_scale, _mut_transposed, _mut_mask_strict,
                                    _mut_lse_no_max, _mut_lse_log2, _mut_column_softmax,
                                    _mut_v_reversed, _mut_dropped_rescale])
def test_pins_catch_planted_mistake(mutant):
    assert pin_failures(mutant), f"{mutant.__name__} slipped through every pin"


# --------------------------------------------------------------- online == two-pass
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L,bq,bk", [(300, 128, 128), (129, 128, 128), (77, 16, 32), (1, 128, 128)])
def test_online_softmax_equals_two_pass(causal, L, bq, bk):
    d = 32
    q = inputs.bf16_normal(101, (L, d), 2.0)
    k = inputs.bf16_normal(102, (L, d), 2.0)
    v = inputs.bf16_normal(103, (L, d))
    o1, l1 = head_fn(q, k, v, causal, 1 / math.sqrt(d))
    o2, l2 = orc.online_softmax_attention(q, k, v, causal, 1 / math.sqrt(d), bq, bk)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def test_online_softmax_uneven_blocks():
    L, d = 211, 8
    q = inputs.bf16_normal(7, (L, d), 3.0)
    k = inputs.bf16_normal(8, (L, d), 3.0)
    v = inputs.bf16_normal(9, (L, d))
    rng = np.random.default_rng(0)
    cuts = np.unique(np.concatenate([[0, L], rng.integers(1, L, 12)])).tolist()
    for causal in (False, True):
        o1, l1 = head_fn(q, k, v, causal, 0.5)
        o2, l2 = orc.online_softmax_attention(q, k, v, causal, 0.5, 50, kv_blocks=cuts)
        assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


# ------------------------------------------------------------ batched entry points
def test_dense_matches_per_head():
    w = configs.custom(40, B=2, H=3, N=70, d=16, causal=True)
    q, k, v, _ = w.make()
    o, lse = orc.attention_dense(q, k, v, True, w.scale)
    for b in range(2):
        for h in range(3):
            oh, lh = head_fn(q[b, h], k[b, h], v[b, h], True, w.scale)
            assert np.array_equal(o[b, h], oh) and np.array_equal(lse[b, h], lh)


def test_varlen_equals_dense_per_sequence():
    lengths = [5, 0, 130, 1, 64]
    H, d = 2, 16
    q, k, v, cu = configs.custom_varlen(41, lengths, H, d, True)
    for causal in (False, True):
        o, lse = orc.attention_varlen(q, k, v, cu, causal, 0.25)
        for s, L in enumerate(lengths):
            a = int(cu[s])
            for h in range(H):
                if L == 0:
                    continue
                oh, lh = head_fn(q[h, a:a + L], k[h, a:a + L], v[h, a:a + L], causal, 0.25)
                assert np.allclose(o[h, a:a + L], oh, atol=1e-13)
                assert np.allclose(lse[h, a:a + L], lh, atol=1e-13)
        assert not np.isnan(o).any()


def test_varlen_single_sequence_is_dense_b1():
    H, N, d = 2, 100, 16
    q, k, v, cu = configs.custom_varlen(42, [N], H, d, True)
    o1, l1 = orc.attention_varlen(q, k, v, cu, True, 0.3)
    o2, l2 = orc.attention_dense(q[None], k[None], v[None], True, 0.3)
    assert np.array_equal(o1, o2[0]) and np.array_equal(l1, l2[0])


def test_sampled_rows_match_full():
    w = configs.custom(43, B=1, H=1, N=600, d=32, causal=True)
    q, k, v, _ = w.make()
    o, lse = head_fn(q[0, 0], k[0, 0], v[0, 0], True, w.scale)
    rows = np.array([0, 1, 255, 256, 599])
    o2, l2 = orc.attention_head_rows(q[0, 0], k[0, 0], v[0, 0], rows, True, w.scale)
    assert np.allclose(o[rows], o2, atol=1e-14) and np.allclose(lse[rows], l2, atol=1e-14)


def test_bf16_decode_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x4049, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -1.0, 0.0, -0.0, 3.140625, 3.3895313892515355e38, 9.183549615799121e-41]
    assert orc.bf16_bits_to_f64(bits).tolist() == want


# ------------------------------------------------------------- grouped-query attention
def _gqa_inputs(seed, B, H, H_kv, N, d):
    w = configs.custom(seed, B, H, N, d, False, H_kv=H_kv)
    q, k, v, _ = w.make()
    return q, k, v


def test_gqa_with_all_heads_is_multi_head():
    q, k, v = _gqa_inputs(60, 2, 4, 4, 50, 16)
    for causal in (False, True):
        a = orc.attention_gqa_dense(q, k, v, causal, 0.3)
        b = orc.attention_dense(q, k, v, causal, 0.3)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("H_kv", [1, 2, 3])
def test_gqa_equals_multi_head_on_repeated_kv(H_kv):
    H = 6
    q, k, v = _gqa_inputs(61, 2, H, H_kv, 40, 8)
    rk, rv = np.repeat(k, H // H_kv, axis=1), np.repeat(v, H // H_kv, axis=1)
    for causal in (False, True):
        a = orc.attention_gqa_dense(q, k, v, causal, 0.35)
        b = orc.attention_dense(q, rk, rv, causal, 0.35)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_gqa_interleaved_grouping_is_caught():
    # planted mistake: query head h reading K/V head h % H_kv instead of h // (H / H_kv)
    q, k, v = _gqa_inputs(62, 1, 4, 2, 30, 8)
    good = orc.attention_gqa_dense(q, k, v, False, 0.4)[0]
    wrong = np.stack([orc.attention_head_rows(q[0, h], k[0, h % 2], v[0, h % 2], np.arange(30),
                                              False, 0.4)[0] for h in range(4)])[None]
    rk, rv = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    ref = orc.attention_dense(q, rk, rv, False, 0.4)[0]
    assert np.array_equal(good, ref) and not np.allclose(wrong, ref)


def test_gqa_varlen_matches_dense_per_sequence():
    lengths = [7, 0, 65]
    q, k, v, cu = configs.custom_varlen(63, lengths, 4, 8, True, H_kv=2)
    o, lse = orc.attention_gqa_varlen(q, k, v, cu, True, 0.5)
    for s, L in enumerate(lengths):
        a = int(cu[s])
        if L == 0:
            continue
        od, ld = orc.attention_gqa_dense(q[None, :, a:a + L], k[None, :, a:a + L],
                                         v[None, :, a:a + L], True, 0.5)
        assert np.allclose(o[:, a:a + L], od[0], atol=1e-14) and np.allclose(lse[:, a:a + L], ld[0], atol=1e-14)


# --------------------------------------------------------- split-KV merge of slices
@pytest.mark.parametrize("causal", [False, True])
def test_merged_slices_equal_definition(causal):
    L, d = 230, 16
    q = inputs.bf16_normal(21, (L, d), 3.0)
    k = inputs.bf16_normal(22, (L, d), 3.0)
    v = inputs.bf16_normal(23, (L, d))
    # uneven slices, one empty, and (causal) slices that early rows cannot see at all
    for cuts in ([0, 100, 100, 170, 230], [0, 1, 2, 229, 230], [0, 230]):
        m, ell, a = orc.slice_partials(q, k, v, causal, 0.3, cuts)
        o1, l1 = head_fn(q, k, v, causal, 0.3)
        o2, l2 = orc.merge_slices(m, ell, a)
        assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12
    if causal:
        m, _, _ = orc.slice_partials(q, k, v, True, 0.3, [0, 100, 230])
        assert np.isneginf(m[1, :100]).all() and np.isfinite(m[1, 100:]).all()


def test_merge_without_slice_weights_is_caught():
    # a merge that forgets the exp(m_s - M) weights gives a different answer
    L, d = 64, 8
    q = inputs.bf16_normal(24, (L, d), 3.0)
    k = inputs.bf16_normal(25, (L, d), 3.0)
    v = inputs.bf16_normal(26, (L, d))
    m, ell, a = orc.slice_partials(q, k, v, False, 0.5, [0, 20, 64])
    bad = (a.sum(axis=0)) / ell.sum(axis=0)[:, None]
    o_ref, _ = head_fn(q, k, v, False, 0.5)
    assert np.max(np.abs(bad - o_ref)) > 1e-3
