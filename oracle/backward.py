"""Float64 CPU oracle for the attention backward pass (dQ, dK, dV).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU
baseline may import this module.  The product path never calls it and shares no code with it.

What the pages fix: the fused forward keeps no N x N matrix, saves one logsumexp per query row,
and the backward rebuilds S and P tile by tile from it ("CS336 Lecture 5" notes, section 6.2,
"反向传播怎么办"; CS336 GPU/attention notes, "为什么 FlashAttention 能减少内存").  The pages do not
write the gradient out; it is the chain rule applied to the definition of section 6.1
(``S = scale Q K^T``, ``P = softmax(S)`` by rows, ``O = P V``), for an upstream gradient dO:

* ``dV = P^T dO`` and ``dP = dO V^T`` (from ``O = P V``);
* softmax by rows: ``dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)``; the inner sum equals
  ``D_i = dO_i . O_i`` because ``sum_k P_ik V_k = O_i``;
* ``dQ = scale dS K`` and ``dK = scale dS^T Q`` (from ``S = scale Q K^T``).

Masked (causal) entries have P = 0 and therefore dS = 0.  All arithmetic is float64; inputs may
be float64 arrays or bf16 bit patterns (uint16), decoded exactly.  Layout: one head ``[L, d]``,
dense batches ``[B, H, N, d]``.
"""
from __future__ import annotations

import numpy as np

from .attention import _as_f64


def _scores(q, k, causal, scale):
    s = scale * (q @ k.T)
    if causal:
        L = s.shape[0]
        s = np.where(np.arange(L)[None, :] <= np.arange(L)[:, None], s, -np.inf)
    return s


def attention_bwd_head(q, k, v, do, causal: bool, scale: float):
    """Gradients of one head from the materialised definition.

    Returns (dq, dk, dv, o, lse): the three gradients [L, d] and the forward's O and LSE
    (natural log) that the backward kernels take as inputs.
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    s = _scores(q, k, causal, scale)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    ell = e.sum(axis=1, keepdims=True)
    p = e / ell                                   # P, zero where masked
    o = p @ v
    lse = (m + np.log(ell))[:, 0]
    dv = p.T @ do
    dp = do @ v.T
    dd = np.sum(do * o, axis=1, keepdims=True)    # D_i = dO_i . O_i
    ds = p * (dp - dd)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, o, lse


def attention_bwd_dense(q, k, v, do, causal: bool, scale: float, heads=None):
    """Dense batch ``[B, H, N, d]`` -> (dq, dk, dv, o, lse); ``heads``: optional (b, h) pairs to
    compute (the others are left NaN)."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    B, H, N, d = q.shape
    out = [np.full((B, H, N, d), np.nan) for _ in range(4)] + [np.full((B, H, N), np.nan)]
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        res = attention_bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
        for dst, src in zip(out, res):
            dst[b, h] = src
    return tuple(out)


def blocked_backward_head(q, k, v, o, lse, do, causal: bool, scale: float, block_q: int = 128,
                          block_kv: int = 128):
    """The pages' recomputation scheme for one head, in float64: nothing N x N is kept; for each
    key block j and query block i, S_ij is recomputed and ``P_ij = exp(S_ij - LSE_i)`` is rebuilt
    from the saved logsumexp, then dV_j, dK_j and dQ_i receive that block's contribution, with
    ``D_i = rowsum(dO_i * O_i)`` computed once from the saved output.

    ``o`` and ``lse`` are the forward's outputs (any precision); returns (dq, dk, dv).
    """
    q, k, v, o, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(o), _as_f64(do)
    lse = np.asarray(lse, dtype=np.float64)
    L, d = q.shape
    dd = np.sum(do * o, axis=1)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for j0 in range(0, L, block_kv):
        j1 = min(L, j0 + block_kv)
        for i0 in range(0, L, block_q):
            i1 = min(L, i0 + block_q)
            if causal and i1 - 1 < j0:
                continue  # every query of the block precedes every key of the block
            s = scale * (q[i0:i1] @ k[j0:j1].T)
            if causal:
                s = np.where(np.arange(j0, j1)[None, :] <= np.arange(i0, i1)[:, None], s,
                             -np.inf)
            p = np.exp(s - lse[i0:i1, None])
            dv[j0:j1] += p.T @ do[i0:i1]
            dp = do[i0:i1] @ v[j0:j1].T
            ds = p * (dp - dd[i0:i1, None])
            dq[i0:i1] += scale * (ds @ k[j0:j1])
            dk[j0:j1] += scale * (ds.T @ q[i0:i1])
    return dq, dk, dv


def attention_gqa_bwd_dense(q, k, v, do, causal: bool, scale: float):
    """Gradients of grouped-query attention (CS336 Lecture 5 notes, section 6.3: query head h
    reads K/V head h // (H // H_kv)), dense: q, do [B, H, N, d]; k, v [B, H_kv, N, d].

    A K/V head feeds every query head of its group, so its gradients are the sums of the
    per-query-head gradients over the group (the chain rule through a shared input).
    Returns (dq [B,H,N,d], dk [B,H_kv,N,d], dv [B,H_kv,N,d], o [B,H,N,d], lse [B,H,N]).
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    group = H // H_kv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros_like(q)
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            g = h // group
            r = attention_bwd_head(q[b, h], k[b, g], v[b, g], do[b, h], causal, scale)
            dq[b, h] = r[0]
            dk[b, g] += r[1]
            dv[b, g] += r[2]
            o[b, h] = r[3]
            lse[b, h] = r[4]
    return dq, dk, dv, o, lse
