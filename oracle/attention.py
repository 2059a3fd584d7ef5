"""Float64 CPU oracle for the IO-aware (FlashAttention-style) attention forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU
baseline may import this module.  The product path (the CUDA library and its Python binding)
never calls it and shares no code with it.

What it computes is the plain definition of scaled dot-product attention, because the fused
algorithm is exact: it changes the order of the computation, not the mathematics
("CS336 Lecture 5" notes, section 6.2, and the CS336 GPU/attention notes, section
"FlashAttention 的核心思想").  Sources, by page title and section:

* definition ``S = Q K^T / sqrt(d)``, ``P = softmax(S)`` row-wise, ``O = P V`` with
  ``Q, K, V in R^{N x d}`` -- CS336 Lecture 5 notes, section 6.1;
* stable softmax of a row: ``m = max s``, ``l = sum exp(s - m)``, ``p = exp(s - m) / l`` --
  CS336 GPU/attention notes, section "Online softmax 回顾";
* the per-row statistics saved for the backward pass are m and l "merged into a
  logsumexp", i.e. ``LSE = m + ln l`` -- CS336 Lecture 5 notes, section 6.2.

Readings where the pages are silent (each is listed in the design notes):

* ``scale`` is a free positive number (the pages use 1/sqrt(d)); it multiplies the scores
  before the softmax, so the LSE is that of the scaled scores, in natural-log units;
* causal masking keeps key j for query i iff ``j <= i`` (positions counted from the start of
  each sequence; queries and keys have the same length, so the two usual alignments agree);
* packed variable-length batches are independent sequences: no query sees a key of another
  sequence;
* a query with no visible key cannot occur (the diagonal is always visible); an empty
  sequence produces no rows.

Layouts: dense ``[B, H, N, d]``; packed ``[H, T, d]`` with ``cu_seqlens`` (int, length n+1).
All arithmetic is float64.  Inputs may be float64 arrays or bf16 bit patterns (uint16),
which are decoded exactly.
"""
from __future__ import annotations

import numpy as np

# rows of S held at once; a whole row is always materialised, this only bounds memory
_ROW_BLOCK = 256


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bfloat16 bit patterns (the bf16 value is the top half of an f32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _as_f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float64)


def attention_head_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows, causal: bool,
                        scale: float):
    """Attention for selected query rows of one head of one sequence.

    ``q``: [L, d], ``k``: [L, d], ``v``: [L, d] (float64 or bf16 bits); ``rows``: query
    indices.  Returns (O [len(rows), d], LSE [len(rows)]).  Each row i materialises the whole
    score row ``s_i = scale * q_i K^T`` over its visible keys, then takes the two-pass stable
    softmax (max, then sum of exponentials) and the probability-weighted sum of V.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    rows = np.asarray(rows, dtype=np.int64)
    L = k.shape[0]
    o = np.empty((len(rows), v.shape[1]), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    for r0 in range(0, len(rows), _ROW_BLOCK):
        rr = rows[r0:r0 + _ROW_BLOCK]
        kmax = L if not causal else int(rr.max()) + 1  # keys beyond the last row are never visible
        s = scale * (q[rr] @ k[:kmax].T)                 # [rows, kmax], every visible score
        if causal:
            j = np.arange(kmax)[None, :]
            s = np.where(j <= rr[:, None], s, -np.inf)   # key j visible to query i iff j <= i
        m = s.max(axis=1, keepdims=True)                 # pass 1: row maximum
        e = np.exp(s - m)                                # masked entries give exp(-inf) = 0
        ell = e.sum(axis=1, keepdims=True)               # pass 2: normaliser
        o[r0:r0 + len(rr)] = (e / ell) @ v[:kmax]
        lse[r0:r0 + len(rr)] = (m + np.log(ell))[:, 0]
    return o, lse


def attention_dense(q, k, v, causal: bool, scale: float, heads=None):
    """Dense batch ``[B, H, N, d]`` -> (O [B,H,N,d], LSE [B,H,N]) in float64.

    ``heads``: optional list of (b, h) pairs to compute; the others are left as NaN.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    o = np.full((B, H, N, d), np.nan)
    lse = np.full((B, H, N), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        o[b, h], lse[b, h] = attention_head_rows(q[b, h], k[b, h], v[b, h], np.arange(N),
                                                 causal, scale)
    return o, lse


def attention_varlen(q, k, v, cu_seqlens, causal: bool, scale: float):
    """Packed batch ``[H, T, d]`` with ``cu_seqlens`` -> (O [H,T,d], LSE [H,T]) in float64.

    Sequence s occupies rows ``cu_seqlens[s] .. cu_seqlens[s+1]-1`` of every head and attends
    only to itself.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    H, T, d = q.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    o = np.full((H, T, d), np.nan)
    lse = np.full((H, T), np.nan)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b == a:
            continue
        for h in range(H):
            o[h, a:b], lse[h, a:b] = attention_head_rows(q[h, a:b], k[h, a:b], v[h, a:b],
                                                         np.arange(b - a), causal, scale)
    return o, lse


def attention_gqa_dense(q, k, v, causal: bool, scale: float, heads=None):
    """Grouped-query attention, dense: q [B, H, N, d], k and v [B, H_kv, N, d] with H_kv | H.

    Query head h attends with key/value head h // (H // H_kv): several query heads share one K/V
    head (CS336 Lecture 5 notes, section 6.3, "MQA / GQA"); H_kv = 1 is multi-query attention.
    Returns (O [B,H,N,d], LSE [B,H,N]); ``heads``: optional (b, h) pairs to compute (others NaN).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    group = H // k.shape[1]
    o = np.full((B, H, N, d), np.nan)
    lse = np.full((B, H, N), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        o[b, h], lse[b, h] = attention_head_rows(q[b, h], k[b, h // group], v[b, h // group],
                                                 np.arange(N), causal, scale)
    return o, lse


def attention_gqa_varlen(q, k, v, cu_seqlens, causal: bool, scale: float):
    """Grouped-query attention on a packed batch: q [H, T, d], k and v [H_kv, T, d]."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    H, T, d = q.shape
    group = H // k.shape[0]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    o = np.full((H, T, d), np.nan)
    lse = np.full((H, T), np.nan)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b == a:
            continue
        for h in range(H):
            o[h, a:b], lse[h, a:b] = attention_head_rows(q[h, a:b], k[h // group, a:b],
                                                         v[h // group, a:b], np.arange(b - a),
                                                         causal, scale)
    return o, lse


def probabilities(q, k, causal: bool, scale: float) -> np.ndarray:
    """The full probability matrix P = softmax(scale * q k^T) of one head ([L, L]; small L)."""
    q, k = _as_f64(q), _as_f64(k)
    s = scale * (q @ k.T)
    if causal:
        L = s.shape[0]
        s = np.where(np.arange(L)[None, :] <= np.arange(L)[:, None], s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True)


def online_softmax_attention(q, k, v, causal: bool, scale: float, block_q: int = 128,
                             block_kv: int = 128, kv_blocks=None):
    """The tiled single-pass algorithm of the pages, in float64, for one head ([L, d]).

    Follows the FlashAttention forward of CS336 Lecture 5 notes, section 6.2 (outer loop over
    query blocks, inner loop over key/value blocks, running row maximum ``m`` and normaliser
    ``l``, the output accumulator rescaled by ``exp(m_old - m_new)`` whenever the maximum
    grows, a single division by ``l`` at the end) with the block merge of the CS336
    GPU/attention notes, section "Online softmax 回顾":
    ``m_new = max(m_old, m_B)``, ``l_new = l_old e^{m_old-m_new} + l_B e^{m_B-m_new}``,
    ``a_new = a_old e^{m_old-m_new} + a_B e^{m_B-m_new}``, output ``a/l``.

    ``kv_blocks``: optional explicit list of key-block boundaries (to test uneven blocks).
    Returns (O [L, d], LSE [L]) where LSE = m + ln l.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    L, d = q.shape
    o = np.empty_like(q)
    lse = np.empty(L)
    if kv_blocks is None:
        kv_blocks = list(range(0, L, block_kv)) + [L]
    for i0 in range(0, L, block_q):
        i1 = min(L, i0 + block_q)
        qi = q[i0:i1]
        m = np.full(i1 - i0, -np.inf)
        ell = np.zeros(i1 - i0)
        acc = np.zeros((i1 - i0, d))
        for j0, j1 in zip(kv_blocks[:-1], kv_blocks[1:]):
            if causal and j0 > i1 - 1:
                break  # every key of this block lies after every query of the block
            s = scale * (qi @ k[j0:j1].T)
            if causal:
                s = np.where(np.arange(j0, j1)[None, :] <= np.arange(i0, i1)[:, None], s,
                             -np.inf)
            m_b = s.max(axis=1)
            m_new = np.maximum(m, m_b)
            # rows that have seen no visible key yet keep m = -inf; use 0 there to avoid inf-inf
            safe = np.where(np.isfinite(m_new), m_new, 0.0)
            e = np.exp(s - safe[:, None])
            ell_b = e.sum(axis=1)
            alpha = np.exp(m - safe)          # correction factor e^{m_old - m_new}
            ell = ell * alpha + ell_b
            acc = acc * alpha[:, None] + e @ v[j0:j1]
            m = m_new
        o[i0:i1] = acc / ell[:, None]
        lse[i0:i1] = m + np.log(ell)
    return o, lse


def slice_partials(q, k, v, causal: bool, scale: float, cuts):
    """Per-slice partial results of one head ([L, d]) for key slices ``cuts[s] .. cuts[s+1]-1``.

    For every slice s and query row: the slice's row maximum ``m_s`` of the scaled visible scores
    (-inf when the slice holds no visible key), ``l_s = sum exp(s - m_s)`` and the unnormalised
    output ``a_s = sum exp(s - m_s) v`` -- the (m, l, a) triple of a block in the CS336
    GPU/attention notes, section "Online softmax 回顾".  Returns arrays m [S, L], l [S, L],
    a [S, L, d].
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    L, d = q.shape
    S = len(cuts) - 1
    m = np.full((S, L), -np.inf)
    ell = np.zeros((S, L))
    a = np.zeros((S, L, d))
    rows = np.arange(L)
    for s in range(S):
        j0, j1 = int(cuts[s]), int(cuts[s + 1])
        if j1 <= j0:
            continue
        sc = scale * (q @ k[j0:j1].T)
        if causal:
            sc = np.where(np.arange(j0, j1)[None, :] <= rows[:, None], sc, -np.inf)
        ms = sc.max(axis=1)
        seen = np.isfinite(ms)
        e = np.exp(sc[seen] - ms[seen, None])
        m[s, seen] = ms[seen]
        ell[s, seen] = e.sum(axis=1)
        a[s, seen] = e @ v[j0:j1]
    return m, ell, a


def merge_slices(m, ell, a):
    """Merge per-slice (m, l, a) triples into (O, LSE) by the block merge of the CS336
    GPU/attention notes, section "Online softmax 回顾", applied to all slices at once:
    ``M = max_s m_s``, each slice weighted by ``exp(m_s - M)``, ``O = sum w a / sum w l``,
    ``LSE = M + ln(sum w l)``.  Slices with ``m_s = -inf`` carry weight 0."""
    M = m.max(axis=0)
    w = np.where(np.isfinite(m), np.exp(m - np.where(np.isfinite(M), M, 0.0)[None, :]), 0.0)
    lw = (w * ell).sum(axis=0)
    o = (w[:, :, None] * a).sum(axis=0) / lw[:, None]
    return o, M + np.log(lw)
