"""GPU parity of the fused forward (through the C ABI) against the float64 oracle.

Small and medium problems are compared element by element over every output; the five
workloads at full size are run in the launch configuration the bench times and compared on
sampled rows the oracle computes one by one, plus properties that hold at any size.
"""
import math

import numpy as np
import pytest
import torch

from gen import configs
from io_aware_attention_attn_gb300 import attn
from oracle import attention as orc

from parity_util import check, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from io_aware_attention_attn_gb300 import build
    build.build()
    yield
    assert attn.last_device_error() == 0


def run_dense(w: configs.Workload):
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    return q, k, v, o, lse


# ---------------------------------------------------------------- full comparisons
DENSE_CASES = [
    # (seed, B, H, N, d, causal)
    (101, 1, 2, 1, 64, False), (102, 1, 2, 1, 128, True),
    (103, 2, 2, 127, 64, False), (104, 2, 2, 127, 128, True),
    (105, 2, 2, 129, 128, False), (106, 2, 2, 129, 64, True),
    (107, 1, 3, 300, 128, True), (108, 1, 3, 300, 64, False),
    (109, 1, 2, 1000, 128, True), (110, 1, 2, 1000, 128, False),
    (111, 1, 1, 4097, 64, True), (112, 1, 1, 4097, 128, False),
    (113, 3, 1, 256, 128, True),
]


@pytest.mark.parametrize("seed,B,H,N,d,causal", DENSE_CASES)
def test_dense_full(seed, B, H, N, d, causal):
    w = configs.custom(seed, B, H, N, d, causal)
    q, k, v, o, lse = run_dense(w)
    o_ref, lse_ref = orc.attention_dense(q, k, v, causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, w.name)


def test_workload1_full():
    w = configs.WORKLOADS[1]
    q, k, v, o, lse = run_dense(w)
    o_ref, lse_ref = orc.attention_dense(q, k, v, w.causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, w.name)


def test_peaky_scores_full():
    # sigma(Q,K) = 2 as in the long causal workload: large running-max jumps and rescales
    w = configs.custom(120, 1, 2, 2000, 128, True, sigma_qk=2.0)
    q, k, v, o, lse = run_dense(w)
    o_ref, lse_ref = orc.attention_dense(q, k, v, True, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, w.name)


def test_scale_is_used_as_given():
    w = configs.custom(121, 1, 2, 300, 64, False)
    q, k, v, _ = w.make()
    for scale in (0.03, 0.5):
        o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=False, scale=scale)
        o_ref, lse_ref = orc.attention_dense(q, k, v, False, scale)
        check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, f"scale {scale}")


VARLEN_CASES = [
    (130, [1, 0, 300, 128, 129, 77], 3, 128, True),
    (131, [1, 0, 300, 128, 129, 77], 3, 128, False),
    (132, [5, 257, 0, 0, 64, 640], 2, 64, True),
    (133, [1], 1, 128, True),
    (134, [1000, 3], 2, 64, False),
]


@pytest.mark.parametrize("seed,lengths,H,d,causal", VARLEN_CASES)
def test_varlen_full(seed, lengths, H, d, causal):
    q, k, v, cu = configs.custom_varlen(seed, lengths, H, d, causal)
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=cu_t, causal=causal,
                           scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_varlen(q, k, v, cu, causal, 1 / math.sqrt(d))
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, f"varlen {lengths}")


def test_varlen_does_not_read_neighbours_v():
    # non-finite values in V rows of the next sequence must not leak into a tail tile
    lengths = [100, 50]
    q, k, v, cu = configs.custom_varlen(135, lengths, 1, 128, False)
    v = v.copy()
    v[:, 100:] = 0x7FC0  # NaN in every V row of the second sequence
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=cu_t, causal=False)
    o1 = to_f64(o)[:, :100]
    o_ref, lse_ref = orc.attention_head_rows(q[0, :100], k[0, :100], v[0, :100], np.arange(100),
                                             False, 1 / math.sqrt(128))
    check(o1[0], lse.cpu().numpy()[0, :100].astype(np.float64), o_ref, lse_ref, "neighbour NaN")


def test_varlen_single_sequence_equals_dense():
    # the packed layout with one sequence is the dense B=1 layout; the two are different kernel
    # instantiations (the compiler may round a few operations differently), so they must agree
    # within the parity tolerance, and each must match the oracle
    w = configs.custom(136, 1, 4, 700, 128, True)
    q, k, v, _ = w.make()
    o_d, l_d = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True)
    cu = torch.tensor([0, 700], dtype=torch.int32, device="cuda")
    o_v, l_v = attn.attn_fwd(to_dev(q[0]), to_dev(k[0]), to_dev(v[0]), cu_seqlens=cu, causal=True)
    od, ov = to_f64(o_d[0]), to_f64(o_v)
    check(od, l_d[0].cpu().numpy().astype(np.float64), ov, l_v.cpu().numpy().astype(np.float64),
          "dense vs packed B=1")
    o_ref, lse_ref = orc.attention_dense(q, k, v, True, w.scale)
    check(ov[None], l_v[None].cpu().numpy().astype(np.float64), o_ref, lse_ref, "packed B=1")


def test_causal_row0_is_v0_exactly():
    w = configs.custom(137, 2, 3, 500, 128, True)
    q, k, v, o, lse = run_dense(w)
    assert np.array_equal(o[:, :, 0].view(torch.int16).cpu().numpy().view(np.uint16), v[:, :, 0])
    s00 = (orc.bf16_bits_to_f64(q[:, :, 0]) * orc.bf16_bits_to_f64(k[:, :, 0])).sum(-1) * w.scale
    assert np.max(np.abs(lse[:, :, 0].cpu().numpy() - s00)) < 1e-4


def test_deterministic():
    w = configs.custom(138, 1, 4, 1500, 128, True)
    q, k, v, _ = w.make()
    a = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True)
    b = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)) and torch.equal(a[1], b[1])


def test_empty_is_noop():
    z = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = attn.attn_fwd(z, z, z)
    assert o.numel() == 0 and lse.numel() == 0


def test_explicit_stream():
    w = configs.custom(139, 1, 2, 256, 64, False)
    q, k, v, _ = w.make()
    s = torch.cuda.Stream()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = attn.attn_fwd(qd, kd, vd, stream=s)
    s.synchronize()
    o_ref, lse_ref = orc.attention_dense(q, k, v, False, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "stream")


# ------------------------------------------------------------ full-size workloads
def _sample_rows(N, rng, extra=64):
    fixed = [0, 1, 2, 126, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = np.unique(np.clip(np.concatenate([fixed, rng.integers(0, N, extra)]), 0, N - 1))
    return rows


def test_full_size_workload_2_every_element():
    """B=4, H=16, N=1024, d=64 causal in full: all 64 heads x 1024 rows against the oracle."""
    w = configs.WORKLOADS[2]
    q, k, v, o, lse = run_dense(w)
    o_ref, lse_ref = orc.attention_dense(q, k, v, w.causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, w.name + " (all rows)")


@pytest.mark.parametrize("index", [3, 4])
def test_full_size_dense_workload(index):
    w = configs.WORKLOADS[index]
    q, k, v, o, lse = run_dense(w)
    o_np = o.view(torch.int16).cpu().numpy().view(np.uint16)
    lse_np = lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(lse_np).all()
    o_all = orc.bf16_bits_to_f64(o_np)
    assert np.isfinite(o_all).all()
    rng = np.random.default_rng(index)
    heads = [(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))]
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b, h in heads:
        rows = _sample_rows(w.N, rng)
        ro, rl = orc.attention_head_rows(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale)
        got_o.append(o_all[b, h, rows]); got_l.append(lse_np[b, h, rows])
        ref_o.append(ro); ref_l.append(rl)
    check(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o),
          np.concatenate(ref_l), w.name)
    # property at any size: O is a convex combination of V rows -> within [min V, max V]
    vf = orc.bf16_bits_to_f64(v)
    assert o_all.max() <= vf.max() + 1e-2 and o_all.min() >= vf.min() - 1e-2


def test_full_size_varlen_workload():
    """The packed workload (16 sequences of U[128, 4096] rows, H=16, causal) at full size: every
    row of every sequence of four of the heads against the oracle."""
    w = configs.WORKLOADS[5]
    q, k, v, cu = w.make()
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=cu_t, causal=True,
                           scale=w.scale)
    torch.cuda.synchronize()
    o_all = to_f64(o)
    lse_np = lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(o_all).all() and np.isfinite(lse_np).all()
    heads = [0, 5, 10, 15]
    o_ref, lse_ref = orc.attention_varlen(q[heads], k[heads], v[heads], cu, True, w.scale)
    check(o_all[heads], lse_np[heads], o_ref, lse_ref, w.name + " (heads 0, 5, 10, 15, all rows)")
