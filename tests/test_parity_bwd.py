"""GPU parity of the backward pass (attn_bwd) against the float64 backward oracle.

The kernel receives the forward's outputs as inputs.  Most cases give it the oracle's O rounded
to bf16 and its LSE in fp32, so the comparison isolates the backward; one case chains the fused
forward into the backward.  The tolerance is derived from the arithmetic in parity_util.
"""

import numpy as np
import pytest
import torch

from gen import configs
from io_aware_attention_attn_gb300 import attn
from oracle import attention as orc
from oracle import backward as bwd

from parity_util import check_grad, grad_bounds, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from io_aware_attention_attn_gb300 import build
    build.build()
    yield
    assert attn.last_device_error() == 0


def f64_to_bf16_dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).cuda()


def make_case(w):
    """Inputs of a backward case: q, k, v and dO (bits) plus the oracle's gradients, O, LSE."""
    q, k, v, _ = w.make()
    do = w.make_dout()
    ref = bwd.attention_bwd_dense(q, k, v, do, w.causal, w.scale)
    return q, k, v, do, ref


def run_bwd(q, k, v, do, o, lse, causal, scale):
    dq, dk, dv = attn.attn_bwd(to_dev(q), to_dev(k), to_dev(v), o, lse, to_dev(do),
                               causal=causal, scale=scale)
    torch.cuda.synchronize()
    return to_f64(dq), to_f64(dk), to_f64(dv)


def check_all(q, k, v, do, grads, ref, causal, scale, what, heads=None):
    dq, dk, dv = grads
    B, H = q.shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        qf, kf, vf, dof = (orc.bf16_bits_to_f64(x[b, h]) for x in (q, k, v, do))
        aq, ak, av = grad_bounds(qf, kf, vf, dof, causal, scale)
        check_grad(dq[b, h], ref[0][b, h], aq, f"{what} dQ ({b},{h})")
        check_grad(dk[b, h], ref[1][b, h], ak, f"{what} dK ({b},{h})")
        check_grad(dv[b, h], ref[2][b, h], av, f"{what} dV ({b},{h})")


@pytest.mark.parametrize("seed,B,H,N,d,causal", [
    (701, 1, 2, 256, 128, False), (702, 1, 2, 256, 128, True),
    (703, 1, 2, 300, 128, True),      # ragged last tile
    (704, 2, 1, 129, 64, True),       # a one-row tail tile
    (705, 1, 3, 777, 64, False),
    (706, 1, 2, 1000, 128, True),
    (707, 1, 1, 1, 64, False),        # one key: dV = dO, dQ = dK = 0
    (708, 1, 2, 512, 128, False),
])
def test_bwd_dense(seed, B, H, N, d, causal):
    w = configs.custom(seed, B, H, N, d, causal)
    q, k, v, do, ref = make_case(w)
    o = f64_to_bf16_dev(ref[3])
    lse = torch.from_numpy(ref[4].astype(np.float32)).cuda()
    grads = run_bwd(q, k, v, do, o, lse, causal, w.scale)
    check_all(q, k, v, do, grads, ref, causal, w.scale, w.name)


def test_bwd_single_key_closed_form():
    w = configs.custom(709, 1, 1, 1, 128, True)
    q, k, v, do, ref = make_case(w)
    o = f64_to_bf16_dev(ref[3])
    lse = torch.from_numpy(ref[4].astype(np.float32)).cuda()
    dq, dk, dv = run_bwd(q, k, v, do, o, lse, True, w.scale)
    assert np.array_equal(dv, orc.bf16_bits_to_f64(do))
    assert np.all(np.abs(dq) < 1e-4) and np.all(np.abs(dk) < 1e-4)


def test_bwd_after_fused_forward():
    # the fused forward's own O and LSE feed the backward (the training use)
    w = configs.custom(710, 1, 2, 640, 128, True, sigma_qk=1.5)
    q, k, v, do, ref = make_case(w)
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=w.scale)
    grads = run_bwd(q, k, v, do, o, lse, True, w.scale)
    check_all(q, k, v, do, grads, ref, True, w.scale, "fwd->bwd")


def test_bwd_deterministic():
    w = configs.custom(711, 1, 2, 384, 64, False)
    q, k, v, do, ref = make_case(w)
    o = f64_to_bf16_dev(ref[3])
    lse = torch.from_numpy(ref[4].astype(np.float32)).cuda()
    a = run_bwd(q, k, v, do, o, lse, False, w.scale)
    b = run_bwd(q, k, v, do, o, lse, False, w.scale)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_full_size_sampled_heads(causal):
    # the headline shape (B=2, H=32, N=4096, d=128); three heads compared in full
    w = configs.custom(712, 2, 32, 4096, 128, causal)
    q, k, v, _ = w.make()
    do = w.make_dout()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=w.scale)
    grads = run_bwd(q, k, v, do, o, lse, causal, w.scale)
    heads = [(0, 0), (1, 17), (1, 31)]
    ref = bwd.attention_bwd_dense(q, k, v, do, causal, w.scale, heads=heads)
    check_all(q, k, v, do, grads, ref, causal, w.scale, w.name, heads=heads)


@pytest.mark.parametrize("seed,B,H,H_kv,N,d,causal", [
    (720, 1, 4, 2, 300, 128, True), (721, 2, 4, 1, 256, 64, False),
    (722, 1, 6, 3, 129, 128, False), (723, 1, 8, 2, 520, 64, True),
])
def test_bwd_gqa(seed, B, H, H_kv, N, d, causal):
    w = configs.custom(seed, B, H, N, d, causal, H_kv=H_kv)
    q, k, v, _ = w.make()
    do = w.make_dout()
    dq, dk, dv, o_ref, lse_ref = bwd.attention_gqa_bwd_dense(q, k, v, do, causal, w.scale)
    o = f64_to_bf16_dev(o_ref)
    lse = torch.from_numpy(lse_ref.astype(np.float32)).cuda()
    g = attn.attn_bwd(to_dev(q), to_dev(k), to_dev(v), o, lse, to_dev(do), causal=causal,
                      scale=w.scale)
    torch.cuda.synchronize()
    gq, gk, gv = (to_f64(x) for x in g)
    group = H // H_kv
    for b in range(B):
        for h in range(H):
            qf, kf, vf, dof = (orc.bf16_bits_to_f64(x) for x in
                               (q[b, h], k[b, h // group], v[b, h // group], do[b, h]))
            aq, _, _ = grad_bounds(qf, kf, vf, dof, causal, w.scale)
            check_grad(gq[b, h], dq[b, h], aq, f"{w.name} dQ ({b},{h})")
        for hk in range(H_kv):
            # the bound of a summed gradient is the sum of its terms' bounds
            ak = np.zeros_like(dk[b, hk]); av = np.zeros_like(dv[b, hk])
            for h in range(hk * group, (hk + 1) * group):
                qf, kf, vf, dof = (orc.bf16_bits_to_f64(x) for x in
                                   (q[b, h], k[b, hk], v[b, hk], do[b, h]))
                _, a_k, a_v = grad_bounds(qf, kf, vf, dof, causal, w.scale)
                ak += a_k; av += a_v
            check_grad(gk[b, hk], dk[b, hk], ak, f"{w.name} dK ({b},{hk})")
            check_grad(gv[b, hk], dv[b, hk], av, f"{w.name} dV ({b},{hk})")


def varlen_reference(q, k, v, do, cu, causal, scale):
    """Per-sequence, per-head backward oracle on packed [H, T, d] inputs (K/V heads may be fewer)."""
    H, T, d = q.shape
    H_kv = k.shape[0]
    group = H // H_kv
    dq = np.zeros((H, T, d)); dk = np.zeros((H_kv, T, d)); dv = np.zeros((H_kv, T, d))
    o = np.zeros((H, T, d)); lse = np.zeros((H, T))
    bounds_q = np.zeros((H, T, d)); bounds_k = np.zeros((H_kv, T, d)); bounds_v = np.zeros((H_kv, T, d))
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b == a:
            continue
        for h in range(H):
            g = h // group
            r = bwd.attention_bwd_head(q[h, a:b], k[g, a:b], v[g, a:b], do[h, a:b], causal, scale)
            dq[h, a:b] = r[0]; dk[g, a:b] += r[1]; dv[g, a:b] += r[2]
            o[h, a:b] = r[3]; lse[h, a:b] = r[4]
            qf, kf, vf, dof = (orc.bf16_bits_to_f64(x) for x in
                               (q[h, a:b], k[g, a:b], v[g, a:b], do[h, a:b]))
            aq, ak, av = grad_bounds(qf, kf, vf, dof, causal, scale)
            bounds_q[h, a:b] = aq; bounds_k[g, a:b] += ak; bounds_v[g, a:b] += av
    return (dq, dk, dv, o, lse), (bounds_q, bounds_k, bounds_v)


@pytest.mark.parametrize("seed,lengths,H,H_kv,d,causal", [
    (730, [1, 300, 0, 129, 640], 4, 4, 128, True),
    (731, [256, 77, 500], 4, 2, 64, False),
    (732, [1000], 2, 1, 128, True),
    (733, [130, 1, 129, 128, 257], 6, 3, 128, False),
])
def test_bwd_varlen(seed, lengths, H, H_kv, d, causal):
    q, k, v, cu = configs.custom_varlen(seed, lengths, H, d, causal, H_kv=H_kv)
    T = int(cu[-1])
    do = configs.custom(seed, 1, H, T, d, causal).make_dout()[0]   # [H, T, d]
    scale = 1 / np.sqrt(d)
    ref, bnd = varlen_reference(q, k, v, do, cu, causal, scale)
    o = f64_to_bf16_dev(ref[3])
    lse = torch.from_numpy(ref[4].astype(np.float32)).cuda()
    cu_d = torch.from_numpy(cu).cuda()
    g = attn.attn_bwd(to_dev(q), to_dev(k), to_dev(v), o, lse, to_dev(do), cu_seqlens=cu_d,
                      causal=causal, scale=scale)
    torch.cuda.synchronize()
    for name, x, r, b in zip(("dQ", "dK", "dV"), g, ref[:3], bnd):
        check_grad(to_f64(x), r, b, f"varlen {lengths} {name}")


def test_bwd_varlen_single_sequence_equals_dense():
    w = configs.custom(734, 1, 2, 300, 128, True)
    q, k, v, _ = w.make()
    do = w.make_dout()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=w.scale)
    a = attn.attn_bwd(to_dev(q), to_dev(k), to_dev(v), o, lse, to_dev(do), causal=True,
                      scale=w.scale)
    cu = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    b = attn.attn_bwd(to_dev(q[0]), to_dev(k[0]), to_dev(v[0]), o[0].contiguous(),
                      lse[0].contiguous(), to_dev(do[0]), cu_seqlens=cu, causal=True,
                      scale=w.scale)
    torch.cuda.synchronize()
    for x, y in zip(a, b):  # the same tiles in the same order: the same bits
        assert torch.equal(x[0].view(torch.int16), y.view(torch.int16))
