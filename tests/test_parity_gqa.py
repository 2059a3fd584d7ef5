"""GPU parity of grouped-query / multi-query attention (attn_fwd_gqa) against the float64 oracle."""
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


@pytest.mark.parametrize("seed,B,H,H_kv,N,d,causal", [
    (501, 2, 8, 2, 300, 128, False), (502, 2, 8, 2, 300, 128, True),
    (503, 1, 8, 1, 517, 64, True), (504, 1, 6, 3, 129, 64, False),
    (505, 2, 4, 4, 256, 128, True), (506, 1, 16, 4, 1000, 128, True),
])
def test_gqa_dense(seed, B, H, H_kv, N, d, causal):
    w = configs.custom(seed, B, H, N, d, causal, H_kv=H_kv)
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_gqa_dense(q, k, v, causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, w.name)


def test_gqa_varlen():
    lengths = [1, 300, 0, 129, 640]
    q, k, v, cu = configs.custom_varlen(507, lengths, 8, 128, True, H_kv=2)
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=torch.from_numpy(cu).cuda(),
                           causal=True, scale=1 / math.sqrt(128))
    o_ref, lse_ref = orc.attention_gqa_varlen(q, k, v, cu, True, 1 / math.sqrt(128))
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "gqa varlen")


def test_gqa_equals_mha_on_repeated_kv_bitwise():
    # the same kernel instantiation reading a shared K/V head or a private copy of it
    w = configs.custom(508, 1, 8, 700, 128, True, H_kv=2)
    q, k, v, _ = w.make()
    a = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True)
    rk, rv = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    lib = attn.lib()
    qd, kd, vd = to_dev(q), to_dev(rk), to_dev(rv)
    o = torch.empty_like(qd)
    l = torch.empty(qd.shape[:-1], dtype=torch.float32, device="cuda")
    assert lib.attn_fwd_gqa(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), l.data_ptr(),
                            None, 1, 8, 8, 700, 128, 1, w.scale, None) == 0
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), o.view(torch.int16)) and torch.equal(a[1], l)


def test_gqa_full_size_sampled():
    w = configs.GQA
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    heads = [(0, 0), (0, 3), (1, 31), (int(rng.integers(2)), int(rng.integers(32)))]
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.integers(0, w.N, 60)]))
    o_np, l_np = to_f64(o), lse.cpu().numpy().astype(np.float64)
    go, gl, ro, rl = [], [], [], []
    for b, h in heads:
        a, c = orc.attention_head_rows(q[b, h], k[b, h // 4], v[b, h // 4], rows, False, w.scale)
        go.append(o_np[b, h, rows]); gl.append(l_np[b, h, rows]); ro.append(a); rl.append(c)
    check(np.concatenate(go), np.concatenate(gl), np.concatenate(ro), np.concatenate(rl), w.name)
