"""GPU parity of the split-KV forward (attn_fwd_splitkv) against the float64 oracle.

Covers explicit slice counts that divide the key tiles evenly and unevenly, counts above the
number of key tiles (lowered), causal problems whose early query pairs leave whole slices empty,
ragged tails, both head dimensions, the library's own choice, and a long sequence checked on
sampled rows."""
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


def run(w, splits):
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd_splitkv(to_dev(q), to_dev(k), to_dev(v), causal=w.causal,
                                   scale=w.scale, num_splits=splits)
    torch.cuda.synchronize()
    return q, k, v, to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("seed,B,H,N,d,causal,splits", [
    (601, 1, 2, 1024, 128, False, 2),   # 8 key tiles, 4 per slice
    (602, 1, 2, 1000, 128, False, 3),   # ragged last tile, uneven slices (3, 3, 2)
    (603, 2, 3, 777, 64, False, 4),
    (604, 1, 2, 1280, 128, True, 4),    # pair 0 covers 2 key tiles: slices 2 and 3 empty
    (605, 1, 4, 1111, 64, True, 3),
    (606, 1, 1, 640, 128, False, 99),   # lowered to the 5 key tiles: one tile per slice
    (607, 1, 2, 2048, 128, True, 0),    # the library's choice
    (608, 1, 1, 129, 64, True, 2),      # two key tiles, second one 1 row long
])
def test_splitkv_dense(seed, B, H, N, d, causal, splits):
    w = configs.custom(seed, B, H, N, d, causal)
    q, k, v, o, lse = run(w, splits)
    o_ref, lse_ref = orc.attention_dense(q, k, v, causal, w.scale)
    check(o, lse, o_ref, lse_ref, f"{w.name} S={splits}")


def test_one_slice_is_the_fused_forward_bitwise():
    # num_splits = 1 takes the plain fused path: same bits as attn_fwd
    w = configs.custom(609, 1, 2, 700, 128, True)
    q, k, v, _ = w.make()
    a = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=w.scale)
    b = attn.attn_fwd_splitkv(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=w.scale,
                              num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)) and torch.equal(a[1], b[1])


def test_splitkv_full_size_sampled():
    w = configs.SPLITKV
    q, k, v, o, lse = run(w, 0)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, w.N - 1],
                                     rng.integers(0, w.N, 80)]))
    go, gl, ro, rl = [], [], [], []
    for b, h in [(bb, hh) for bb in range(w.B) for hh in range(w.H)]:
        a, c = orc.attention_head_rows(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale)
        go.append(o[b, h, rows]); gl.append(lse[b, h, rows]); ro.append(a); rl.append(c)
    check(np.concatenate(go), np.concatenate(gl), np.concatenate(ro), np.concatenate(rl), w.name)


def test_splitkv_causal_long_sampled():
    # a long causal row reaches across all 32 slices; early rows leave most slices empty
    w = configs.custom(610, 1, 1, 8192, 128, True, sigma_qk=2.0)
    q, k, v, o, lse = run(w, 32)
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 4096, w.N - 1],
                                     rng.integers(0, w.N, 60)]))
    a, c = orc.attention_head_rows(q[0, 0], k[0, 0], v[0, 0], rows, True, w.scale)
    check(o[0, 0, rows], lse[0, 0, rows], a, c, w.name)
