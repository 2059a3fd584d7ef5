"""GPU parity of the unfused three-kernel comparison path against the float64 oracle, and its
agreement with the fused path."""
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


CASES = [
    (201, 1, 2, 1, 64, False), (202, 1, 1, 1, 128, True),
    (203, 2, 2, 127, 128, True), (204, 2, 2, 129, 64, False),
    (205, 1, 3, 300, 128, False), (206, 1, 3, 300, 64, True),
    (207, 1, 2, 1000, 128, True), (208, 2, 1, 517, 128, False),
]


@pytest.mark.parametrize("seed,B,H,N,d,causal", CASES)
def test_unfused_full(seed, B, H, N, d, causal):
    w = configs.custom(seed, B, H, N, d, causal)
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd_unfused(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_dense(q, k, v, causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "unfused " + w.name)


def test_unfused_peaky():
    w = configs.custom(209, 1, 2, 1500, 128, True, sigma_qk=2.0)
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd_unfused(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=w.scale)
    o_ref, lse_ref = orc.attention_dense(q, k, v, True, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "unfused peaky")


@pytest.mark.parametrize("index", [1, 2, 3])
def test_unfused_matches_fused_full_size(index):
    w = configs.WORKLOADS[index]
    q, k, v, _ = w.make()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    of, lf = attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    ou, lu = attn.attn_fwd_unfused(qd, kd, vd, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    # both paths against the oracle on sampled rows of two heads
    rng = np.random.default_rng(index)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.integers(0, w.N, 40)]))
    for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
        ro, rl = orc.attention_head_rows(q[b, h], k[b, h], v[b, h], rows, w.causal, w.scale)
        for o, l, name in ((of, lf, "fused"), (ou, lu, "unfused")):
            check(to_f64(o[b, h])[rows], l[b, h].cpu().numpy().astype(np.float64)[rows], ro, rl,
                  f"{name} {w.name} head {b},{h}")
    # and against each other everywhere (both carry only bf16-rounding differences)
    diff = (of.float() - ou.float()).abs()
    assert diff.max().item() <= 2e-2 and diff.mean().item() <= 1e-3
    assert (lf - lu).abs().max().item() <= 1e-3


def test_unfused_rejects_small_workspace():
    w = configs.custom(210, 1, 1, 256, 64, False)
    q, k, v, _ = w.make()
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_unfused(to_dev(q), to_dev(k), to_dev(v), workspace=ws)
    assert e.value.code == -8
