"""Failure detection without a GPU fault: a bounded pipeline wait that runs out reports a status
word, the kernel returns, and the context stays usable."""
import numpy as np
import pytest
import torch

from gen import configs
from io_aware_attention_attn_gb300 import attn
from oracle import attention as orc

from parity_util import check, to_dev, to_f64


def test_decode_status():
    assert attn.decode_status(1 | (6 << 8) | (1 << 16)) == {"kind": 1, "role": 6, "site": 1}
    assert attn.decode_status(0) == {"kind": 0, "role": 0, "site": 0}


@pytest.mark.gpu
def test_wait_timeout_reports_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from io_aware_attention_attn_gb300 import build
    build.build()
    assert attn.last_device_error() == 0
    attn.selftest_wait_timeout()
    code = attn.last_device_error()          # synchronises: the wait gives up after ~1 s
    assert attn.decode_status(code) == {"kind": 1, "role": 6, "site": 1}
    assert attn.last_device_error() == 0      # reading clears it
    w = configs.custom(300, 1, 2, 300, 128, True)
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=w.scale)
    o_ref, lse_ref = orc.attention_dense(q, k, v, True, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "after timeout")
    assert attn.last_device_error() == 0


@pytest.mark.gpu
def test_bad_cu_seqlens_is_reported_not_faulted():
    # a decreasing offset: the kernel clamps every offset into [0, N], computes, and reports kind 2
    import math
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from io_aware_attention_attn_gb300 import build
    build.build()
    q, k, v, _ = configs.custom_varlen(950, [100, 200], 2, 64, True)
    bad = torch.tensor([0, 150, 100, 300], dtype=torch.int32, device="cuda")
    assert attn.last_device_error() == 0
    attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=bad, causal=True,
                  scale=1 / math.sqrt(64))
    code = attn.last_device_error()
    assert attn.decode_status(code)["kind"] == 2, code
    assert attn.last_device_error() == 0  # cleared by the read
    good = torch.tensor([0, 100, 300], dtype=torch.int32, device="cuda")
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=good, causal=True,
                           scale=1 / math.sqrt(64))
    assert attn.last_device_error() == 0 and torch.isfinite(lse).all()
