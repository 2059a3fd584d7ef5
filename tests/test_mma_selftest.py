"""The tcgen05 operand encodings of the fused kernel in isolation: one 128-row product of each
shape against a float64 matmul of the same bf16 values."""
import numpy as np
import pytest
import torch

from io_aware_attention_attn_gb300 import attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from io_aware_attention_attn_gb300 import build
    build.build()


@pytest.mark.parametrize("dim", [64, 128])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_single_tile_product(mode, dim):
    g = torch.Generator().manual_seed(7 + dim + mode)
    a_cols = dim if mode == 0 else 128
    a = torch.randn(128, a_cols, generator=g).to(torch.bfloat16)
    b = torch.randn(128, dim, generator=g).to(torch.bfloat16)
    d = attn.selftest_mma(a.cuda(), b.cuda(), mode).cpu().double()
    a64, b64 = a.double(), b.double()
    ref = a64 @ b64.T if mode == 0 else a64 @ b64
    err = (d - ref).abs().max().item()
    assert err < 1e-3 * max(1.0, ref.abs().max().item()), err
