"""Every entry point that takes a caller-provided workspace stays inside the bytes it asked for.

Each call gets exactly the size its ``*_workspace_bytes`` query returns, carved from a larger
buffer whose tail is a canary pattern; after the call (and a synchronize) the canary must be
intact.  The split-KV cases include causal problems whose early query pairs leave whole key
slices empty, the path that writes placeholder statistics instead of partial results.
"""
import numpy as np
import pytest
import torch

from gen import configs
from io_aware_attention_attn_gb300 import attn

from parity_util import to_dev

pytestmark = pytest.mark.gpu

CANARY = 0xA5
TAIL = 1 << 20  # 1 MiB of canary after the workspace


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from io_aware_attention_attn_gb300 import build
    build.build()
    yield
    assert attn.last_device_error() == 0


def guarded(need: int):
    buf = torch.full((need + TAIL,), CANARY, dtype=torch.uint8, device="cuda")
    return buf, buf[:need]


def assert_canary(buf, need):
    torch.cuda.synchronize()
    tail = buf[need:].cpu().numpy()
    bad = np.nonzero(tail != CANARY)[0]
    assert bad.size == 0, f"{bad.size} bytes past the workspace were written (first at +{bad[0]})"


@pytest.mark.parametrize("seed,B,H,N,d,causal,splits", [
    (501, 1, 2, 1000, 128, True, 8),     # early pairs leave slices 2..7 empty
    (502, 1, 3, 700, 64, True, 6),
    (503, 2, 1, 2048, 128, False, 5),
    (504, 1, 1, 4097, 128, True, 32),
])
def test_splitkv_workspace(seed, B, H, N, d, causal, splits):
    w = configs.custom(seed, B, H, N, d, causal)
    q, k, v, _ = w.make()
    need = attn.splitkv_workspace_bytes(B, H, N, d, splits)
    assert need > 0
    buf, ws = guarded(need)
    attn.attn_fwd_splitkv(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=w.scale,
                          num_splits=splits, workspace=ws)
    assert_canary(buf, need)


@pytest.mark.parametrize("seed,B,H,N,d,causal", [
    (511, 1, 2, 300, 128, True), (512, 2, 2, 129, 64, False),
])
def test_backward_workspace(seed, B, H, N, d, causal):
    w = configs.custom(seed, B, H, N, d, causal)
    q, k, v, _ = w.make()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, scale=w.scale)
    dout = to_dev(w.make_dout())
    need = attn.bwd_workspace_bytes(B, H, N, d)
    buf, ws = guarded(need)
    attn.attn_bwd(qd, kd, vd, o, lse, dout, causal=causal, scale=w.scale, workspace=ws)
    assert_canary(buf, need)


def test_backward_varlen_workspace():
    lengths = [5, 130, 257]
    T, H, d = sum(lengths), 2, 128
    rng = np.random.default_rng(7)
    q, k, v, dout = (torch.from_numpy(rng.standard_normal((T, H, d)).astype(np.float32))
                     .to(torch.bfloat16).cuda().transpose(0, 1).contiguous() for _ in range(4))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32,
                      device="cuda")
    o, lse = attn.attn_fwd(q, k, v, cu_seqlens=cu, causal=True)
    need = int(attn.lib().attn_bwd_varlen_workspace_bytes(len(lengths), H, T, d))
    buf, ws = guarded(need)
    attn.attn_bwd(q, k, v, o, lse, dout, cu_seqlens=cu, causal=True, workspace=ws)
    assert_canary(buf, need)


def test_unfused_workspace():
    w = configs.custom(521, 1, 2, 300, 128, True)
    q, k, v, _ = w.make()
    need = attn.unfused_workspace_bytes(1, 2, 300, 128)
    buf, ws = guarded(need)
    attn.attn_fwd_unfused(to_dev(q), to_dev(k), to_dev(v), causal=True, scale=w.scale,
                          workspace=ws)
    assert_canary(buf, need)
