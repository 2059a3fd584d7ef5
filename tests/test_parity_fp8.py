"""GPU parity of the FP8 (E4M3) path: the quantizer bit for bit against the oracle's codes and
scales, and the FP8 forward against exact attention of the dequantized inputs (tolerance derived
in parity_util)."""
import numpy as np
import pytest
import torch

from gen import configs
from io_aware_attention_attn_gb300 import attn
from oracle import fp8 as ofp8

from parity_util import check_fp8, fp8_bound, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from io_aware_attention_attn_gb300 import build
    build.build()
    yield
    assert attn.last_device_error() == 0


@pytest.mark.parametrize("seed,B,H,N,d,sigma", [
    (801, 1, 2, 256, 128, 1.0), (802, 2, 1, 300, 64, 3.0), (803, 1, 3, 129, 128, 0.01),
    (804, 1, 1, 1, 64, 1.0), (805, 1, 2, 1000, 128, 40.0),
])
def test_quantizer_bit_exact(seed, B, H, N, d, sigma):
    w = configs.custom(seed, B, H, N, d, False, sigma_qk=sigma)
    x, _, _, _ = w.make()
    xd = to_dev(x)
    codes, scales = ofp8.quantize_tiles(x)
    c_gpu, s_gpu = attn.quantize_fp8(xd)
    ct_gpu, st_gpu = attn.quantize_fp8(xd, transpose=True)
    torch.cuda.synchronize()
    assert np.array_equal(s_gpu.cpu().numpy(), scales)
    assert np.array_equal(st_gpu.cpu().numpy(), scales)
    assert np.array_equal(c_gpu.cpu().numpy(), codes)
    T = -(-N // 128)
    ct = ct_gpu.cpu().numpy()
    assert ct.shape == (B, H, d, T * 128)
    assert np.array_equal(ct[..., :N], codes.transpose(0, 1, 3, 2))
    assert np.all(ct[..., N:] == 0)


def test_quantizer_quotient_equals_ieee_division_for_every_bf16_pair():
    # every bf16 x against every tile maximum amax >= |x|: the quantizer's multiply-and-correct
    # quotient must give the code of the correctly rounded division (the oracle's), so the
    # bit-exact cases above hold for every input, not only the sampled ones
    assert attn.selftest_fp8_quotients() == 0


def test_quantizer_zero_tile_and_negative_underflow():
    x = np.zeros((1, 1, 200, 128), dtype=np.uint16)
    x[0, 0, 150, 3] = 0x3F80            # 1.0 in the second tile
    x[0, 0, 151, 4] = 0xB3D6            # about -1e-7: rounds to -0 at scale 1/448
    codes, scales = ofp8.quantize_tiles(x)
    c_gpu, s_gpu = attn.quantize_fp8(to_dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(s_gpu.cpu().numpy(), scales) and scales[0, 0, 0] == 1.0
    assert np.array_equal(c_gpu.cpu().numpy(), codes)
    assert codes[0, 0, 151, 4] == 0x80


def run_fp8(w):
    q, k, v, _ = w.make()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    q8, sq = attn.quantize_fp8(qd)
    k8, sk = attn.quantize_fp8(kd)
    vt8, sv = attn.quantize_fp8(vd, transpose=True)
    o, lse = attn.attn_fwd_fp8(q8, sq, k8, sk, vt8, sv, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    return q, k, v, to_f64(o), lse.cpu().numpy().astype(np.float64)


def reference(q, k, v, causal, scale, heads):
    qc, sq = ofp8.quantize_tiles(q)
    kc, sk = ofp8.quantize_tiles(k)
    vc, sv = ofp8.quantize_tiles(v)
    o_ref, lse_ref = ofp8.attention_fp8_dense(qc, sq, kc, sk, vc, sv, causal, scale, heads=heads)
    Q, K, V = (ofp8.dequantize(c, s) for c, s in ((qc, sq), (kc, sk), (vc, sv)))
    bounds = {(b, h): fp8_bound(Q[b, h], K[b, h], V[b, h], causal, scale) for b, h in heads}
    return o_ref, lse_ref, bounds


@pytest.mark.parametrize("seed,B,H,N,causal,sigma", [
    (811, 1, 2, 256, False, 1.0), (812, 1, 2, 256, True, 1.0),
    (813, 1, 2, 300, True, 1.0),       # ragged last tile
    (814, 2, 1, 129, False, 2.0),
    (815, 1, 2, 1000, True, 2.0),      # peaky rows
    (816, 1, 1, 640, False, 0.25),     # flat rows
])
def test_fp8_forward(seed, B, H, N, causal, sigma):
    w = configs.custom(seed, B, H, N, 128, causal, sigma_qk=sigma)
    q, k, v, o, lse = run_fp8(w)
    heads = [(b, h) for b in range(B) for h in range(H)]
    o_ref, lse_ref, bounds = reference(q, k, v, causal, w.scale, heads)
    for b, h in heads:
        check_fp8(o[b, h], lse[b, h], o_ref[b, h], lse_ref[b, h], bounds[(b, h)],
                  f"{w.name} ({b},{h})")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_full_size_sampled_heads(causal):
    w = configs.custom(817, 2, 32, 4096, 128, causal)
    q, k, v, o, lse = run_fp8(w)
    heads = [(0, 0), (1, 30)]
    o_ref, lse_ref, bounds = reference(q, k, v, causal, w.scale, heads)
    for b, h in heads:
        check_fp8(o[b, h], lse[b, h], o_ref[b, h], lse_ref[b, h], bounds[(b, h)],
                  f"{w.name} ({b},{h})")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_many_units_per_cluster(causal):
    # 3 query pairs x 96 heads = 288 units of 256 query rows, more than the GPU holds at once;
    # the last pair of every head is ragged (its second tile ends at row 700).  Every head is
    # compared.
    w = configs.custom(818 + int(causal), 2, 48, 700, 128, causal)
    q, k, v, o, lse = run_fp8(w)
    heads = [(b, h) for b in range(2) for h in range(48)]
    o_ref, lse_ref, bounds = reference(q, k, v, causal, w.scale, heads)
    for b, h in heads:
        check_fp8(o[b, h], lse[b, h], o_ref[b, h], lse_ref[b, h], bounds[(b, h)],
                  f"{w.name} ({b},{h})")
