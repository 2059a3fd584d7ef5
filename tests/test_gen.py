"""The seeded generator: published test vectors, determinism, bf16 rounding, moments."""
import math

import numpy as np
import pytest
import torch

from gen import configs, inputs


def test_splitmix64_published_vectors():
    # reference outputs of splitmix64 for seeds 0 and 1234567 (Vigna's splitmix64.c)
    assert [int(x) for x in inputs.splitmix64(0, 0, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [int(x) for x in inputs.splitmix64(1234567, 0, 5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_counter_based_chunking():
    full = inputs.splitmix64(99, 0, 1000)
    assert np.array_equal(full[500:], inputs.splitmix64(99, 500, 500))
    n = inputs._CHUNK + 1001  # crosses a chunk boundary with an odd tail
    a = inputs.normal_f64(5, n)
    assert np.array_equal(a[:2000], inputs.normal_f64(5, 2000))


def test_box_muller_pairs():
    u = inputs.uniform01(17, 0, 200)
    z = inputs.normal_f64(17, 200)
    r2 = z[0::2] ** 2 + z[1::2] ** 2
    assert np.allclose(r2, -2.0 * np.log(u[0::2]), rtol=1e-12)
    assert np.all((u > 0) & (u <= 1))


def test_normal_moments():
    z = inputs.normal_f64(2026, 1 << 20, sigma=2.0)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 2.0) < 0.01
    assert abs(np.mean((z / 2.0) ** 4) - 3.0) < 0.05  # Gaussian kurtosis


def test_bf16_rne_ties_and_torch():
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 1.0 + 2.0 ** -8 + 2.0 ** -40,
                  0.0, -0.0, 3.0, 1e-3])
    bits = inputs.f64_to_bf16_bits(x)
    assert bits[0] == 0x3F80          # tie -> even (1.0)
    assert bits[1] == 0x3F82          # tie -> even (1 + 2^-6)
    assert bits[2] == 0xBF80
    assert bits[3] == 0x3F81          # just above the tie rounds up (no double rounding)
    assert bits[4] == 0 and bits[5] == 0x8000
    # float32-representable values: agree with torch's round-to-nearest-even conversion
    f = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 3
    mine = inputs.f64_to_bf16_bits(f.astype(np.float64))
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_rounding_error_bound():
    x = inputs.normal_f64(3, 10000)
    b = inputs.f64_to_bf16_bits(x)
    y = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.abs(y - x) <= np.abs(x) * 2.0 ** -8 + 1e-300)


def test_workloads():
    w = configs.WORKLOADS
    assert (w[3].B, w[3].H, w[3].N, w[3].d, w[3].causal) == (2, 32, 4096, 128, False)
    assert w[4].sigma_qk == 2.0 and w[4].causal
    L = w[5].lengths()
    assert len(L) == 16 and L.min() >= 128 and L.max() <= 4096
    cu = w[5].cu_seqlens()
    assert cu.dtype == np.int32 and cu[0] == 0 and np.array_equal(np.diff(cu), L)
    assert np.array_equal(w[5].lengths(), L)  # deterministic
    q, k, v, cu1 = w[1].make()
    assert q.shape == (1, 2, 256, 64) and q.dtype == np.uint16 and cu1 is None
    q2, _, _, _ = w[1].make()
    assert np.array_equal(q, q2) and not np.array_equal(q, k)
    assert math.isclose(w[1].scale, 0.125)
