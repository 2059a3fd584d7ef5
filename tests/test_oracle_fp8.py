"""Pins for the FP8 (E4M3) oracle: the format the pages give (1 sign, 4 exponent, 3 mantissa bits,
largest magnitude 448), a brute-force nearest-even search over every code, and closed forms of
the per-tile quantization.  Planted mistakes in copies of the encoder must fail."""
import math

import numpy as np
import pytest

from gen import inputs
from oracle import attention as orc
from oracle import fp8


def brute_encode(x: float) -> int:
    """Nearest E4M3 code by search over all 254 finite codes; ties to the even code; saturating."""
    x = max(-448.0, min(448.0, float(x)))
    best, best_d = None, None
    for c in range(256):
        v = float(fp8.e4m3_value(np.uint8(c)))
        if math.isnan(v) or c == 0x80:
            continue
        d = abs(x - v)
        if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    if best == 0 and math.copysign(1.0, x) < 0:
        best = 0x80  # a negative value that rounds to zero keeps its sign
    return best


def pin_failures(encode):
    fails = []

    def check(name, ok):
        if not ok:
            fails.append(name)

    # the pages' format: largest finite magnitude 448, 3 mantissa bits, 4 exponent bits
    vals = fp8.e4m3_value(np.arange(256, dtype=np.uint8))
    finite = vals[np.isfinite(vals)]
    check("max 448", finite.max() == 448.0 and finite.min() == -448.0)
    check("two NaN codes", int(np.isnan(vals).sum()) == 2)
    check("one above 1", float(fp8.e4m3_value(np.uint8(0x39))) == 1.125)
    check("min subnormal", float(fp8.e4m3_value(np.uint8(1))) == 2.0 ** -9)
    check("min normal", float(fp8.e4m3_value(np.uint8(8))) == 2.0 ** -6)
    check("monotone", np.all(np.diff(fp8.e4m3_value(np.arange(0x7F, dtype=np.uint8))) > 0))
    # round trip of every finite non-negative and negative code
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    check("round trip", np.array_equal(encode(fp8.e4m3_value(codes)), codes))
    # ties go to the even code, saturation at 448
    check("tie 1.0625", int(encode(np.array([1.0625]))[0]) == 0x38)
    check("tie 1.1875", int(encode(np.array([1.1875]))[0]) == 0x3A)
    check("tie subnormal", int(encode(np.array([2.0 ** -10]))[0]) == 0 and
          int(encode(np.array([3 * 2.0 ** -10]))[0]) == 2)
    check("saturate", list(encode(np.array([1000.0, -1000.0, 464.0]))) == [0x7E, 0xFE, 0x7E])
    check("negative underflow", list(encode(np.array([-1e-6, -0.0, 0.0]))) == [0x80, 0x80, 0])
    # brute force on values spread over the whole range
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.uniform(-500, 500, 300), rng.normal(0, 1, 300),
                         rng.normal(0, 0.01, 200), np.exp2(rng.uniform(-12, 9, 200))])
    check("brute force", all(int(encode(np.array([x]))[0]) == brute_encode(x) for x in xs))
    return fails


def test_encoder_passes_all_pins():
    assert pin_failures(fp8.e4m3_encode) == []


def _mut_half_up(x):  # ties away from zero
    x = np.asarray(x, float)
    out = fp8.e4m3_encode(x)
    for i, xv in enumerate(x.ravel()):
        lo = fp8.e4m3_encode(np.array([xv]))[0]
        v = float(fp8.e4m3_value(lo))
        nxt = (int(lo) & 0x80) | min((int(lo) & 0x7F) + 1, 0x7E)
        vn = float(fp8.e4m3_value(np.uint8(nxt)))
        if abs(abs(xv) - (abs(v) + abs(vn)) / 2) == 0 and abs(vn) > abs(v):
            out.ravel()[i] = nxt
    return out


def _mut_truncate(x):  # round toward zero
    x = np.asarray(x, float)
    a = np.minimum(np.abs(x), 448.0)
    idx = np.searchsorted(fp8._POS_VALUES, a, side="right") - 1
    c = fp8._POS_CODES[idx]
    return np.where(np.signbit(x), c | 0x80, c).astype(np.uint8)


def _mut_no_saturation(x):  # wraps large values to the NaN code instead of 448
    x = np.asarray(x, float)
    c = fp8.e4m3_encode(x)
    return np.where(np.abs(x) > 448.0, np.uint8(0x7F), c).astype(np.uint8)


def _mut_e5m2_grid(x):  # a 2-bit mantissa grid
    x = np.asarray(x, float)
    return fp8.e4m3_encode(np.round(x * 4) / 4)


@pytest.mark.parametrize("mutant", [_mut_half_up, _mut_truncate, _mut_no_saturation,
                                    _mut_e5m2_grid])
def test_pins_catch_planted_mistake(mutant):
    assert pin_failures(mutant), mutant.__name__


# ------------------------------------------------------------------ per-tile quantization
def test_tile_amax_maps_to_448_and_error_bound():
    x = inputs.bf16_normal(61, (2, 3, 300, 64), 1.7)
    codes, scales = fp8.quantize_tiles(x)
    xf = orc.bf16_bits_to_f64(x)
    assert scales.shape == (2, 3, 3)
    for b in range(2):
        for h in range(3):
            for t in range(3):
                blk = xf[b, h, t * 128:(t + 1) * 128]
                amax = np.abs(blk).max()
                assert scales[b, h, t] == np.float32(np.float32(amax) / np.float32(448))
                c = codes[b, h, t * 128:(t + 1) * 128]
                i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
                assert c[i] & 0x7F == 0x7E
    deq = fp8.dequantize(codes, scales)
    s = np.repeat(scales.astype(np.float64), 128, axis=2)[:, :, :300, None]
    # relative error <= 2^-4 in the normal range, absolute <= 2^-10 * scale below it
    err = np.abs(deq - xf)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(xf), 2.0 ** -10 * s) * (1 + 1e-6))


def test_zero_tile_and_exact_inputs():
    # an all-zero tile gets scale 1 and zero codes
    z = np.zeros((1, 1, 130, 64), dtype=np.uint16)
    codes, scales = fp8.quantize_tiles(z)
    assert np.all(codes == 0) and np.all(scales == 1.0)
    # values on the E4M3 grid times 2^-6 with a tile amax of 7 = 448 * 2^-6: exact round trip,
    # and the FP8 reference equals the bf16 reference
    rng = np.random.default_rng(5)
    grid = fp8._POS_VALUES[(fp8._POS_VALUES > 0) & (fp8._POS_VALUES <= 448)]

    def exact(shape):
        v = rng.choice(grid, size=shape) * rng.choice([-1.0, 1.0], size=shape)
        v[..., 0, 0] = 448.0
        v = v * 2.0 ** -6
        return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)

    q, k, v = exact((1, 2, 128, 64)), exact((1, 2, 128, 64)), exact((1, 2, 128, 64))
    qc, sq = fp8.quantize_tiles(q)
    kc, sk = fp8.quantize_tiles(k)
    vc, sv = fp8.quantize_tiles(v)
    assert np.all(sq == 2.0 ** -6)
    assert np.array_equal(fp8.dequantize(qc, sq), orc.bf16_bits_to_f64(q))
    o1, l1 = fp8.attention_fp8_dense(qc, sq, kc, sk, vc, sv, True, 0.125)
    o2, l2 = orc.attention_dense(q, k, v, True, 0.125)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
