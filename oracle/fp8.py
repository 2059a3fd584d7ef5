"""CPU oracle of the FP8 (E4M3) attention forward with per-tile scales.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU
baseline may import this module.  The product path never calls it and shares no code with it.

Sources, by page title and section:

* the E4M3 format -- 1 sign bit, 4 exponent bits, 3 mantissa bits, largest magnitude 448 -- and
  its use for forward activations with fine-grained per-tile scaling: "CS336 Lecture 5" notes,
  section 3.1 (format table and the paragraph on the two FP8 variants);
* FP8 as a FlashAttention-3 feature: the same notes, section 6.3.

Readings (the pages give the format and the idea of per-tile scales, not an algorithm):

* E4M3 is the variant without infinities: exponent bias 7, normal values 2^(e-7) (1 + m/8) for
  e = 1..15 except e = 15, m = 7 (NaN), subnormals 2^-6 (m/8); so the largest finite value is
  2^8 x 1.75 = 448, as the pages state, and the smallest positive value is 2^-9.
* a tile is 128 consecutive rows of one head (all d columns), matching the kernel's tiles; its
  scale is amax / 448 in fp32 (1 when the tile is all zero), so the largest magnitude maps to 448;
* codes are round-to-nearest-even of x / scale, saturating at +-448; the sign bit is the
  input's, so a negative value that rounds to zero is the code of -0 (0x80), as IEEE rounding
  gives.  Because a floating-point division decides an integer code, the decision is taken in
  the kernel's precision: fp32 ``amax / 448`` and fp32 ``x / scale`` (IEEE, correctly rounded),
  then the exact RNE of that fp32 value to E4M3;
* the attention of the FP8 path is the plain definition applied to the dequantized inputs
  ``code value x tile scale`` (so the oracle's output carries the inputs' quantization and the
  comparison measures what the kernel adds: the E4M3 rounding of the probabilities and fp32
  accumulation).

V is quantized like Q and K (per 128-row tile of the head); the kernel stores its codes
transposed, [d][N rounded up to 128], which does not change the values.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_dense, bf16_bits_to_f64

E4M3_MAX = 448.0
TILE = 128


def e4m3_value(code) -> np.ndarray:
    """float64 value of E4M3 codes (uint8); NaN for the two NaN codes (0x7F, 0xFF)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# every finite non-negative E4M3 value, ascending, with its code
_POS_CODES = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7E
_POS_VALUES = e4m3_value(_POS_CODES)


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even of float values to E4M3 codes, saturating at +-448 (no NaN input)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # index of the largest representable value <= a, and the next one up
    lo = np.searchsorted(_POS_VALUES, a, side="right") - 1
    hi = np.minimum(lo + 1, len(_POS_VALUES) - 1)
    vlo, vhi = _POS_VALUES[lo], _POS_VALUES[hi]
    dlo, dhi = a - vlo, vhi - a
    even_lo = (_POS_CODES[lo] & 1) == 0
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ~even_lo & (hi != lo))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    # the sign bit follows the input's sign, also when the magnitude rounds to zero (-0)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def quantize_tiles(x_bits: np.ndarray):
    """Per-tile E4M3 quantization of a dense bf16 tensor [B, H, N, d] (uint16 bit patterns).

    Returns (codes uint8 [B, H, N, d], scales float32 [B, H, ceil(N/128)]).  For every tile of
    128 rows of a head: scale = fp32(amax) / 448 in fp32 (1 if amax = 0); code = RNE_E4M3(fp32(x)
    / scale) with the division in fp32.
    """
    x32 = bf16_bits_to_f64(x_bits).astype(np.float32)
    B, H, N, d = x32.shape
    nt = -(-N // TILE)
    codes = np.empty((B, H, N, d), dtype=np.uint8)
    scales = np.empty((B, H, nt), dtype=np.float32)
    for t in range(nt):
        blk = x32[:, :, t * TILE:(t + 1) * TILE, :]
        amax = np.abs(blk).max(axis=(2, 3))
        sc = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        scales[:, :, t] = sc
        v = (blk / sc[:, :, None, None]).astype(np.float32)   # fp32 IEEE division
        codes[:, :, t * TILE:(t + 1) * TILE, :] = e4m3_encode(v.astype(np.float64))
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 values ``code value x tile scale`` of a [B, H, N, d] code tensor."""
    v = e4m3_value(codes)
    s = np.repeat(scales.astype(np.float64), TILE, axis=2)[:, :, :codes.shape[2]]
    return v * s[..., None]


def attention_fp8_dense(qc, sq, kc, sk, vc, sv, causal: bool, scale: float, heads=None):
    """The FP8 path's reference: exact attention (float64) of the dequantized inputs.
    Codes [B, H, N, d] (V in the same layout as Q and K), scales [B, H, ceil(N/128)]."""
    return attention_dense(dequantize(qc, sq), dequantize(kc, sk), dequantize(vc, sv), causal,
                           scale, heads=heads)
