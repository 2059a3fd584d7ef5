"""The bench's FLOP / byte / roofline helpers against numbers printed on the pages."""
import json
import math
import os

import numpy as np

from io_aware_attention_attn_gb300 import accounting as acc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "pages_worked_examples.json")))


def test_matmul_n4096_fp32_exact():
    g = GOLD["matmul_fp32_n4096"]
    n = g["n"]
    assert acc.matmul_flops(n, n, n) == g["flops"]
    assert acc.matmul_bytes(n, n, n, g["elem_bytes"]) == g["bytes"]
    ai = acc.matmul_flops(n, n, n) / acc.matmul_bytes(n, n, n, 4)
    assert round(ai) == g["ai_approx"]


def test_matmul_n8192_bf16():
    g = GOLD["matmul_bf16_n8192"]
    n = g["n"]
    f, b = acc.matmul_flops(n, n, n), acc.matmul_bytes(n, n, n, 2)
    assert math.isclose(f, g["flops_approx"], rel_tol=0.01)
    assert math.isclose(b, g["bytes_approx"], rel_tol=0.01)
    assert math.isclose(f / b, g["ai_approx"], rel_tol=0.02)


def test_elementwise_add_roofline():
    g = GOLD["elementwise_add_bf16_n8192"]
    n = g["n"]
    flops, nbytes = n * n, 3 * n * n * 2
    assert math.isclose(flops, g["flops_approx"], rel_tol=0.01)
    assert math.isclose(flops / nbytes, g["ai_exact"], rel_tol=1e-12)
    att = acc.roofline(989e12, g["bandwidth"], flops / nbytes)
    assert math.isclose(att / 1e12, g["attainable_tflops_approx"], rel_tol=0.01)


def test_ridge_points():
    g = GOLD["ridge_h100"]
    assert round(acc.ridge_point(g["peak"], g["bandwidth"])) == g["ridge_approx"]
    g = GOLD["ridge_a100"]
    assert round(acc.ridge_point(g["peak"], g["bandwidth"])) == g["ridge_approx"]
    assert acc.roofline(100.0, 2.0, 10.0) == 20.0 and acc.roofline(100.0, 2.0, 1e3) == 100.0


def test_score_matrix_32mb():
    g = GOLD["score_matrix_n4096_bf16"]
    assert acc.score_matrix_bytes(g["n"], g["elem_bytes"]) == g["bytes"] == 32 * 2 ** 20


def test_layernorm_bytes_and_time():
    g = GOLD["layernorm_8x512x4096_bf16"]
    assert 8 * 512 * 4096 == g["elements"]
    nbytes = 2 * g["elements"] * acc.BF16
    assert math.isclose(nbytes, g["bytes_approx"], rel_tol=0.01)
    assert math.isclose(nbytes / g["bandwidth"], g["seconds_approx"], rel_tol=0.02)


def test_attention_counts():
    # headline workload: 4 B H N^2 d
    assert acc.attention_flops(32, [4096, 4096], 128, False) == 4 * 2 * 32 * 4096 ** 2 * 128
    assert acc.attention_flops(32, [16384], 128, True) == 2 * 32 * 16384 ** 2 * 128
    # exact causal pair count vs the halved headline count
    assert acc.visible_pairs(4, True) == 10 and acc.visible_pairs(4, False) == 16
    assert acc.attention_exact_flops(1, [4], 2, True) == 4 * 10 * 2
    assert acc.attention_ideal_bytes(32, 2 * 4096, 128) == 269484032
    assert acc.attention_ideal_bytes(32, 16384, 128) == 538968064
    # unfused: S fp32 and P bf16 each written and read once: 12 B per score + the minimum
    assert acc.unfused_bytes(2, 32, 4096, 128) == 12 * 64 * 4096 ** 2 + 269484032


def test_bf16_half_ulp():
    assert acc.bf16_half_ulp(1.0) == 2.0 ** -8
    assert acc.bf16_half_ulp(5.0) == 2.0 ** -6
    assert acc.bf16_half_ulp(0.75) == 2.0 ** -9
    x = np.array([1.0, 5.0, -3.0])
    assert np.array_equal(acc.bf16_half_ulp(x), [2.0 ** -8, 2.0 ** -6, 2.0 ** -7])
