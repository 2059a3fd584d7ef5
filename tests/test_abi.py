"""The C-ABI library on the host: it builds, loads, exports what the header declares, and its
argument validation returns the documented codes before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from io_aware_attention_attn_gb300 import attn, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "attn_gb300.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_functions()
    assert set(names) == set(attn.SIGNATURES), names
    for must in ("attn_fwd", "attn_fwd_unfused", "attn_fwd_unfused_workspace_bytes",
                 "attn_get_last_device_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.attn_version() >= 100


def test_only_the_api_is_exported(lib):
    out = os.popen(f"nm -D --defined-only {attn.LIB_PATH}").read().split("\n")
    exported = {l.split()[-1] for l in out if re.search(r" [TD] ", l)}
    assert {n for n in exported if not n.startswith("_")} <= set(attn.SIGNATURES) | {"_init", "_fini"}


ALIGNED = 0x10000  # fake, never dereferenced: validation fails before any CUDA call


def call(lib, q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=ALIGNED, cu=None, B=1, H=1, N=128,
         d=128, causal=0, scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, cu, B, H, N, d, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), -3), (dict(H=-2), -3), (dict(N=-5), -3),
    (dict(d=96), -2), (dict(d=256), -2), (dict(d=0), -2),
    (dict(q=None), -1), (dict(lse=None), -1), (dict(o=None), -1),
    (dict(k=ALIGNED + 8), -4), (dict(o=ALIGNED + 2), -4), (dict(lse=ALIGNED + 4), -4),
    (dict(cu=ALIGNED + 2), -4),
    (dict(scale=0.0), -7), (dict(scale=-1.0), -7), (dict(scale=float("inf")), -7),
    (dict(scale=float("nan")), -7),
    (dict(cu=ALIGNED, B=0, N=5), -3),
    (dict(N=(1 << 31) - 1, B=1 << 10, H=1 << 10), -3),
])
def test_validation_codes(lib, kw, code):
    assert call(lib, **kw) == code


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0), dict(N=0, q=None, o=None),
                                dict(cu=ALIGNED, N=0, B=3)])
def test_empty_problems_are_noops(lib, kw):
    assert call(lib, **kw) == 0


def test_unfused_workspace_bytes(lib):
    assert lib.attn_fwd_unfused_workspace_bytes(2, 32, 4096, 128) == 64 * 4096 * (4096 * 6 + 4)
    assert lib.attn_fwd_unfused_workspace_bytes(1, 1, 100, 64) == 51200 + 25600 + 512
    assert lib.attn_fwd_unfused_workspace_bytes(1, 1, 100, 96) == 0
    assert lib.attn_fwd_unfused_workspace_bytes(0, 1, 100, 64) == 0


def test_unfused_validation(lib):
    f = lib.attn_fwd_unfused
    assert f(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, None, 1, 1, 128, 64, 0, 0.125,
             None, 1 << 20, None) == -8
    assert f(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, None, 1, 1, 128, 64, 0, 0.125,
             ALIGNED, 100, None) == -8
    assert f(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, None, 1, 1, 128, 64, 0, 0.125,
             ALIGNED + 16, 1 << 20, None) == -8
    assert f(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 1, 1, 128, 64, 0, 0.125,
             ALIGNED, 1 << 20, None) == -9
    assert f(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, None, 1, 1, 128, 80, 0, 0.125,
             ALIGNED, 1 << 20, None) == -2


def test_selftest_validation(lib):
    assert lib.attn_selftest_mma(None, ALIGNED, ALIGNED, 0, 128, None) == -1
    assert lib.attn_selftest_mma(ALIGNED, ALIGNED, ALIGNED, 0, 32, None) == -2
    assert lib.attn_selftest_mma(ALIGNED, ALIGNED, ALIGNED, 7, 64, None) == -9
    assert lib.attn_selftest_mma(ALIGNED, ALIGNED, ALIGNED, -1, 64, None) == -9
    assert lib.attn_selftest_fp8_quotients(None, None) == -1
    assert lib.attn_selftest_fp8_quotients(ALIGNED + 4, None) == -4


def test_gqa_validation(lib):
    f = lib.attn_fwd_gqa
    A = ALIGNED
    assert f(A, A, A, A, A, None, 1, 8, 3, 128, 128, 0, 0.1, None) == -3   # 3 does not divide 8
    assert f(A, A, A, A, A, None, 1, 8, 0, 128, 128, 0, 0.1, None) == -3
    assert f(A, A, A, A, A, None, 1, 8, -1, 128, 128, 0, 0.1, None) == -3
    assert f(A, A, A, A, A, None, 1, 8, 2, 128, 96, 0, 0.1, None) == -2
    assert f(A, A, A, A, A, None, 1, 0, 0, 128, 128, 0, 0.1, None) == 0    # nothing to do


def test_splitkv_workspace_bytes(lib):
    f = lib.attn_fwd_splitkv_workspace_bytes
    # head dim 128: a unit is a cluster on two SMs, 76 at once.  B=1, H=1, N=8192: 32 query pairs
    # over 64 key tiles; cost(1) = 66, cost(2) = 1 wave x 34, cost(3) = 2 waves x 24 -> 2 slices
    rows = 8192
    assert f(1, 1, 8192, 128, 0) == 2 * rows * 128 * 4 + 2 * 2 * rows * 4
    # B=1, H=2, N=8192 already fills 128 SMs in one slice: cost(1) = 66 < cost(2) = 2 x 34
    assert f(1, 2, 8192, 128, 0) == 0
    # head dim 64: one CTA per unit, 152 at once.  B=1, H=1, N=16384: 64 pairs, 128 key tiles;
    # 7 slices (3 waves x 21) beat 2 (1 x 66)
    rows = 16384
    assert f(1, 1, 16384, 64, 0) == 7 * rows * 64 * 4 + 2 * 7 * rows * 4
    assert f(1, 2, 8192, 128, 5) == 5 * 2 * 8192 * 128 * 4 + 2 * 5 * 2 * 8192 * 4
    # an explicit count above the 8 key tiles of N=1000 is lowered to 8 (regions 256-aligned)
    rows = 1000
    o_bytes = -(-8 * rows * 64 * 4 // 256) * 256
    assert f(1, 1, 1000, 64, 100) == o_bytes + -(-2 * 8 * rows * 4 // 256) * 256
    assert f(1, 1, 1 << 20, 64, 1000) == 32 * (1 << 20) * 64 * 4 + 2 * 32 * (1 << 20) * 4
    assert f(1, 1, 8192, 128, 1) == 0        # one slice: plain fused forward, no workspace
    assert f(2, 32, 4096, 128, 0) == 0       # 1024 pairs already fill the GPU
    assert f(1, 1, 100, 64, 4) == 0          # a single key tile cannot be split
    assert f(1, 1, 1000, 96, 2) == 0
    assert f(0, 1, 1000, 64, 2) == 0


def test_splitkv_slices(lib):
    f = lib.attn_fwd_splitkv_slices
    # both head dims run on clusters of two SMs (76 at once): the same slice model
    assert f(1, 1, 8192, 128, 0) == 2 and f(1, 2, 8192, 128, 0) == 1
    assert f(1, 2, 8192, 64, 0) == 1 and f(1, 1, 16384, 64, 0) == 7
    assert f(2, 32, 4096, 128, 0) == 1
    assert f(1, 1, 1000, 64, 0) == 8 and f(1, 1, 1000, 64, 3) == 3 and f(1, 1, 1000, 64, 50) == 8
    assert f(1, 1, 1 << 20, 64, 1000) == 32 and f(1, 1, 100, 64, 0) == 1
    assert f(0, 1, 100, 64, 0) == 0 and f(1, 1, -5, 64, 0) == 0 and f(1, 1, 1000, 96, 0) == 0


def test_splitkv_validation(lib):
    f = lib.attn_fwd_splitkv
    A = ALIGNED
    big = 1 << 30
    assert f(A, A, A, A, A, 1, 2, 8192, 128, 0, 0.1, 4, None, big, None) == -8
    assert f(A, A, A, A, A, 1, 2, 8192, 128, 0, 0.1, 4, A + 16, big, None) == -8
    assert f(A, A, A, A, A, 1, 2, 8192, 128, 0, 0.1, 4, A, 1 << 20, None) == -8
    assert f(A, A, A, A, A, 1, 2, 8192, 96, 0, 0.1, 4, A, big, None) == -2
    assert f(A, A, A, A, A, 1, 2, 8192, 128, 0, 0.0, 4, A, big, None) == -7
    assert f(A + 2, A, A, A, A, 1, 2, 8192, 128, 0, 0.1, 4, A, big, None) == -4
    assert f(None, A, A, A, A, 1, 2, 8192, 128, 0, 0.1, 4, A, big, None) == -1
    assert f(A, A, A, A, A, -1, 2, 8192, 128, 0, 0.1, 4, A, big, None) == -3
    assert f(A, A, A, A, A, 0, 2, 8192, 128, 0, 0.1, 4, None, 0, None) == 0


def test_bwd_workspace_bytes(lib):
    f = lib.attn_bwd_workspace_bytes
    assert f(2, 32, 4096, 128) == 2 * 2 * 32 * 4096 * 4
    assert f(1, 1, 100, 64) == 2 * 512           # 128 padded rows x 4 bytes, per plane
    assert f(1, 3, 129, 64) == 2 * 3 * 256 * 4
    assert f(1, 1, 100, 96) == 0 and f(0, 1, 100, 64) == 0 and f(1, 1, 0, 64) == 0


def test_bwd_validation(lib):
    f = lib.attn_bwd
    A = ALIGNED
    big = 1 << 30

    def call_bwd(**kw):
        a = dict(q=A, k=A, v=A, o=A, lse=A, do=A, dq=A, dk=A, dv=A, B=1, H=2, N=300, d=128,
                 causal=1, scale=0.1, ws=A, ws_bytes=big)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"],
                 a["B"], a["H"], a["N"], a["d"], a["causal"], a["scale"], a["ws"], a["ws_bytes"],
                 None)

    assert call_bwd(d=96) == -2
    assert call_bwd(B=-1) == -3
    assert call_bwd(do=None) == -1 and call_bwd(dk=None) == -1 and call_bwd(o=None) == -1
    assert call_bwd(dv=A + 4) == -4 and call_bwd(do=A + 2) == -4 and call_bwd(lse=A + 4) == -4
    assert call_bwd(scale=float("nan")) == -7
    assert call_bwd(ws=None) == -8 and call_bwd(ws=A + 16) == -8 and call_bwd(ws_bytes=100) == -8
    assert call_bwd(N=0) == 0 and call_bwd(H=0, dq=None) == 0


def test_fp8_validation(lib):
    A = ALIGNED
    q = lib.attn_quantize_fp8
    assert q(A, A, A, 1, 2, 300, 96, 0, None) == -2
    assert q(None, A, A, 1, 2, 300, 128, 0, None) == -1
    assert q(A, A + 8, A, 1, 2, 300, 128, 1, None) == -4
    assert q(A, A, A + 2, 1, 2, 300, 128, 1, None) == -4
    assert q(A, A, A, -1, 2, 300, 128, 0, None) == -3
    assert q(A, A, A, 1, 2, 0, 128, 0, None) == 0
    f = lib.attn_fwd_fp8
    assert f(A, A, A, A, A, A, A, A, 1, 2, 300, 64, 0, 0.1, None) == -2    # head dim 128 only
    assert f(A, A, None, A, A, A, A, A, 1, 2, 300, 128, 0, 0.1, None) == -1
    assert f(A, A, A, A, A + 8, A, A, A, 1, 2, 300, 128, 0, 0.1, None) == -4
    assert f(A, A + 2, A, A, A, A, A, A, 1, 2, 300, 128, 0, 0.1, None) == -4
    assert f(A, A, A, A, A, A, A, A, 1, 2, 300, 128, 0, -1.0, None) == -7
    assert f(A, A, A, A, A, A, A, A, 1, 0, 300, 128, 0, 0.1, None) == 0


def test_bwd_gqa_validation(lib):
    f = lib.attn_bwd_gqa
    A = ALIGNED

    def c(H, H_kv, d=128, N=300):
        return f(A, A, A, A, A, A, A, A, A, 1, H, H_kv, N, d, 1, 0.1, A, 1 << 30, None)

    assert c(8, 3) == -3 and c(8, 0) == -3 and c(8, -2) == -3
    assert c(8, 2, d=96) == -2
    assert c(0, 0) == 0 and c(8, 2, N=0) == 0


def test_bwd_varlen_validation(lib):
    f = lib.attn_bwd_varlen
    A = ALIGNED
    big = 1 << 30

    def c(cu=A, B=3, H=4, H_kv=2, T=300, d=128, ws=A, nb=big):
        return f(A, A, A, A, A, A, A, A, A, cu, B, H, H_kv, T, d, 1, 0.1, ws, nb, None)

    assert c(cu=None) == -1
    assert c(cu=A + 2) == -4
    assert c(H_kv=3) == -3
    assert c(d=96) == -2
    assert c(ws=None) == -8 and c(nb=100) == -8
    assert c(B=0, T=5) == -3          # rows but no sequences
    assert c(T=0) == 0
    w = lib.attn_bwd_varlen_workspace_bytes
    assert w(3, 4, 300, 128) == 2 * 4 * 128 * (3 + 3) * 4
    assert w(1, 1, 1, 64) == 2 * 1024 and w(0, 1, 10, 64) == 0 and w(1, 1, 10, 96) == 0
