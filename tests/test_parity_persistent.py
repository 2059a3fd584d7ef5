"""GPU parity of the head-dim-128 forward when each persistent cluster runs several work units.

The head-dim-128 forward keeps one cluster of two CTAs per pair of SMs resident and walks the
work units (256 query rows x key slice) in rounds, so state carried from one unit to the next
(the Q double buffer, ring and buffer phases, the reference maximum and row sums, the O
accumulator) is only exercised when there are more units than clusters.  These shapes have
several rounds each, ragged sequence ends, causal masks, grouped-query heads and split-KV slices,
and every output element is compared with the float64 oracle.
"""
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


@pytest.mark.parametrize("seed,B,H,N,causal", [
    (701, 3, 16, 1000, False),   # 4 pairs x 48 heads = 192 units, ragged last pair
    (702, 3, 16, 1000, True),
    (703, 2, 40, 777, True),     # 4 pairs x 80 heads, last pair half empty
    (704, 1, 64, 300, False),    # 2 pairs x 64 heads, second pair's rank 1 rows all past N
])
def test_many_units_per_cluster(seed, B, H, N, causal):
    w = configs.custom(seed, B, H, N, 128, causal)
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_dense(q, k, v, causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, w.name)


@pytest.mark.parametrize("causal", [False, True])
def test_many_units_grouped_query(causal):
    # 3 pairs x 96 query heads, four query heads per K/V head
    w = configs.custom(711 + int(causal), 2, 48, 640, 128, causal, H_kv=12)
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_gqa_dense(q, k, v, causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, w.name)


@pytest.mark.parametrize("causal,splits", [(False, 3), (True, 5)])
def test_many_units_split_kv(causal, splits):
    # units = pairs x heads x slices, several rounds; causal pairs near the start leave slices
    # empty, units a cluster skips in the middle of its walk
    w = configs.custom(721 + splits, 2, 24, 1500, 128, causal)
    q, k, v, _ = w.make()
    o, lse = attn.attn_fwd_splitkv(to_dev(q), to_dev(k), to_dev(v), causal=causal,
                                   scale=w.scale, num_splits=splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_dense(q, k, v, causal, w.scale)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
          f"{w.name} S={splits}")


def test_repeated_calls_are_bitwise_equal():
    # the walk over units is fixed by the grid; results must not depend on timing
    w = configs.custom(731, 2, 32, 1024, 128, True)
    q, k, v, _ = w.make()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    a = attn.attn_fwd(qd, kd, vd, causal=True, scale=w.scale)
    b = attn.attn_fwd(qd, kd, vd, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)) and torch.equal(a[1], b[1])


# Packed batches on the head-dim-128 kernel: units are (query pair, head, sequence) in bands of
# pair levels; lengths that are not multiples of 32 leave a softmax warp whose rows run past the
# end of its sequence (its rows are written one by one instead of by the TMA store), empty and
# one-row sequences have no units or a single half-empty one.
PACKED_MANY = [1, 0, 700, 1500, 256, 257, 3000, 0, 129, 1024, 511, 2049]  # 41 pairs per head


@pytest.mark.parametrize("causal", [False, True])
def test_many_units_packed(causal):
    H = 8  # 328 units over the resident clusters: several rounds each
    q, k, v, cu = configs.custom_varlen(741 + int(causal), PACKED_MANY, H, 128, causal)
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=cu_t, causal=causal,
                           scale=128 ** -0.5)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_varlen(q, k, v, cu, causal, 128 ** -0.5)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
          f"packed {'causal' if causal else 'full'} H{H}")


def test_many_units_packed_grouped_query():
    lengths = [33, 900, 0, 1, 2100, 383]
    q, k, v, cu = configs.custom_varlen(743, lengths, 24, 128, True, H_kv=6)
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=cu_t, causal=True,
                           scale=128 ** -0.5)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_gqa_varlen(q, k, v, cu, True, 128 ** -0.5)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "packed GQA")


def test_packed_neighbours_not_read_or_written():
    # non-finite Q, K and V in the rows of each sequence's neighbours must not reach its output,
    # and no row of a sequence may be overwritten by the unit of another: the second sequence is
    # computed from finite inputs and compared in full; the first holds NaN everywhere
    lengths = [300, 700, 45]
    q, k, v, cu = configs.custom_varlen(744, lengths, 4, 128, True)
    q, k, v = q.copy(), k.copy(), v.copy()
    for x in (q, k, v):
        x[:, :300] = 0x7FC0
        x[:, 1000:] = 0x7FC0
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=cu_t, causal=True,
                           scale=128 ** -0.5)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_varlen(q[:, 300:1000], k[:, 300:1000], v[:, 300:1000],
                                          np.array([0, 700], dtype=np.int32), True, 128 ** -0.5)
    check(to_f64(o)[:, 300:1000], lse.cpu().numpy()[:, 300:1000].astype(np.float64), o_ref,
          lse_ref, "packed middle sequence between NaN neighbours")


def test_packed_repeated_calls_are_bitwise_equal():
    q, k, v, cu = configs.custom_varlen(745, PACKED_MANY, 4, 128, True)
    cu_t = torch.from_numpy(cu).cuda()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    a = attn.attn_fwd(qd, kd, vd, cu_seqlens=cu_t, causal=True)
    b = attn.attn_fwd(qd, kd, vd, cu_seqlens=cu_t, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("d,causal", [(128, True), (64, True), (64, False)])
def test_packed_many_sequences(d, causal):
    # more sequences than a warp's 32 lanes: the device walk takes the sequences in chunks of 32
    # within every band; lengths from empty to several pairs
    rng = np.random.default_rng(761 + d + int(causal))
    lengths = [int(x) for x in rng.integers(0, 700, size=70)]
    lengths[3] = 0
    lengths[40] = 1
    q, k, v, cu = configs.custom_varlen(761 + d, lengths, 3, d, causal)
    cu_t = torch.from_numpy(cu).cuda()
    o, lse = attn.attn_fwd(to_dev(q), to_dev(k), to_dev(v), cu_seqlens=cu_t, causal=causal,
                           scale=d ** -0.5)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.attention_varlen(q, k, v, cu, causal, d ** -0.5)
    check(to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref,
          f"packed 70 sequences d{d} {'causal' if causal else 'full'}")
