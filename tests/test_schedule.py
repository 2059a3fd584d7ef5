"""Properties of the persistent forward's work distribution, checked on the host.

The head-dim-128 forward runs G clusters that each walk the work units c, 2G-1-c, 2G+c, 4G-1-c,
... (rounds of G units, alternately forward and backward), and splits a query pair's key tiles
into slices of ceil(n / S) tiles.  These tests restate those two formulas as the kernel states
them and check what the kernel relies on: every unit is taken by exactly one cluster, each
cluster's units come in increasing rounds, the slices of a pair cover its key tiles exactly once,
and a causal pair's key range reaches the diagonal of its last row.  The slice-count choice made
by the library is checked through the C ABI (no GPU needed).

The backward's tile passes are restated the same way: the warp scan that maps a packed batch's
tile slot to (sequence, tile) must reach every tile of every sequence exactly once within the
slots the host sizes the workspace for, with the slot equal to its row block in the -lse2 / -D
planes; the dense slot orders must cover every (head, tile) once, heaviest first when causal.
"""
import pytest

from io_aware_attention_attn_gb300 import attn

BM = BN = 128


def next_unit(k, c, G):
    return k * G + ((G - 1 - c) if (k & 1) else c)


def walk(c, G, n_units):
    k, u = 0, c
    out = []
    while u < n_units:
        out.append(u)
        k += 1
        u = next_unit(k, c, G)
    return out


@pytest.mark.parametrize("G", [1, 2, 3, 7, 64, 75, 76])
@pytest.mark.parametrize("n_units", [1, 5, 75, 76, 77, 151, 152, 1024, 1500])
def test_every_unit_exactly_once(G, n_units):
    seen = {}
    for c in range(G):
        units = walk(c, G, n_units)
        assert units == sorted(units)  # rounds in order: Q buffers and phases advance monotonically
        for u in units:
            assert u not in seen, (u, c, seen.get(u))
            seen[u] = c
    assert sorted(seen) == list(range(n_units))
    # balance: no cluster takes more than one unit beyond another
    counts = [len(walk(c, G, n_units)) for c in range(G)]
    assert max(counts) - min(counts) <= 1


def key_slices(n_full, n_splits):
    chunk = (n_full + n_splits - 1) // n_splits
    out = []
    for split in range(n_splits):
        kb = split * chunk
        n = max(0, min(kb + chunk, n_full) - kb)
        out.append((kb, n))
    return out


@pytest.mark.parametrize("n_full", [1, 2, 3, 7, 8, 31, 32, 64, 128])
@pytest.mark.parametrize("n_splits", [1, 2, 3, 5, 8, 16])
def test_key_slices_cover_once(n_full, n_splits):
    covered = []
    for kb, n in key_slices(n_full, n_splits):
        covered.extend(range(kb, kb + n))
    assert covered == list(range(n_full))


@pytest.mark.parametrize("N", [1, 127, 128, 129, 255, 256, 300, 1000, 4096])
def test_causal_pair_reaches_its_diagonal(N):
    n_keytiles = (N + BN - 1) // BN
    n_pairs = (N + 2 * BM - 1) // (2 * BM)
    for pt in range(n_pairs):
        n_full = min(n_keytiles, 2 * pt + 2)
        last_row = min(N, (2 * pt + 2) * BM) - 1
        # the key tiles cover every key <= the pair's last row, and stay inside the sequence
        assert n_full * BN > last_row
        assert (n_full - 1) * BN < N


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 8192, 128), (1, 1, 256, 64), (2, 32, 4096, 128),
                                     (1, 4, 16384, 64), (1, 1, 100, 128)])
def test_slice_count_is_within_key_tiles(B, H, N, d):
    s = attn.splitkv_slices(B, H, N, d, 0)
    key_tiles = (N + BN - 1) // BN
    assert 1 <= s <= max(1, key_tiles)
    # an explicit request is clamped to the key tiles, never raised
    assert attn.splitkv_slices(B, H, N, d, 3) == min(3, key_tiles)


# ---- packed batches: the band walk of the head-dim-128 forward, restated with its warp chunks
BAND = 4


def seq_pairs(cu, N):
    out = []
    for s in range(len(cu) - 1):
        a = min(max(cu[s], 0), N)
        b = min(max(cu[s + 1], a), N)
        out.append((a, b - a, (b - a + 2 * BM - 1) // (2 * BM)))
    return out


class PackedWalker:
    """The kernel's incremental walk: current band, units before it, and the 32-sequence chunk
    reached within it (a warp handles 32 sequences per step)."""

    def __init__(self, seqs, H):
        self.seqs, self.H = seqs, H
        max_pairs = max([p for _, _, p in seqs] + [0])
        self.b = (max_pairs + BAND - 1) // BAND - 1
        self.cum, self.cs, self.ccum = 0, 0, 0
        self.cnt = self.band_count(self.b) if self.b >= 0 else 0

    def band_units(self, s, b):
        if s >= len(self.seqs):
            return 0
        return min(max(self.seqs[s][2] - BAND * b, 0), BAND)

    def band_count(self, b):
        return self.H * sum(self.band_units(s, b) for s in range(len(self.seqs)))

    def at(self, u):
        while u >= self.cum + self.cnt and self.b > 0:
            self.cum += self.cnt
            self.b -= 1
            self.cnt = self.band_count(self.b)
            self.cs = self.ccum = 0
        i = u - self.cum
        while True:
            wgt = [self.H * self.band_units(self.cs + lane, self.b) for lane in range(32)]
            total = sum(wgt)
            if i < self.ccum + total or self.cs + 32 >= len(self.seqs):
                r = i - self.ccum
                incl = 0
                for lane in range(32):
                    if incl <= r < incl + wgt[lane]:
                        s = self.cs + lane
                        m = wgt[lane] // self.H
                        r2 = r - incl
                        return s, r2 // m, BAND * self.b + m - 1 - r2 % m
                    incl += wgt[lane]
                return None
            self.ccum += total
            self.cs += 32


@pytest.mark.parametrize("lengths,H,G", [
    ([1, 0, 700, 1500, 256, 257, 3000, 0, 129, 1024, 511, 2049], 8, 76),
    ([4096] * 3 + [128] * 40 + [0, 1, 2], 3, 76),   # more than 32 sequences: several chunks
    ([300], 1, 76),
    ([0, 0, 5], 2, 7),
    ([257 * k for k in range(70)], 2, 76),
])
def test_packed_walk_takes_every_unit_once(lengths, H, G):
    import numpy as np
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int).tolist()
    seqs = seq_pairs(cu, cu[-1])
    n_units = H * sum(p for _, _, p in seqs)
    expected = {(s, h, pt) for s, (_, _, p) in enumerate(seqs) for h in range(H)
                for pt in range(p)}
    seen = {}
    for c in range(G):
        w = PackedWalker(seqs, H)
        for u in walk(c, G, n_units):
            unit = w.at(u)
            assert unit is not None and unit not in seen, (u, unit)
            seen[unit] = u
    assert set(seen) == expected
    # the order is band by band from the top, then sequence, head, and pair level downwards
    order = sorted(seen, key=lambda x: seen[x])
    keys = [(-(pt // BAND), s, h, -pt) for s, h, pt in order]
    assert keys == sorted(keys)


# ---- dense causal batches: bands of four pair levels from the top, a head's pairs together
DENSE_BAND = 4


def dense_causal_unit(L, n_qt, BH):
    if n_qt <= 2 * DENSE_BAND:  # short sequences: level by level across the heads
        return L % BH, n_qt - 1 - L // BH
    top = (n_qt - 1) // DENSE_BAND
    m_top = n_qt - DENSE_BAND * top
    if L < BH * m_top:
        b, i, m = top, L, m_top
    else:
        L2 = L - BH * m_top
        b, i, m = top - 1 - L2 // (BH * DENSE_BAND), L2 % (BH * DENSE_BAND), DENSE_BAND
    return i // m, DENSE_BAND * b + m - 1 - i % m


@pytest.mark.parametrize("n_qt,BH", [(1, 1), (1, 5), (3, 2), (4, 64), (5, 3), (16, 32), (64, 32),
                                     (9, 7)])
def test_dense_causal_order_takes_every_pair_once_heaviest_band_first(n_qt, BH):
    units = [dense_causal_unit(L, n_qt, BH) for L in range(n_qt * BH)]
    assert sorted(units) == sorted((z, pt) for z in range(BH) for pt in range(n_qt))
    levels = [pt // (DENSE_BAND if n_qt > 2 * DENSE_BAND else 1) for _, pt in units]
    assert levels == sorted(levels, reverse=True)


# ---- backward: tile slots of packed batches, and the dense slot orders of the two tile passes

def bwd_locate_tile(cu, n_seqs, N, slot):
    """The backward kernels' warp scan over cu_seqlens, 32 sequences per step, offsets clamped
    into [0, N]: (start row, length, tile within the sequence, tiles of the earlier sequences);
    tile -1 for a slot past the last tile."""
    import itertools
    remaining, before = slot, 0
    for b0 in range(0, n_seqs, 32):
        spans, nts = [], []
        for lane in range(32):
            s = b0 + lane
            a = e = 0
            if s < n_seqs:
                a = min(max(cu[s], 0), N)
                e = min(max(cu[s + 1], a), N)
            spans.append((a, e))
            nts.append((e - a + BM - 1) // BM)
        incl = list(itertools.accumulate(nts))
        if remaining < incl[-1]:
            src = next(lane for lane in range(32) if incl[lane] - nts[lane] <= remaining < incl[lane])
            a, e = spans[src]
            ex = incl[src] - nts[src]
            return a, e - a, remaining - ex, before + ex
        remaining -= incl[-1]
        before += incl[-1]
    return 0, 0, -1, 0


@pytest.mark.parametrize("cu,N", [
    ([0, 1, 1, 701, 2201, 2457, 2714, 5714, 5714, 5843, 6867, 7378, 9427], 9427),
    ([0] + [128 * (k + 1) for k in range(45)], 45 * 128),   # more than 32 sequences
    ([0, 300], 300),
    ([0, 0, 0, 5], 5),
    ([0, 257, 200, 900, 5000], 900),   # decreasing and past-the-end offsets are clamped
])
def test_bwd_packed_slots_cover_every_tile_once(cu, N):
    n_seqs = len(cu) - 1
    n_slots = (N + BM - 1) // BM + n_seqs   # the host's slots per head (workspace planes)
    expected = set()
    for s in range(n_seqs):
        a = min(max(cu[s], 0), N)
        e = min(max(cu[s + 1], a), N)
        expected |= {(a, t) for t in range((e - a + BM - 1) // BM)}
    assert len(expected) <= n_slots
    seen = set()
    for slot in range(n_slots + 3):
        a, length, tile, base = bwd_locate_tile(cu, n_seqs, N, slot)
        if tile < 0:
            assert slot >= len(expected)
            continue
        assert (a, tile) not in seen
        seen.add((a, tile))
        assert base + tile == slot        # the -lse2 / -D plane rows of the slot: 128 * slot ..
        assert 0 <= tile * BM < length and a + length <= N
    assert seen == expected


def bwd_dkdv_slot(L, B, H_kv, n_tiles, causal):
    if causal:
        return L % (B * H_kv), L // (B * H_kv)
    return L // n_tiles, L % n_tiles


def bwd_dq_slot(L, B, H, n_tiles, causal):
    if causal:
        return L % (B * H), n_tiles - 1 - L // (B * H)
    return L // n_tiles, L % n_tiles


@pytest.mark.parametrize("B,H,H_kv,n_tiles", [(1, 1, 1, 1), (2, 32, 32, 32), (2, 32, 8, 32),
                                               (3, 6, 2, 5), (4, 16, 16, 8)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_dense_slots_cover_every_tile_once(B, H, H_kv, n_tiles, causal):
    kv = [bwd_dkdv_slot(L, B, H_kv, n_tiles, causal) for L in range(B * H_kv * n_tiles)]
    assert sorted(kv) == [(z, j) for z in range(B * H_kv) for j in range(n_tiles)]
    dq = [bwd_dq_slot(L, B, H, n_tiles, causal) for L in range(B * H * n_tiles)]
    assert sorted(dq) == [(z, i) for z in range(B * H) for i in range(n_tiles)]
    if causal:
        # heaviest CTAs first: a key tile j visits n_tiles - j query tiles, a query tile i visits
        # i + 1 key tiles
        kv_work = [n_tiles - j for _, j in kv]
        dq_work = [i + 1 for _, i in dq]
        assert kv_work == sorted(kv_work, reverse=True)
        assert dq_work == sorted(dq_work, reverse=True)
    else:
        # a head's tiles are adjacent, so its streamed tiles are shared in L2
        assert [z for z, _ in kv] == sorted(z for z, _ in kv)
        assert [z for z, _ in dq] == sorted(z for z, _ in dq)
