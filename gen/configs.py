"""The five attention-forward workloads and their seeded input recipes.

Each workload is described by what it is (shape, masking, value distribution); the inputs
are bf16 bit patterns from :mod:`gen.inputs`.  Recipe:

* Q, K, V iid N(0, sigma^2) in float64, rounded to bf16 (RNE); Q, K and V use the
  independent splitmix64 streams ``3*seed``, ``3*seed+1`` and ``3*seed+2`` with
  ``seed = 20260000 + index``.
* ``scale = 1/sqrt(d)``.
* Backward cases add dO iid N(0, 1), rounded to bf16, on the stream ``4*seed + 3``.
* The packed variable-length batch draws its 16 lengths uniformly from [128, 4096] with the
  stream ``seed`` itself, and ``cu_seqlens`` is their int32 exclusive prefix sum.

Dense tensors are ``[B, H, N, d]`` (d innermost); packed tensors are ``[H, T, d]`` with
``T = cu_seqlens[-1]``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import inputs


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    H: int
    N: int           # dense: sequence length; packed: total tokens T (filled in by lengths())
    d: int
    causal: bool
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    varlen: bool = False
    H_kv: int = 0    # key/value heads (0: same as H); H_kv < H is grouped-query attention
    n_seqs: int = 0
    len_lo: int = 0
    len_hi: int = 0

    @property
    def seed(self) -> int:
        return 20260000 + self.index

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def lengths(self) -> np.ndarray:
        """Per-sequence lengths (dense: B copies of N)."""
        if not self.varlen:
            return np.full(self.B, self.N, dtype=np.int64)
        return inputs.uniform_int(self.seed, self.n_seqs, self.len_lo, self.len_hi)

    def cu_seqlens(self) -> np.ndarray | None:
        return inputs.cu_seqlens_from_lengths(self.lengths()) if self.varlen else None

    def total_tokens(self) -> int:
        return int(self.lengths().sum()) if self.varlen else self.B * self.N

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    def shape(self, heads=None) -> tuple:
        h = self.H if heads is None else heads
        if self.varlen:
            return (h, self.total_tokens(), self.d)
        return (self.B, h, self.N, self.d)

    def describe(self) -> dict:
        out = {"workload": self.name, "heads": self.H, "kv_heads": self.kv_heads, "head_dim": self.d,
               "causal": self.causal, "sigma_qk": self.sigma_qk, "sigma_v": self.sigma_v}
        if self.varlen:
            out.update({"layout": "packed [H,T,d] + cu_seqlens", "n_seqs": self.n_seqs,
                        "len_range": [self.len_lo, self.len_hi],
                        "total_tokens": self.total_tokens()})
        else:
            out.update({"layout": "[B,H,N,d]", "batch": self.B, "seq_len": self.N})
        return out

    def make_dout(self):
        """The upstream gradient dO for a backward case: iid N(0, 1) rounded to bf16, shaped like
        Q, on the splitmix64 stream ``4*seed + 3``."""
        return inputs.bf16_normal(4 * self.seed + 3, self.shape(), 1.0)

    def make(self, shape=None):
        """(q, k, v) as uint16 bf16 bit arrays, plus cu_seqlens (int32) or None.  K and V have
        ``kv_heads`` heads."""
        qshape = self.shape() if shape is None else shape
        kvshape = self.shape(self.kv_heads) if shape is None else shape
        q = inputs.bf16_normal(3 * self.seed + 0, qshape, self.sigma_qk)
        k = inputs.bf16_normal(3 * self.seed + 1, kvshape, self.sigma_qk)
        v = inputs.bf16_normal(3 * self.seed + 2, kvshape, self.sigma_v)
        return q, k, v, self.cu_seqlens()


WORKLOADS = {
    1: Workload(1, "B1-H2-N256-d64", B=1, H=2, N=256, d=64, causal=False),
    2: Workload(2, "B4-H16-N1024-d64-causal", B=4, H=16, N=1024, d=64, causal=True),
    3: Workload(3, "B2-H32-N4096-d128", B=2, H=32, N=4096, d=128, causal=False),
    4: Workload(4, "B1-H32-N16384-d128-causal-peaky", B=1, H=32, N=16384, d=128, causal=True,
                sigma_qk=2.0, sigma_v=1.0),
    5: Workload(5, "varlen16xU[128,4096]-H16-d128-causal", B=16, H=16, N=0, d=128,
                causal=True, varlen=True, n_seqs=16, len_lo=128, len_hi=4096),
}

# The headline throughput workload (B=2, H=32, N=4096, d=128, non-causal).
HEADLINE = 3

# Grouped-query variant of the headline shape (32 query heads sharing 8 K/V heads).
GQA = Workload(6, "B2-H32-KV8-N4096-d128", B=2, H=32, N=4096, d=128, causal=False, H_kv=8)

# Few heads, long sequence: 32 query pairs (64 SMs at head dim 128) leave most of the 152 SMs
# idle unless the key range is split (the split-KV case).
SPLITKV = Workload(7, "B1-H1-N8192-d128", B=1, H=1, N=8192, d=128, causal=False)


def custom(index_seed: int, B: int, H: int, N: int, d: int, causal: bool,
           sigma_qk: float = 1.0, sigma_v: float = 1.0, H_kv: int = 0) -> Workload:
    """A dense workload with the same recipe and an arbitrary seed (edge-shape tests)."""
    kv = f"-KV{H_kv}" if H_kv else ""
    return Workload(index_seed, f"B{B}-H{H}{kv}-N{N}-d{d}{'-causal' if causal else ''}",
                    B=B, H=H, N=N, d=d, causal=causal, sigma_qk=sigma_qk, sigma_v=sigma_v,
                    H_kv=H_kv)


def custom_varlen(index_seed: int, lengths, H: int, d: int, causal: bool, H_kv: int = 0) -> tuple:
    """Packed inputs for explicit lengths: (q, k, v, cu_seqlens) bit arrays (K/V with H_kv heads)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    T = int(lengths.sum())
    seed = 20260000 + index_seed
    q = inputs.bf16_normal(3 * seed + 0, (H, T, d))
    k = inputs.bf16_normal(3 * seed + 1, (H_kv or H, T, d))
    v = inputs.bf16_normal(3 * seed + 2, (H_kv or H, T, d))
    return q, k, v, inputs.cu_seqlens_from_lengths(lengths)
