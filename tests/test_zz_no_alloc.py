"""The no-allocation entry point (attn_fwd_unfused_noalloc): the unfused path with the library's
built-in scratch array, for callers that cannot allocate device memory.  Its output must match
the workspace entry point (attn_fwd_unfused) within the parity tolerance on two calls in a row,
and problems larger than the built-in scratch must be refused before the GPU is touched.

Collected last on purpose (file name), so a run that stops at the first failure has run every
other test first.  It passes alone in a fresh process and after the other tests."""
import os
import re

import numpy as np
import pytest
import torch

from gen import configs
from io_aware_attention_attn_gb300 import attn, build

from parity_util import check, to_dev, to_f64



def _scratch_limit() -> int:
    """ATTN_NOALLOC_SCRATCH_BYTES as the public header defines it (one source for the limit)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "include", "attn_gb300.h")) as f:
        m = re.search(r"#define\s+ATTN_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)",
                      f.read())
    assert m, "ATTN_NOALLOC_SCRATCH_BYTES not found in include/attn_gb300.h"
    return int(m.group(1)) << int(m.group(2))


SCRATCH_LIMIT = _scratch_limit()


def test_refuses_problems_beyond_the_scratch_limit():
    build.build()
    lib = attn.lib()
    # the largest single-head problem that fits, and the next size up, straddle the limit
    assert lib.attn_fwd_unfused_workspace_bytes(1, 1, 3328, 128) <= SCRATCH_LIMIT
    assert lib.attn_fwd_unfused_workspace_bytes(1, 1, 3329, 128) > SCRATCH_LIMIT
    B, H, N, d = 4, 16, 1024, 64  # needs about 400 MB of scratch
    assert lib.attn_fwd_unfused_workspace_bytes(B, H, N, d) > SCRATCH_LIMIT
    fake = 0x10000  # never dereferenced: the size check comes first
    assert lib.attn_fwd_unfused_noalloc(fake, fake, fake, fake, fake, B, H, N, d, 1, 0.125,
                                        None) == -10
    assert lib.attn_fwd_unfused_noalloc(fake, fake, fake, fake, fake, 1, 1, 100, 96, 0, 0.1,
                                        None) == -2


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build.build()
    # two calls in a row of different sizes (the array keeps the last contents), then a problem
    # that fills 99 % of the array, so its top end is written and read back
    cases = [configs.custom(401, 2, 3, 700, 128, True), configs.custom(402, 1, 2, 300, 64, False),
             configs.custom(403, 1, 1, 3327, 128, True)]
    for w in cases:
        q, k, v, _ = w.make()
        qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
        assert attn.unfused_workspace_bytes(w.B, w.H, w.N, w.d) <= SCRATCH_LIMIT
        if w.N == 3327:
            assert attn.unfused_workspace_bytes(w.B, w.H, w.N, w.d) > 0.98 * SCRATCH_LIMIT
        o_ref, l_ref = attn.attn_fwd_unfused(qd, kd, vd, causal=w.causal, scale=w.scale)
        o_na, l_na = attn.attn_fwd_unfused_noalloc(qd, kd, vd, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        check(to_f64(o_na), l_na.cpu().numpy().astype(np.float64), to_f64(o_ref),
              l_ref.cpu().numpy().astype(np.float64), f"no-alloc vs workspace {w.name}")
    assert attn.last_device_error() == 0
