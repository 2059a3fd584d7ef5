"""Float64 CPU oracle for the attention forward.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()`` and the bench's
CPU baseline, never by the product path.
"""
from .attention import (  # noqa: F401
    attention_dense, attention_gqa_dense, attention_gqa_varlen, attention_head_rows,
    attention_varlen, bf16_bits_to_f64,
    online_softmax_attention, probabilities,
)
