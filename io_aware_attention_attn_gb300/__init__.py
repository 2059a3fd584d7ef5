"""GB300-native IO-aware fused attention forward (sm_103a CUDA, C-ABI library + thin binding).

The compute path lives in ``libattn_gb300.so`` (built from ``csrc/``); :mod:`.attn` marshals
torch tensors into its C entry points.  Importing this package does not load the library;
the first call does, and fails loudly if the library is missing.
"""
__all__ = ["attn_fwd", "attn_bwd", "bwd_workspace_bytes", "attn_fwd_splitkv", "quantize_fp8", "attn_fwd_fp8", "splitkv_workspace_bytes", "attn_fwd_unfused",
           "unfused_workspace_bytes", "last_device_error"]


def __getattr__(name):
    if name in __all__:
        from . import attn
        return getattr(attn, name)
    raise AttributeError(name)
