"""Thin Python binding of ``libattn_gb300.so`` (ctypes): argument marshalling only.

Every step of the attention forward runs in the library's CUDA kernels; PyTorch only supplies
device memory, streams and the output allocations.  There is no fallback: if the library is
missing or the GPU is not an sm_103 part, calls raise.

Layouts (same as the C ABI in ``include/attn_gb300.h``):
  dense  q, k, v, o: [B, H, N, d] bf16 contiguous; lse [B, H, N] fp32
  packed q, k, v, o: [H, T, d] bf16 contiguous + cu_seqlens int32 [n+1]; lse [H, T] fp32
"""
from __future__ import annotations

import ctypes
import math
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn_gb300.so")

STATUS = {
    0: "ATTN_OK", -1: "ATTN_ERR_NULL", -2: "ATTN_ERR_HEAD_DIM", -3: "ATTN_ERR_SHAPE",
    -4: "ATTN_ERR_ALIGN", -5: "ATTN_ERR_LAUNCH", -6: "ATTN_ERR_DEVICE", -7: "ATTN_ERR_SCALE",
    -8: "ATTN_ERR_WORKSPACE", -9: "ATTN_ERR_UNSUPPORTED", -10: "ATTN_ERR_SCRATCH_LIMIT",
}

# exported C symbols and their ctypes signatures (kept in step with include/attn_gb300.h)
_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_gqa": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "attn_fwd_splitkv_workspace_bytes": (_S, [_I, _I, _I, _I, _I]),
    "attn_fwd_splitkv_slices": (_I, [_I, _I, _I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _S, _P]),
    "attn_bwd_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P,
                          _S, _P]),
    "attn_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                             _F, _P, _S, _P]),
    "attn_bwd_varlen_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "attn_bwd_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "attn_quantize_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "attn_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_unfused": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _S, _P]),
    "attn_fwd_unfused_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "attn_fwd_unfused_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "attn_get_last_device_error": (_I, [_P]),
    "attn_selftest_mma": (_I, [_P, _P, _P, _I, _I, _P]),
    "attn_selftest_wait_timeout": (_I, [_P]),
    "attn_selftest_fp8_quotients": (_I, [_P, _P]),
    "attn_version": (_I, []),
}


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load the library once (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m io_aware_attention_attn_gb300.build`"
                " (or __graft_entry__.build())")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _lib = handle
    return _lib


def _check(name: str, rc: int):
    if rc != 0:
        raise AttnError(name, rc)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_inputs(q, k, v, cu_seqlens, allow_kv_heads=False):
    """Returns (B, H, H_kv, N, d).  K and V may have fewer heads than Q when allow_kv_heads."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
        if t.dim() != q.dim() or t.device != q.device:
            raise ValueError("q, k and v must have the same rank and device")
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    hd = 1 if cu_seqlens is None else 0  # index of the head axis
    if q.shape[:hd] + q.shape[hd + 1:] != k.shape[:hd] + k.shape[hd + 1:]:
        raise ValueError("q and k/v differ in a dimension other than heads")
    if not allow_kv_heads and k.shape != q.shape:
        raise ValueError("q, k and v must have the same shape")
    if cu_seqlens is None:
        if q.dim() != 4:
            raise ValueError("dense inputs are [B, H, N, d]")
        B, H, N, d = q.shape
    else:
        if q.dim() != 3:
            raise ValueError("packed inputs are [H, T, d] with cu_seqlens")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or \
                not cu_seqlens.is_contiguous() or cu_seqlens.dim() != 1 or \
                cu_seqlens.device != q.device:
            raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor on q's device")
        H, N, d = q.shape
        B = cu_seqlens.numel() - 1
    H_kv = k.shape[hd]
    if H_kv == 0 or H % H_kv != 0:
        raise ValueError("the number of K/V heads must divide the number of query heads")
    return B, H, H_kv, N, d


def attn_fwd(q, k, v, cu_seqlens=None, causal: bool = False, scale: float | None = None,
             out=None, lse=None, stream=None):
    """Fused attention forward.  Returns (O bf16 like q, LSE fp32).

    k and v may have fewer heads than q (grouped-query / multi-query attention: query head h
    reads K/V head h // (H // H_kv)); then the attn_fwd_gqa entry point is called."""
    import torch
    B, H, H_kv, N, d = _check_inputs(q, k, v, cu_seqlens, allow_kv_heads=True)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    cu = cu_seqlens.data_ptr() if cu_seqlens is not None else None
    with torch.cuda.device(q.device):
        st = _stream_handle(stream, q.device)
        if H_kv == H:
            rc = lib().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), cu, B, H, N, d, int(bool(causal)), float(scale), st)
        else:
            rc = lib().attn_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), cu, B, H, H_kv, N, d, int(bool(causal)),
                                    float(scale), st)
    _check("attn_fwd_gqa" if H_kv != H else "attn_fwd", rc)
    return out, lse


def splitkv_workspace_bytes(B: int, H: int, N: int, d: int, num_splits: int = 0) -> int:
    return int(lib().attn_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits))


def splitkv_slices(B: int, H: int, N: int, d: int, num_splits: int = 0) -> int:
    return int(lib().attn_fwd_splitkv_slices(B, H, N, d, num_splits))


def attn_fwd_splitkv(q, k, v, causal: bool = False, scale: float | None = None,
                     num_splits: int = 0, workspace=None, out=None, lse=None, stream=None):
    """Split-KV fused forward (dense [B, H, N, d] only): the key range of every query pair is
    cut into ``num_splits`` slices (0: the library chooses) whose partial results a second kernel
    merges.  Returns (O bf16 like q, LSE fp32)."""
    import torch
    B, H, _, N, d = _check_inputs(q, k, v, None)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = splitkv_workspace_bytes(B, H, N, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                    int(num_splits), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream, q.device))
    _check("attn_fwd_splitkv", rc)
    return out, lse


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, H, N, d))


def attn_bwd(q, k, v, o, lse, dout, cu_seqlens=None, causal: bool = False,
             scale: float | None = None, workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Backward pass: gradients (dQ, dK, dV) of the fused forward for the upstream gradient
    ``dout``, given the forward's ``o`` and ``lse``.  Dense [B, H, N, d], or packed [H, T, d] with
    ``cu_seqlens`` (attn_bwd_varlen); k and v may have fewer heads than q (grouped-query: dK and dV
    summed over each group)."""
    import torch
    B, H, H_kv, N, d = _check_inputs(q, k, v, cu_seqlens, allow_kv_heads=True)
    for name, t in (("o", o), ("dout", dout)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape != q.shape or \
                t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.shape != q.shape[:-1] or \
            lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 tensor of shape [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = (bwd_workspace_bytes(B, H, N, d) if cu_seqlens is None
            else int(lib().attn_bwd_varlen_workspace_bytes(B, H, N, d)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    with torch.cuda.device(q.device):
        st = _stream_handle(stream, q.device)
        if cu_seqlens is not None:
            rc = lib().attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(), cu_seqlens.data_ptr(), B, H,
                                       H_kv, N, d, int(bool(causal)), float(scale), *ws, st)
        elif H_kv == H:
            rc = lib().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale), *ws, st)
        else:
            rc = lib().attn_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                    dv.data_ptr(), B, H, H_kv, N, d, int(bool(causal)),
                                    float(scale), *ws, st)
    _check("attn_bwd_varlen" if cu_seqlens is not None else
           ("attn_bwd_gqa" if H_kv != H else "attn_bwd"), rc)
    return dq, dk, dv


def quantize_fp8(x, transpose: bool = False, stream=None):
    """Per-tile E4M3 quantization of a dense bf16 tensor [B, H, N, d].  Returns (codes uint8,
    scales fp32 [B, H, ceil(N/128)]); codes are [B, H, N, d], or [B, H, d, Npad] when
    ``transpose`` (the V operand of attn_fwd_fp8)."""
    import torch
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.dim() != 4:
        raise ValueError("x must be a contiguous [B, H, N, d] bf16 CUDA tensor")
    B, H, N, d = x.shape
    T = -(-N // 128)
    shape = (B, H, d, T * 128) if transpose else (B, H, N, d)
    codes = torch.empty(shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, H, T), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib().attn_quantize_fp8(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), B, H, N,
                                     d, int(bool(transpose)), _stream_handle(stream, x.device))
    _check("attn_quantize_fp8", rc)
    return codes, scales


def attn_fwd_fp8(q8, sq, k8, sk, vt8, sv, causal: bool = False, scale: float | None = None,
                 out=None, lse=None, stream=None):
    """FP8 fused forward on quantized inputs (see quantize_fp8).  Returns (O bf16, LSE fp32)."""
    import torch
    if q8.dtype != torch.uint8 or q8.dim() != 4 or not q8.is_contiguous():
        raise ValueError("q8 must be contiguous [B, H, N, 128] uint8 codes")
    B, H, N, d = q8.shape
    T = -(-N // 128)
    if k8.shape != q8.shape or vt8.shape != (B, H, d, T * 128) or \
            sq.shape != (B, H, T) or sk.shape != (B, H, T) or sv.shape != (B, H, T):
        raise ValueError("k8, vt8 and the scales must match q8 (vt8 is [B, H, d, Npad])")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    with torch.cuda.device(q8.device):
        rc = lib().attn_fwd_fp8(q8.data_ptr(), sq.data_ptr(), k8.data_ptr(), sk.data_ptr(),
                                vt8.data_ptr(), sv.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                B, H, N, d, int(bool(causal)), float(scale),
                                _stream_handle(stream, q8.device))
    _check("attn_fwd_fp8", rc)
    return out, lse


def unfused_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().attn_fwd_unfused_workspace_bytes(B, H, N, d))


def attn_fwd_unfused(q, k, v, causal: bool = False, scale: float | None = None, workspace=None,
                     out=None, lse=None, stream=None):
    """Unfused three-kernel comparison path (S and P through HBM).  Dense layout only."""
    import torch
    B, H, _, N, d = _check_inputs(q, k, v, None)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = unfused_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_unfused(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), None, B, H, N, d, int(bool(causal)),
                                    float(scale), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(),
                                    _stream_handle(stream, q.device))
    _check("attn_fwd_unfused", rc)
    return out, lse


def attn_fwd_unfused_noalloc(q, k, v, causal: bool = False, scale: float | None = None,
                             out=None, lse=None, stream=None):
    """The unfused path using the library's built-in scratch instead of a workspace (for callers
    that cannot allocate device memory; outputs may still be allocated here when not given)."""
    import torch
    B, H, _, N, d = _check_inputs(q, k, v, None)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_unfused_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            out.data_ptr(), lse.data_ptr(), B, H, N, d,
                                            int(bool(causal)), float(scale),
                                            _stream_handle(stream, q.device))
    _check("attn_fwd_unfused_noalloc", rc)
    return out, lse


def last_device_error(stream=None, device=None) -> int:
    """Device status word of the kernels on ``stream`` (0 = every pipeline wait completed)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        rc = lib().attn_get_last_device_error(_stream_handle(stream, dev))
    if rc < 0:
        raise AttnError("attn_get_last_device_error", rc)
    return rc


def selftest_mma(a, b, mode: int):
    """Diagnostic single-tile tensor-core product (see attn_selftest_mma in the header)."""
    import torch
    dim = b.shape[1]
    n_out = 128 if mode == 0 else dim
    d = torch.empty((128, n_out), dtype=torch.float32, device=a.device)
    with torch.cuda.device(a.device):
        rc = lib().attn_selftest_mma(a.data_ptr(), b.data_ptr(), d.data_ptr(), mode, dim,
                                     _stream_handle(None, a.device))
    _check("attn_selftest_mma", rc)
    return d


def selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test (returns at once; the status appears after ~1 s)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    _check("attn_selftest_wait_timeout",
           lib().attn_selftest_wait_timeout(_stream_handle(stream, dev)))


def selftest_fp8_quotients(stream=None) -> int:
    """Pairs (x, tile maximum) whose quantizer code differs from the code of the IEEE quotient
    (see attn_selftest_fp8_quotients in the header); synchronises the stream."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    out = torch.zeros(1, dtype=torch.int64, device=dev)
    _check("attn_selftest_fp8_quotients",
           lib().attn_selftest_fp8_quotients(out.data_ptr(), _stream_handle(stream, dev)))
    torch.cuda.synchronize(dev)
    return int(out.item())


def decode_status(code: int) -> dict:
    """Split a device status word into kind, role and wait site."""
    return {"kind": code & 0xFF, "role": (code >> 8) & 0xFF, "site": (code >> 16) & 0xFF}


def version() -> int:
    return int(lib().attn_version())
