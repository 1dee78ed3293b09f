"""Tensor-level convenience wrapper over the C ABI.

PyTorch only provides the device memory and the stream here; the computation
is the CUDA library's.
"""
from __future__ import annotations

import math

from . import _lib


def attention_forward(q, k, v, scale: float | None = None, causal: bool = False,
                      kv_valid_len=None, out=None, lse=None, stream=None, n_splits: int | None = None):
    """O and LSE for bf16 CUDA tensors q [B,H,S_q,D], k/v [B,H,S_kv,D].

    kv_valid_len: int32 CUDA tensor [B] or None.  n_splits: key chunks (None
    picks attn_fwd_splitkv_suggest's count; more than 1 takes a torch-allocated
    workspace).  Returns (o, lse) with o bf16 [B,H,S_q,D] and lse fp32 [B,H,S_q].
    """
    import torch

    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bfloat16")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous [B,H,S,D]")
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    if tuple(k.shape) != (B, H, S_kv, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B,H,S_kv,D] matching q")
    if kv_valid_len is not None:
        if kv_valid_len.dtype != torch.int32 or not kv_valid_len.is_cuda or kv_valid_len.numel() != B:
            raise ValueError("kv_valid_len must be an int32 CUDA tensor with B entries")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S_q), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if n_splits is None:
        n_splits = _lib.attn_fwd_splitkv_suggest(B, H, S_q, S_kv, D, causal)
    if n_splits > 1:
        nbytes = _lib.attn_fwd_splitkv_workspace_bytes(B, H, S_q, D, n_splits)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
        _lib.attn_fwd_splitkv(q, k, v, out, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len,
                              n_splits, ws, nbytes, stream)
    else:
        _lib.attn_fwd(q, k, v, out, lse, B, H, S_q, S_kv, D, scale, causal, kv_valid_len, stream)
    return out, lse


def attention_backward(q, k, v, o, lse, d_o, scale: float | None = None, causal: bool = False,
                       kv_valid_len=None, stream=None):
    """dQ, dK, dV (bf16) for the forward pass that produced (o, lse) from q, k, v.

    All tensors are contiguous CUDA tensors as attention_forward uses them; d_o
    is bf16 [B,H,S_q,D].  The fp32 workspace comes from torch's allocator.
    """
    import torch

    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    for t in (q, k, v, o, d_o):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, d_o must be contiguous bf16 CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = _lib.attn_bwd_workspace_bytes(B, H, S_q, D)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    _lib.attn_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B, H, S_q, S_kv, D, scale, causal, kv_valid_len,
                  ws, nbytes, stream)
    return dq, dk, dv
