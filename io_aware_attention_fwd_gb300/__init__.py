"""Fused scaled-dot-product attention forward for GB300 (sm_103a).

``attn_fwd`` and friends mirror the C ABI of ``include/attn_fwd.h``;
``attention_forward`` is a tensor-level convenience wrapper, and
``HostForward`` runs the forward pass on pinned host buffers with the copies
overlapped.  The CUDA
library is loaded on first use and must have been built (``build_ext``).
"""
from ._lib import (ATTN_ERR_ALIGNMENT, ATTN_ERR_DEVICE, ATTN_ERR_INVALID_ARG, ATTN_ERR_LAUNCH,
                   ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED, ATTN_OK, EXPORTED, AttnError, attn_fwd,
                   attn_fwd_fp8, attn_bwd, attn_bwd_workspace_bytes,
                   attn_fwd_abi_version, attn_fwd_debug_status, attn_fwd_schedule, attn_fwd_splitkv,
                   attn_fwd_splitkv_static, attn_fwd_splitkv_suggest,
                   attn_fwd_splitkv_workspace_bytes, attn_fwd_status,
                   STATIC_SCRATCH_BYTES, attn_merge, attn_status_str, attn_watchdog_selftest, call_status,
                   load)
from .api import attention_backward, attention_forward
from .host import HostForward, plan_pieces
from .build_ext import LIB_PATH, build

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_ALIGNMENT",
    "ATTN_ERR_LAUNCH", "ATTN_ERR_TIMEOUT", "ATTN_ERR_DEVICE", "EXPORTED", "AttnError",
    "attn_fwd", "attn_fwd_fp8", "attn_bwd", "attn_bwd_workspace_bytes", "attention_backward",
    "attn_fwd_status", "attn_fwd_schedule", "attn_fwd_splitkv", "attn_fwd_splitkv_suggest",
    "attn_fwd_splitkv_workspace_bytes", "attn_fwd_splitkv_static", "STATIC_SCRATCH_BYTES",
    "attn_merge", "call_status",
    "attn_status_str",
    "attn_fwd_debug_status",
    "attn_watchdog_selftest", "attn_fwd_abi_version", "attention_forward", "load", "build",
    "LIB_PATH", "HostForward", "plan_pieces",
]
