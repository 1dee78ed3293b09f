"""ctypes binding of the C ABI declared in ``include/attn_fwd.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library.  If the library has not been built, calls raise ``RuntimeError``;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import threading

from .build_ext import LIB_PATH

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ALIGNMENT = 3
ATTN_ERR_LAUNCH = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_DEVICE = 6

# every extern "C" function include/attn_fwd.h declares
EXPORTED = ("attn_fwd", "attn_fwd_fp8", "attn_bwd", "attn_bwd_workspace_bytes", "attn_fwd_splitkv", "attn_fwd_splitkv_workspace_bytes",
            "attn_fwd_splitkv_suggest", "attn_fwd_schedule", "attn_merge", "attn_fwd_splitkv_static", "attn_status_str", "attn_fwd_debug_status",
            "attn_watchdog_selftest", "attn_fwd_abi_version")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A non-zero attn_status_t returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {attn_status_str(status)} (status {status})")


def load() -> ctypes.CDLL:
    """Load the built library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                                   "(run __graft_entry__.build() or "
                                   "python -m io_aware_attention_fwd_gb300.build_ext)")
            lib = ctypes.CDLL(str(LIB_PATH))
            p, i = ctypes.c_void_p, ctypes.c_int
            lib.attn_fwd.restype = i
            lib.attn_fwd.argtypes = [p, p, p, p, p, i, i, i, i, i, ctypes.c_float, i, p, p]
            u64, i64 = ctypes.c_uint64, ctypes.c_int64
            lib.attn_fwd_splitkv.restype = i
            lib.attn_fwd_splitkv.argtypes = [p, p, p, p, p, i, i, i, i, i, ctypes.c_float, i, p, i, p, u64, p]
            lib.attn_fwd_splitkv_workspace_bytes.restype = u64
            lib.attn_fwd_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
            lib.attn_fwd_splitkv_suggest.restype = i
            lib.attn_fwd_splitkv_suggest.argtypes = [i, i, i, i, i, i]
            lib.attn_fwd_schedule.restype = i
            lib.attn_fwd_schedule.argtypes = [i, i, i, i, i, i, i, p, p, i]
            f = ctypes.c_float
            lib.attn_bwd.restype = i
            lib.attn_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, f, i, p, p, u64, p]
            lib.attn_bwd_workspace_bytes.restype = u64
            lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
            lib.attn_fwd_fp8.restype = i
            lib.attn_fwd_fp8.argtypes = [p, p, p, p, p, i, i, i, i, i, f, f, f, f, i, p, p]
            lib.attn_fwd_splitkv_static.restype = i
            lib.attn_fwd_splitkv_static.argtypes = [p, p, p, p, p, i, i, i, i, i, ctypes.c_float, i, p, i, p]
            lib.attn_merge.restype = i
            lib.attn_merge.argtypes = [p, p, i, i64, i, p, p, p]
            lib.attn_status_str.restype = ctypes.c_char_p
            lib.attn_status_str.argtypes = [i]
            lib.attn_fwd_debug_status.restype = i
            lib.attn_fwd_debug_status.argtypes = [p]
            lib.attn_watchdog_selftest.restype = i
            lib.attn_watchdog_selftest.argtypes = [ctypes.c_uint64, p]
            lib.attn_fwd_abi_version.restype = i
            lib.attn_fwd_abi_version.argtypes = []
            _lib = lib
    return _lib


def _addr(x):
    """Device address of a tensor-like (``data_ptr()``) or a plain int/None."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def attn_status_str(status: int) -> str:
    return load().attn_status_str(int(status)).decode()


def attn_fwd(q, k, v, o, lse, B: int, H: int, S_q: int, S_kv: int, D: int, scale: float,
             causal: bool, kv_valid_len=None, stream=None) -> None:
    """Enqueue the attention forward pass (see include/attn_fwd.h).

    q, k, v, o, lse, kv_valid_len: device buffers (tensors or raw addresses).
    Raises AttnError on a non-zero status.
    """
    st = load().attn_fwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                         int(S_q), int(S_kv), int(D), float(scale), int(bool(causal)),
                         _addr(kv_valid_len), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")


def attn_fwd_fp8(q, k, v, o, lse, B: int, H: int, S_q: int, S_kv: int, D: int, scale: float,
                 q_descale: float, k_descale: float, v_descale: float, causal: bool,
                 kv_valid_len=None, stream=None) -> None:
    """Enqueue the FP8 (e4m3) forward pass (see include/attn_fwd.h)."""
    st = load().attn_fwd_fp8(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                             int(S_q), int(S_kv), int(D), float(scale), float(q_descale),
                             float(k_descale), float(v_descale), int(bool(causal)),
                             _addr(kv_valid_len), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_fp8")


def attn_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B: int, H: int, S_q: int, S_kv: int, D: int,
             scale: float, causal: bool, kv_valid_len, workspace, workspace_bytes: int,
             stream=None) -> None:
    """Enqueue the backward pass (see include/attn_fwd.h)."""
    st = load().attn_bwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(d_o), _addr(dq),
                         _addr(dk), _addr(dv), int(B), int(H), int(S_q), int(S_kv), int(D),
                         float(scale), int(bool(causal)), _addr(kv_valid_len), _addr(workspace),
                         int(workspace_bytes), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")


def attn_bwd_workspace_bytes(B: int, H: int, S_q: int, D: int) -> int:
    return int(load().attn_bwd_workspace_bytes(int(B), int(H), int(S_q), int(D)))


def attn_fwd_splitkv(q, k, v, o, lse, B: int, H: int, S_q: int, S_kv: int, D: int, scale: float,
                     causal: bool, kv_valid_len, n_splits: int, workspace, workspace_bytes: int,
                     stream=None) -> None:
    """Enqueue the key-split forward pass (see include/attn_fwd.h)."""
    st = load().attn_fwd_splitkv(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H),
                                 int(S_q), int(S_kv), int(D), float(scale), int(bool(causal)),
                                 _addr(kv_valid_len), int(n_splits), _addr(workspace),
                                 int(workspace_bytes), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv")


def attn_fwd_splitkv_workspace_bytes(B: int, H: int, S_q: int, D: int, n_splits: int) -> int:
    return int(load().attn_fwd_splitkv_workspace_bytes(int(B), int(H), int(S_q), int(D), int(n_splits)))


def attn_fwd_splitkv_suggest(B: int, H: int, S_q: int, S_kv: int, D: int, causal: bool) -> int:
    return int(load().attn_fwd_splitkv_suggest(int(B), int(H), int(S_q), int(S_kv), int(D),
                                               int(bool(causal))))


def attn_fwd_schedule(B: int, H: int, S_q: int, S_kv: int, D: int, elem_bytes: int, sms: int):
    """The host-built unit order of a causal launch of this shape (see
    include/attn_fwd.h): (off, unit) as lists, CTA c running
    unit[off[c]:off[c + 1]]; None where the launch has no such order."""
    n_pairs = -(-int(S_q) // 256)
    cap = max(1, int(B) * int(H) * n_pairs)
    off = (ctypes.c_uint16 * (max(1, int(sms)) + 1))()
    unit = (ctypes.c_uint16 * cap)()
    n = load().attn_fwd_schedule(int(B), int(H), int(S_q), int(S_kv), int(D), int(elem_bytes), int(sms),
                                 ctypes.addressof(off), ctypes.addressof(unit), cap)
    if n < 0:
        raise ValueError("attn_fwd_schedule: invalid arguments")
    if n == 0:
        return None
    G = min(n, int(sms))
    return list(off[:G + 1]), list(unit[:n])


def attn_merge(o_parts, lse_parts, n_parts: int, rows: int, D: int, o, lse, stream=None) -> None:
    """Enqueue the log-sum-exp merge of per-key-set results (see include/attn_fwd.h)."""
    st = load().attn_merge(_addr(o_parts), _addr(lse_parts), int(n_parts), int(rows), int(D),
                           _addr(o), _addr(lse), _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_merge")


# Size of the library's fixed scratch (ATTN_STATIC_SCRATCH_BYTES in the header).
STATIC_SCRATCH_BYTES = 32 << 20


def attn_fwd_splitkv_static(q, k, v, o, lse, B: int, H: int, S_q: int, S_kv: int, D: int,
                            scale: float, causal: bool, kv_valid_len, n_splits: int,
                            stream=None) -> None:
    """Key-split forward using the library's fixed scratch instead of a
    workspace, for callers that cannot allocate device memory (see
    include/attn_fwd.h: 32 MiB cap, one call at a time on the GPU)."""
    st = load().attn_fwd_splitkv_static(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B),
                                        int(H), int(S_q), int(S_kv), int(D), float(scale),
                                        int(bool(causal)), _addr(kv_valid_len), int(n_splits),
                                        _stream(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv_static")


def call_status(fn, *args, **kwargs) -> int:
    """Run one of the raising wrappers above and return its status instead."""
    try:
        fn(*args, **kwargs)
    except AttnError as e:
        return e.status
    return ATTN_OK


def attn_fwd_status(*args, **kwargs) -> int:
    """Same as attn_fwd but returns the raw status instead of raising."""
    try:
        attn_fwd(*args, **kwargs)
    except AttnError as e:
        return e.status
    return ATTN_OK


def attn_fwd_debug_status(stream=None) -> int:
    return int(load().attn_fwd_debug_status(_stream(stream)))


def attn_watchdog_selftest(timeout_ns: int, stream=None) -> int:
    return int(load().attn_watchdog_selftest(int(timeout_ns), _stream(stream)))


def attn_fwd_abi_version() -> int:
    return int(load().attn_fwd_abi_version())
