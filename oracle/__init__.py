"""fp64 CPU oracle for the fused attention forward pass -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does.

The attention arithmetic lives in ``attn_ref.cpp`` (plain float64 C++, one
materialised score row per query, two-pass softmax).  This module compiles it
with the host C++ compiler on first use (or from ``build()``) and calls it
through ctypes; ``merge_f64`` (the log-sum-exp merge of results over disjoint
key sets) and ``attention_bwd_f64`` (the gradients, per head with P
materialised) are plain float64 numpy here.

Parity pins: ``tests/test_oracle_pins.py`` and ``tests/test_oracle_mutants.py``
(forward, merge); ``tests/test_oracle_bwd_pins.py`` (gradients: finite
differences of the C++ forward, torch float64 autograd, closed-form sums).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "attn_ref.cpp"
BUILD_DIR = _HERE / "_build"
LIB_PATH = BUILD_DIR / "libattn_ref.so"

_lib = None


def compile_library(source: Path = SOURCE, out: Path = LIB_PATH, extra_flags=()) -> Path:
    """Compile ``source`` into the shared library ``out`` (atomic rename)."""
    out.parent.mkdir(parents=True, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=str(out.parent))
    os.close(fd)
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
           *extra_flags, str(source), "-o", tmp]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> Path:
    """Build the oracle library if it is missing or older than its source."""
    if force or not LIB_PATH.exists() or LIB_PATH.stat().st_mtime < SOURCE.stat().st_mtime:
        compile_library()
    return LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.attn_ref_f64.restype = ctypes.c_int
    lib.attn_ref_f64.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_double,
                                 ctypes.c_int, p, p, i64, p, p, ctypes.c_int]
    lib.attn_ref_score_buffer_bytes.restype = ctypes.c_uint64
    lib.attn_ref_score_buffer_bytes.argtypes = [i64, i64, i64, i64]
    lib.attn_ref_hardware_threads.restype = ctypes.c_int
    lib.attn_ref_hardware_threads.argtypes = []
    lib.attn_ref_f64_dbl.restype = ctypes.c_int
    lib.attn_ref_f64_dbl.argtypes = lib.attn_ref_f64.argtypes
    return lib


def load_library(path: Path | None = None) -> ctypes.CDLL:
    """Load the default oracle library (building it if needed), or ``path``."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(str(build())))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def attention_f64(q_bits, k_bits, v_bits, scale: float, causal: bool,
                  kv_valid_len=None, rows=None, threads: int = 0, lib=None):
    """Reference O and LSE in float64.

    q_bits: uint16 bf16 bits [B,H,S_q,D]; k_bits, v_bits: [B,H,S_kv,D].
    kv_valid_len: ints of length B or None.  rows: flat row ids
    ``(b*H + h)*S_q + i`` or None for all rows.
    Returns (o [n_rows, D] float64, lse [n_rows] float64).
    """
    lib = lib or load_library()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    if k.shape != (B, H, S_kv, D) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    kvl = None if kv_valid_len is None else np.ascontiguousarray(kv_valid_len, dtype=np.int32)
    if kvl is not None and kvl.shape != (B,):
        raise ValueError("kv_valid_len must have one entry per batch")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_rows = B * H * S_q if r is None else int(r.shape[0])
    o = np.empty((n_rows, D), dtype=np.float64)
    lse = np.empty((n_rows,), dtype=np.float64)
    rc = lib.attn_ref_f64(_ptr(q), _ptr(k), _ptr(v), B, H, S_q, S_kv, D, float(scale),
                          int(bool(causal)), _ptr(kvl), _ptr(r), n_rows, _ptr(o), _ptr(lse),
                          int(threads))
    if rc != 0:
        raise ValueError(f"attn_ref_f64 rejected its arguments (rc={rc})")
    return o, lse


def attention_f64_dbl(q, k, v, scale: float, causal: bool, kv_valid_len=None, rows=None,
                      threads: int = 0, lib=None):
    """attention_f64 on float64 inputs (same layouts), through the same C++ code."""
    lib = lib or load_library()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    kvl = None if kv_valid_len is None else np.ascontiguousarray(kv_valid_len, dtype=np.int32)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_rows = B * H * S_q if r is None else int(r.shape[0])
    o = np.empty((n_rows, D), dtype=np.float64)
    lse = np.empty((n_rows,), dtype=np.float64)
    rc = lib.attn_ref_f64_dbl(_ptr(q), _ptr(k), _ptr(v), B, H, S_q, S_kv, D, float(scale),
                              int(bool(causal)), _ptr(kvl), _ptr(r), n_rows, _ptr(o), _ptr(lse),
                              int(threads))
    if rc != 0:
        raise ValueError(f"attn_ref_f64_dbl rejected its arguments (rc={rc})")
    return o, lse


def _widen(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:  # bf16 bit patterns
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def attention_bwd_f64(q, k, v, d_o, scale: float, causal: bool, kv_valid_len=None, heads=None):
    """Gradients of the attention forward pass, in float64.

    q, d_o: [B,H,S_q,D]; k, v: [B,H,S_kv,D], as bf16 bit patterns (uint16) or
    float arrays.  For each (b, h), with the masked score matrix
    S = scale * Q K^T (masked entries -inf) and P = softmax(S) row by row (a
    row with no allowed key is all zero):
        dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(P * dP)),
        dQ = scale * dS K,  dK = scale * dS^T Q.
    These are the chain rule through O = P V and the softmax; the forward
    pass is the one the pages define ("Attention memory" page, "What this
    memory is"; masked keys as in the masked_fill sentences of the "PyTorch
    attention backends" story).  P is materialised per head: plain, slow,
    obviously correct.  ``heads``: optional list of (b, h) pairs to compute
    (the gradients of every other head are left at zero), for checking a
    sample of the heads of a large problem.  Returns (dq, dk, dv) as float64
    arrays.
    """
    q, k, v, d_o = (_widen(x) for x in (q, k, v, d_o))
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    i = np.arange(S_q)[:, None]
    j = np.arange(S_kv)[None, :]
    for b in range(B):
        valid = S_kv if kv_valid_len is None else min(max(int(kv_valid_len[b]), 0), S_kv)
        allowed = np.broadcast_to(j < valid, (S_q, S_kv))
        if causal:
            allowed = allowed & (j <= i)
        for h in range(H):
            if heads is not None and (b, h) not in heads:
                continue
            s = scale * (q[b, h] @ k[b, h].T)
            s = np.where(allowed, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.where(allowed, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)
            l = e.sum(axis=1, keepdims=True)
            p = np.divide(e, l, out=np.zeros_like(e), where=l > 0)
            dv[b, h] = p.T @ d_o[b, h]
            dp = d_o[b, h] @ v[b, h].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv


def score_buffer_bytes(B: int, H: int, s: int, e: int, lib=None) -> int:
    """Bytes of a materialised B x H x s x s score matrix, e bytes per score."""
    lib = lib or load_library()
    return int(lib.attn_ref_score_buffer_bytes(B, H, s, e))


def hardware_threads(lib=None) -> int:
    lib = lib or load_library()
    return int(lib.attn_ref_hardware_threads())


def merge_f64(o_parts, lse_parts):
    """Combine attention results over disjoint key sets, in float64.

    o_parts: [n_parts, rows, D]; lse_parts: [n_parts, rows] (natural log,
    -inf for a part with no keys).  Returns (o [rows, D], lse [rows]):
    lse = ln sum_k exp(lse_k) and o = sum_k exp(lse_k - lse) o_k; a row with no
    keys in any part gets o = 0 and lse = -inf.  This is the softmax over the
    union of the key sets written per part ("Flash attention" glossary page,
    paragraphs 2 and 4: running softmax statistics, and the same tiling spread
    over devices).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    rows = lse_parts.shape[1]
    o = np.zeros(o_parts.shape[1:], dtype=np.float64)
    lse = np.full(rows, -np.inf)
    for r in range(rows):
        m = lse_parts[:, r].max()
        if m == -np.inf:
            continue
        w = np.exp(lse_parts[:, r] - m)          # weight of each part, up to a common factor
        lse[r] = m + np.log(w.sum())
        o[r] = (w[:, None] * o_parts[:, r, :]).sum(axis=0) / w.sum()
    return o, lse
