"""Helpers shared by the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, and compare with the fp64 oracle on the same rows.

Tolerances (the parity bar): bf16 O within max-abs 2e-2 and
relative RMS 1e-2 of the oracle; fp32 LSE within 1e-3 absolute.  A row with
no allowed key must give O = 0 and LSE = -inf on both sides.
"""
from __future__ import annotations

import numpy as np

import oracle
import seeded_inputs as si

O_MAX_ABS = 2e-2
O_REL_RMS = 1e-2
LSE_ABS = 1e-3


def to_device(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def run_cuda(q_bits, k_bits, v_bits, scale, causal, kv_valid_len=None, device="cuda:0", stream=None,
             tensors=None):
    """Run attn_fwd on uploaded copies of the inputs; returns (o, lse) tensors on the device."""
    import torch
    import io_aware_attention_fwd_gb300 as attn

    B, H, S_q, D = q_bits.shape
    S_kv = k_bits.shape[2]
    tq, tk, tv = tensors if tensors is not None else (to_device(x, device) for x in (q_bits, k_bits, v_bits))
    o = torch.full((B, H, S_q, D), float("nan"), dtype=torch.bfloat16, device=device)
    lse = torch.full((B, H, S_q), float("nan"), dtype=torch.float32, device=device)
    kvl = None
    if kv_valid_len is not None:
        kvl = torch.tensor(list(kv_valid_len), dtype=torch.int32, device=device)
    if stream is None:
        stream = torch.cuda.current_stream(device)
    attn.attn_fwd(tq, tk, tv, o, lse, B, H, S_q, S_kv, D, scale, causal, kvl, stream)
    torch.cuda.synchronize(device)
    st = attn.attn_fwd_debug_status(stream)
    assert st == attn.ATTN_OK, attn.attn_status_str(st)
    return o, lse


def gather_rows(o, lse, rows=None):
    """Rows (flat ids) of the device outputs as float64 numpy arrays."""
    import torch
    D = o.shape[-1]
    of = o.reshape(-1, D)
    lf = lse.reshape(-1)
    if rows is not None:
        idx = torch.as_tensor(np.asarray(rows), device=o.device, dtype=torch.long)
        of, lf = of[idx], lf[idx]
    return of.float().cpu().numpy().astype(np.float64), lf.cpu().numpy().astype(np.float64)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, max_abs=O_MAX_ABS, rel_rms=O_REL_RMS, lse_abs=LSE_ABS):
    """Asserts the parity bar (the bf16 bar unless given); returns the errors."""
    assert o_gpu.shape == o_ref.shape and lse_gpu.shape == lse_ref.shape
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), empty), "rows without keys differ"
    assert np.all(o_gpu[empty] == 0.0), "rows without keys must give O = 0"
    full = ~empty
    assert np.all(np.isfinite(o_gpu[full])) and np.all(np.isfinite(lse_gpu[full])), "non-finite output"
    err = {"max_abs": 0.0, "rel_rms": 0.0, "lse_abs": 0.0, "rows": int(full.sum())}
    if full.any():
        d = o_gpu[full] - o_ref[full]
        err["max_abs"] = float(np.abs(d).max())
        err["rel_rms"] = float(np.linalg.norm(d) / max(np.linalg.norm(o_ref[full]), 1e-300))
        err["lse_abs"] = float(np.abs(lse_gpu[full] - lse_ref[full]).max())
    assert err["max_abs"] <= max_abs, err
    assert err["rel_rms"] <= rel_rms, err
    assert err["lse_abs"] <= lse_abs, err
    return err


def check_against_oracle(q, k, v, scale, causal, kv_valid_len=None, rows=None, tensors=None, **kw):
    o, lse = run_cuda(q, k, v, scale, causal, kv_valid_len, tensors=tensors, **kw)
    o_gpu, lse_gpu = gather_rows(o, lse, rows)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, scale, causal, kv_valid_len=kv_valid_len, rows=rows)
    return compare(o_gpu, lse_gpu, o_ref, lse_ref)


def head_rows(b, h, H, S_q, local_rows):
    return (b * H + h) * S_q + np.asarray(local_rows, dtype=np.int64)


def sampled_rows(seed, B, H, S_q, per_head, full_heads=(), must_include=()):
    """Flat row ids: every row of the heads in ``full_heads`` (pairs (b,h)) and
    ``per_head`` seeded rows of every other head."""
    out = []
    full = set(full_heads)
    for b in range(B):
        for h in range(H):
            if (b, h) in full:
                out.append(head_rows(b, h, H, S_q, np.arange(S_q)))
            else:
                local = si.sample_rows(seed * 1000003 + b * H + h, S_q, per_head, must_include)
                out.append(head_rows(b, h, H, S_q, local))
    return np.concatenate(out)
