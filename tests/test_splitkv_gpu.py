"""Key-split forward and the log-sum-exp merge kernel on GB300, against the
fp64 oracle (attention over all keys, and the oracle's merge of per-chunk
results)."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import io_aware_attention_fwd_gb300 as attn
    attn.build()
    return torch.device("cuda:0")


def run_split(q, k, v, scale, causal, n_splits, kv_valid_len=None, device="cuda:0", rows=None):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    tq, tk, tv = (parity.to_device(x, device) for x in (q, k, v))
    o = torch.full((B, H, S_q, D), float("nan"), dtype=torch.bfloat16, device=device)
    lse = torch.full((B, H, S_q), float("nan"), dtype=torch.float32, device=device)
    kvl = None if kv_valid_len is None else torch.tensor(kv_valid_len, dtype=torch.int32, device=device)
    nbytes = attn.attn_fwd_splitkv_workspace_bytes(B, H, S_q, D, n_splits)
    ws = torch.full((max(nbytes, 16),), 0xFF, dtype=torch.uint8, device=device)  # NaN-filled scratch
    attn.attn_fwd_splitkv(tq, tk, tv, o, lse, B, H, S_q, S_kv, D, scale, causal, kvl, n_splits, ws, nbytes)
    torch.cuda.synchronize()
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK
    return parity.gather_rows(o, lse, rows)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_splits", [2, 5, 16])
def test_splitkv_matches_oracle(dev, D, causal, n_splits):
    q, k, v = si.qkv_bf16(900 + n_splits, 1, 2, 300, 2000, D)
    o, l = run_split(q, k, v, 1 / math.sqrt(D), causal, n_splits)
    o_ref, l_ref = oracle.attention_f64(q, k, v, 1 / math.sqrt(D), causal)
    parity.compare(o, l, o_ref, l_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_with_padding_and_empty_chunks(dev, causal):
    # more chunks than kv tiles, padding lengths 0 / 1 / 129 / 1000: many chunks
    # see no key and must contribute nothing
    valid = [1000, 0, 1, 129]
    q, k, v = si.qkv_bf16(910, 4, 1, 257, 1000, 128)
    for n_splits in (3, 12, 64):
        o, l = run_split(q, k, v, 0.1, causal, n_splits, kv_valid_len=valid)
        o_ref, l_ref = oracle.attention_f64(q, k, v, 0.1, causal, kv_valid_len=valid)
        parity.compare(o, l, o_ref, l_ref)


def test_splitkv_agrees_with_unsplit_kernel(dev):
    import torch
    q, k, v = si.qkv_bf16(920, 2, 4, 512, 4096, 128, q_mult=2.0)
    o1, l1 = run_split(q, k, v, 0.09, True, 7)
    o2, l2 = parity.gather_rows(*parity.run_cuda(q, k, v, 0.09, True))
    # the two paths round P to bf16 against different running maxima, so they
    # agree to the parity bar rather than bit for bit; LSE agrees more tightly
    parity.compare(o1, l1, o2, l2)
    assert np.abs(l1 - l2).max() <= 1e-4
    assert np.linalg.norm(o1 - o2) <= 3e-3 * np.linalg.norm(o2)


def test_decode_shape_sampled_rows(dev):
    # one query pair per head and 32k keys: the shape key splitting exists for
    import io_aware_attention_fwd_gb300 as attn
    B, H, S_q, S_kv, D = 1, 8, 256, 32768, 128
    n = attn.attn_fwd_splitkv_suggest(B, H, S_q, S_kv, D, False)
    assert n > 1
    q, k, v = si.qkv_bf16(930, B, H, S_q, S_kv, D)
    rows = parity.sampled_rows(930, B, H, S_q, 32, must_include=[0, 255])
    o, l = run_split(q, k, v, 1 / math.sqrt(D), False, n, rows=rows)
    o_ref, l_ref = oracle.attention_f64(q, k, v, 1 / math.sqrt(D), False, rows=rows)
    parity.compare(o, l, o_ref, l_ref)


def test_api_picks_split_automatically(dev):
    import io_aware_attention_fwd_gb300 as attn
    q, k, v = si.qkv_bf16(940, 1, 2, 128, 8192, 64)
    t = [parity.to_device(x, dev) for x in (q, k, v)]
    assert attn.attn_fwd_splitkv_suggest(1, 2, 128, 8192, 64, False) > 1
    o, lse = attn.attention_forward(*t)
    o_g, l_g = parity.gather_rows(o, lse)
    o_ref, l_ref = oracle.attention_f64(q, k, v, 1 / 8, False)
    parity.compare(o_g, l_g, o_ref, l_ref)


@pytest.mark.parametrize("D", [64, 128])
def test_merge_kernel_matches_oracle_merge(dev, D):
    """Per-chunk oracle results (as fp32) merged on the GPU equal the oracle's
    merge and the oracle's attention over all keys."""
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S_q, S_kv = 1, 3, 70, 600
    q, k, v = si.qkv_bf16(950 + D, B, H, S_q, S_kv, D)
    cuts = [0, 100, 101, 350, 600]
    parts = [oracle.attention_f64(q, k[:, :, a:b].copy(), v[:, :, a:b].copy(), 0.2, False)
             for a, b in zip(cuts[:-1], cuts[1:])]
    rows = B * H * S_q
    o_parts = np.stack([p[0] for p in parts]).astype(np.float32)
    l_parts = np.stack([p[1] for p in parts]).astype(np.float32)
    # an extra part without keys, and a row where no part has keys
    o_parts = np.concatenate([o_parts, np.zeros((1, rows, D), np.float32)])
    l_parts = np.concatenate([l_parts, np.full((1, rows), -np.inf, np.float32)])
    l_parts[:, 5] = -np.inf
    o_parts[:, 5] = 0
    to = torch.from_numpy(o_parts).to(dev)
    tl = torch.from_numpy(l_parts).to(dev)
    out = torch.full((rows, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((rows,), float("nan"), dtype=torch.float32, device=dev)
    attn.attn_merge(to, tl, o_parts.shape[0], rows, D, out, lse)
    torch.cuda.synchronize()
    o_gpu, l_gpu = parity.gather_rows(out, lse)
    o_ref, l_ref = oracle.merge_f64(o_parts.astype(np.float64), l_parts.astype(np.float64))
    parity.compare(o_gpu, l_gpu, o_ref, l_ref)
    assert np.all(o_gpu[5] == 0) and np.isneginf(l_gpu[5])
    o_full, l_full = oracle.attention_f64(q, k, v, 0.2, False)
    keep = np.ones(rows, bool)
    keep[5] = False
    parity.compare(o_gpu[keep], l_gpu[keep], o_full[keep], l_full[keep])
