"""Backward pass on GB300 against the fp64 oracle's gradients.

The GPU gradients come from the library's own forward outputs (O, LSE), as a
training step would use them.  Tolerance, derived from the arithmetic:
P and dS enter the tensor-core products as bf16 (relative rounding error
2^-9, RMS about 1.1e-3 each), Delta is formed from the bf16 O, and every
product accumulates in fp32; the expected relative RMS error of dQ, dK and dV
is a few 1e-3.  The bar is relative RMS 2e-2 for each gradient and an
absolute error of at most 5e-2 times the largest reference magnitude.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

REL_RMS = 2e-2
MAX_ABS_REL = 5e-2


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import io_aware_attention_fwd_gb300 as attn
    attn.build()
    return torch.device("cuda:0")


def run_bwd(bits, scale, causal, kv_valid_len=None, device="cuda:0"):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    q, k, v, d_o = (parity.to_device(x, device) for x in bits)
    kvl = None if kv_valid_len is None else torch.tensor(kv_valid_len, dtype=torch.int32, device=device)
    o, lse = attn.attention_forward(q, k, v, scale=scale, causal=causal, kv_valid_len=kvl, n_splits=1)
    dq, dk, dv = attn.attention_backward(q, k, v, o, lse, d_o, scale=scale, causal=causal, kv_valid_len=kvl)
    torch.cuda.synchronize()
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK
    return [x.float().cpu().numpy().astype(np.float64) for x in (dq, dk, dv)]


def compare_grads(got, ref):
    errs = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(g)), name
        scale_r = max(np.abs(r).max(), 1e-6)
        nrm = max(np.linalg.norm(r), 1e-30)
        errs[name] = (float(np.linalg.norm(g - r) / nrm), float(np.abs(g - r).max() / scale_r))
        if np.linalg.norm(r) == 0:
            assert np.all(g == 0), name
            continue
        assert errs[name][0] <= REL_RMS, (name, errs)
        assert errs[name][1] <= MAX_ABS_REL, (name, errs)
    return errs


def check(seed, B, H, S_q, S_kv, D, causal, kv_valid_len=None, q_mult=1.0, scale=None):
    bits = [si.normal_bf16(seed, t, B * H * n * D, q_mult if t == si.TID_Q else 1.0).reshape(B, H, n, D)
            for t, n in ((si.TID_Q, S_q), (si.TID_K, S_kv), (si.TID_V, S_kv), (5, S_q))]
    scale = scale or 1 / math.sqrt(D)
    got = run_bwd(bits, scale, causal, kv_valid_len)
    ref = oracle.attention_bwd_f64(*bits, scale, causal, kv_valid_len=kv_valid_len)
    return compare_grads(got, ref)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [128, 256, 384])
def test_bwd_square(dev, D, causal, S):
    check(1200 + S, 1, 2, S, S, D, causal)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S_q,S_kv", [(200, 200), (100, 300), (300, 100), (129, 257)])
def test_bwd_ragged_and_unequal(dev, D, causal, S_q, S_kv):
    check(1210 + S_q + S_kv, 2, 1, S_q, S_kv, D, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_padding(dev, causal):
    check(1220, 4, 1, 300, 300, 128, causal, kv_valid_len=[300, 77, 0, 129])


def test_bwd_peaked(dev):
    check(1230, 1, 2, 256, 256, 128, True, q_mult=4.0)


def test_bwd_2k(dev):
    check(1240, 1, 4, 2048, 2048, 128, True)
    check(1241, 2, 2, 1024, 1024, 64, False)


def test_bwd_allocates_only_its_workspace(dev):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S, D = 1, 2, 512, 128
    t = [parity.to_device(si.normal_bf16(1250, i, B * H * S * D).reshape(B, H, S, D), dev) for i in (1, 2, 3, 5)]
    o, lse = attn.attention_forward(*t[:3], n_splits=1)
    dq, dk, dv = (torch.empty_like(x) for x in t[:3])
    nbytes = attn.attn_bwd_workspace_bytes(B, H, S, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    attn.attn_bwd(*t[:3], o, lse, t[3], dq, dk, dv, B, H, S, S, D, 0.1, True, None, ws, nbytes)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    attn.attn_bwd(*t[:3], o, lse, t[3], dq, dk, dv, B, H, S, S, D, 0.1, True, None, ws, nbytes)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free0


@pytest.mark.parametrize("shape", ["b1_h32_s8192_d128", "b4_h16_s1024_d64"])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_bench_size_sampled_heads(dev, causal, shape):
    """The backward workloads the benchmark times (B=1, H=32, S=8192, D=128
    and B=4, H=16, S=1024, D=64; seed 8, inputs drawn on the device, one
    attn_bwd call over all heads), checked on two seeded heads against the
    oracle's full gradients of those heads."""
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S, D = {"b1_h32_s8192_d128": (1, 32, 8192, 128), "b4_h16_s1024_d64": (4, 16, 1024, 64)}[shape]
    seed = 8
    scale = 1 / math.sqrt(D)
    q, k, v = si.qkv_bf16_torch(seed, B, H, S, S, D, device=dev)
    d_o = si.normal_bf16_torch(seed, 5, B * H * S * D, device=dev).view(B, H, S, D)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    attn.attn_fwd(q, k, v, o, lse, B, H, S, S, D, scale, causal, None)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = attn.attn_bwd_workspace_bytes(B, H, S, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    attn.attn_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B, H, S, S, D, scale, causal, None, ws, nbytes)
    torch.cuda.synchronize()
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK
    # two seeded (batch, head) pairs; the first batch always included
    picks = [int(x) for x in si.sample_rows(seed * 7 + int(causal), B * H, 2, must_include=(0,))]
    for bh in picks:
        b, h = divmod(bh, H)
        bits = lambda t: t[b:b + 1, h:h + 1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        ref = oracle.attention_bwd_f64(bits(q), bits(k), bits(v), bits(d_o), scale, causal)
        got = [x[b:b + 1, h:h + 1].float().cpu().numpy().astype(np.float64) for x in (dq, dk, dv)]
        compare_grads(got, ref)


def test_bwd_causal_partial_head_group(dev):
    """Causal CTAs run in groups of heads sized so that a group's fp32 dQ
    accumulators fit in 32 MiB: at 5000 tokens and D = 128 that is 8 heads,
    so 12 heads form one group of 8 and one of 4 (and the last tile is
    ragged).  Heads from both groups are checked against the oracle."""
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S, D = 1, 12, 5000, 128
    assert 16 * S * D * 4 > 32 << 20 >= 8 * S * D * 4
    seed = 1260
    scale = 1 / math.sqrt(D)
    q, k, v = si.qkv_bf16_torch(seed, B, H, S, S, D, device=dev)
    d_o = si.normal_bf16_torch(seed, 5, B * H * S * D, device=dev).view(B, H, S, D)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    attn.attn_fwd(q, k, v, o, lse, B, H, S, S, D, scale, True, None)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = attn.attn_bwd_workspace_bytes(B, H, S, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    attn.attn_bwd(q, k, v, o, lse, d_o, dq, dk, dv, B, H, S, S, D, scale, True, None, ws, nbytes)
    torch.cuda.synchronize()
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK
    for h in (0, 7, 8, 11):  # first and last head of each group
        bits = lambda t: t[:, h:h + 1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        ref = oracle.attention_bwd_f64(bits(q), bits(k), bits(v), bits(d_o), scale, True)
        got = [x[:, h:h + 1].float().cpu().numpy().astype(np.float64) for x in (dq, dk, dv)]
        compare_grads(got, ref)
