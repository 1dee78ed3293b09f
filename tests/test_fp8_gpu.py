"""FP8 (e4m3) forward pass on GB300 against the fp64 oracle.

The oracle computes exact attention of the real inputs q_descale*Q8,
k_descale*K8, v_descale*V8: every e4m3 value is exactly a bf16 value, so the
oracle reads the e4m3 codes widened to bf16, takes scale*q_descale*k_descale as
its scale, and its O is multiplied by v_descale.

Tolerance, derived from the arithmetic (the bf16 bar does not apply):
  * S is exact up to fp32 accumulation, and l sums the unrounded fp32 P, so
    LSE keeps the bf16 path's bar: 1e-3 absolute.
  * P enters P.V as e4m3: round-to-nearest with 3 mantissa bits gives each
    p a relative error of at most 2^-4, close to uniform, RMS 2^-4/sqrt(3) =
    0.036.  For value rows of zero mean the relative RMS error of
    O = sum p~ v / l is the RMS of those per-element errors, 0.036; the bar is
    0.08.  The error of one O element is at most 2^-4 * max|v|, about 0.3 for
    N(0,1) values; the bar is 0.25 on max-abs.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

FP8_MAX_ABS = 0.25
FP8_REL_RMS = 0.08
FP8_LSE_ABS = 1e-3


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import io_aware_attention_fwd_gb300 as attn
    attn.build()
    return torch.device("cuda:0")


def run_fp8(q8, k8, v8, scale, descales, causal, kv_valid_len=None, rows=None, device="cuda:0"):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S_q, D = q8.shape
    S_kv = k8.shape[2]
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)).to(device) for x in (q8, k8, v8))
    o = torch.full((B, H, S_q, D), float("nan"), dtype=torch.bfloat16, device=device)
    lse = torch.full((B, H, S_q), float("nan"), dtype=torch.float32, device=device)
    kvl = None if kv_valid_len is None else torch.tensor(kv_valid_len, dtype=torch.int32, device=device)
    attn.attn_fwd_fp8(tq, tk, tv, o, lse, B, H, S_q, S_kv, D, scale, *descales, causal, kvl)
    torch.cuda.synchronize()
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK
    return parity.gather_rows(o, lse, rows)


def oracle_fp8(q8, k8, v8, scale, descales, causal, kv_valid_len=None, rows=None):
    qd, kd, vd = descales
    o, l = oracle.attention_f64(si.e4m3_bits_to_bf16_bits(q8), si.e4m3_bits_to_bf16_bits(k8),
                                si.e4m3_bits_to_bf16_bits(v8), scale * qd * kd, causal,
                                kv_valid_len=kv_valid_len, rows=rows)
    return o * vd, l


def check(q8, k8, v8, scale, descales, causal, **kw):
    o, l = run_fp8(q8, k8, v8, scale, descales, causal, **kw)
    o_ref, l_ref = oracle_fp8(q8, k8, v8, scale, descales, causal, **kw)
    return parity.compare(o, l, o_ref, l_ref, FP8_MAX_ABS, FP8_REL_RMS, FP8_LSE_ABS)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [128, 256, 300, 1000])
def test_fp8_unit_scales(dev, causal, S):
    q8, k8, v8 = si.qkv_e4m3(1100 + S, 1, 2, S, S, 128)
    check(q8, k8, v8, 1 / math.sqrt(128), (1.0, 1.0, 1.0), causal)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_per_tensor_descales(dev, causal):
    # stored values use the e4m3 range (x16, x16, x64); the descales undo it
    q8, k8, v8 = si.qkv_e4m3(1110, 2, 2, 512, 512, 128, mults=(16.0, 16.0, 64.0))
    err = check(q8, k8, v8, 1 / math.sqrt(128), (1 / 16, 1 / 16, 1 / 64), causal)
    assert err["rel_rms"] < 0.06


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_padding_and_unequal_lengths(dev, causal):
    q8, k8, v8 = si.qkv_e4m3(1120, 3, 1, 200, 700, 128, mults=(8.0, 8.0, 8.0))
    check(q8, k8, v8, 0.1, (0.125, 0.125, 0.125), causal, kv_valid_len=[700, 333, 0])


def test_fp8_8k_sampled_rows(dev):
    q8, k8, v8 = si.qkv_e4m3(1130, 2, 8, 8192, 8192, 128, mults=(16.0, 16.0, 16.0))
    rows = parity.sampled_rows(1130, 2, 8, 8192, 64, must_include=[0, 8191])
    for causal in (False, True):
        check(q8, k8, v8, 1 / math.sqrt(128), (1 / 16, 1 / 16, 1 / 16), causal, rows=rows)


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_bench_size_32k_sampled_rows(dev, causal):
    """The e4m3 workload the benchmark times at 32k (B=1, H=32, S=32768,
    D=128, seed 6, N(0,1) x 16 rounded to e4m3 on the device, descales 1/16,
    one launch over all heads), checked on seeded rows of every head,
    including the first and last positions."""
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S, D, seed, m8 = 1, 32, 32768, 128, 6, 16.0
    q, k, v = (si.normal_e4m3_torch(seed, tid, B * H * S * D, m8, device=dev).view(B, H, S, D)
               for tid in (si.TID_Q, si.TID_K, si.TID_V))
    o = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    scale, d8 = 1 / math.sqrt(D), 1 / m8
    attn.attn_fwd_fp8(q, k, v, o, lse, B, H, S, S, D, scale, d8, d8, d8, causal, None)
    torch.cuda.synchronize()
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK
    rows = parity.sampled_rows(seed * 3 + int(causal), B, H, S, 8, must_include=[0, S // 2, S - 1])
    og, lg = parity.gather_rows(o, lse, rows)
    host = [x.view(torch.uint8).cpu().numpy() for x in (q, k, v)]
    o_ref, l_ref = oracle_fp8(*host, scale, (d8, d8, d8), causal, rows=rows)
    parity.compare(og, lg, o_ref, l_ref, FP8_MAX_ABS, FP8_REL_RMS, FP8_LSE_ABS)


def test_fp8_close_to_bf16_path_on_the_same_values(dev):
    # the same (e4m3-representable) values through the bf16 kernel: the two
    # differ only by P's rounding (e4m3 vs bf16)
    q8, k8, v8 = si.qkv_e4m3(1140, 1, 4, 640, 640, 128)
    o8, l8 = run_fp8(q8, k8, v8, 0.09, (1.0, 1.0, 1.0), True)
    bf = [si.e4m3_bits_to_bf16_bits(x) for x in (q8, k8, v8)]
    o16, l16 = parity.gather_rows(*parity.run_cuda(*bf, 0.09, True))
    assert np.abs(l8 - l16).max() <= 1e-4
    parity.compare(o8, l8, o16, l16, FP8_MAX_ABS, FP8_REL_RMS, FP8_LSE_ABS)
