"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on GB300.

The five workloads of the target (small, 1k, 4k causal, 8k padded, 32k causal)
plus edge cases: ragged tails, S_q != S_kv, key-padding lengths around tile
boundaries, empty inputs, peaked softmax, determinism, no device allocation,
and the watchdog's failure path.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

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


def qkv(seed, B, H, S_q, S_kv, D, q_mult=1.0, k_mult=1.0):
    return si.qkv_bf16(seed, B, H, S_q, S_kv, D, q_mult, k_mult)


# --- the five workloads --------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_c1_small_all_rows(dev, causal):
    q, k, v = qkv(1, 1, 2, 128, 128, 64)
    parity.check_against_oracle(q, k, v, 1 / 8, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("peaked", [False, True])
def test_c2_1k_all_rows(dev, causal, peaked):
    seed, mult = (3, 8.0) if peaked else (2, 1.0)
    q, k, v = qkv(seed, 4, 16, 1024, 1024, 64, q_mult=mult)
    parity.check_against_oracle(q, k, v, 1 / 8, causal)


@pytest.fixture(scope="module")
def c3(dev):
    q, k, v = qkv(4, 1, 32, 4096, 4096, 128)
    return q, k, v, tuple(parity.to_device(x, dev) for x in (q, k, v))


@pytest.mark.parametrize("causal", [True, False])
def test_c3_4k_d128(c3, causal):
    q, k, v, t = c3
    heads = [(0, h) for h in si.sample_rows(40, 32, 4)]
    rows = parity.sampled_rows(4, 1, 32, 4096, 256, full_heads=heads, must_include=[0, 4095])
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(128), causal, rows=rows, tensors=t)


def test_c4_8k_padded(dev):
    q, k, v = qkv(5, 2, 32, 8192, 8192, 128)
    rows = parity.sampled_rows(5, 2, 32, 8192, 256, must_include=[0, 4999, 5000, 8191])
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(128), False, kv_valid_len=[8192, 5000], rows=rows)


@pytest.fixture(scope="module")
def c5(dev):
    S = 32768
    q, k, v = qkv(6, 1, 32, S, S, 128, q_mult=2.0, k_mult=2.0)
    return q, k, v, tuple(parity.to_device(x, dev) for x in (q, k, v))


@pytest.mark.parametrize("causal", [True, False])
def test_c5_32k(c5, causal):
    q, k, v, t = c5
    S = 32768
    rows = parity.sampled_rows(6, 1, 32, S, 128, must_include=[0, 1, 127, 128, S // 2, S - 1])
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(128), causal, rows=rows, tensors=t)


@pytest.mark.parametrize("D,S,H", [(128, 9000, 16), (64, 17000, 16)])
def test_long_causal_host_schedule_ragged(dev, D, S, H):
    # Causal launches whose heads' K and V exceed 64 MB run the units in a
    # host-computed order (a per-CTA unit table); here with a ragged last
    # tile and a head count that does not divide the SM count.
    assert H * S * D * 2 * 2 > 64 << 20
    q, k, v = qkv(950 + D, 1, H, S, S, D)
    rows = parity.sampled_rows(950 + D, 1, H, S, 64, must_include=[0, 1, 255, 256, S // 2, S - 129, S - 1])
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(D), True, rows=rows)


@pytest.mark.parametrize("D,S_q,S_kv,H", [(128, 3000, 20000, 16), (128, 12000, 8200, 32)])
def test_long_causal_host_schedule_unequal_lengths(dev, D, S_q, S_kv, H):
    # The host-computed order with S_q != S_kv: the causal mask is aligned top
    # left (key j is allowed for query i when j <= i), so with S_kv > S_q the
    # last keys are never seen, and with S_q > S_kv the rows past S_kv see
    # every key.
    import io_aware_attention_fwd_gb300 as attn
    assert H * S_kv * D * 2 * 2 > 64 << 20
    assert attn.attn_fwd_schedule(1, H, S_q, S_kv, D, 2, 152) is not None
    q, k, v = qkv(960 + S_q % 97, 1, H, S_q, S_kv, D)
    rows = parity.sampled_rows(960 + S_q % 97, 1, H, S_q, 48,
                               must_include=[0, 1, 127, 128, min(S_q, S_kv) - 1, S_q - 1])
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(D), True, rows=rows)



@pytest.mark.parametrize("D,S,H", [(128, 8192, 32), (64, 17000, 16)])
def test_host_schedule_is_bit_identical_to_the_formula_order(dev, D, S, H):
    # The host-built order only changes which CTA computes a unit and when;
    # every row's arithmetic is the same.  A launch with kv_valid_len = S_kv
    # for every batch computes the same attention but keeps the formula
    # (longest-first) order, so O and LSE must agree bit for bit.
    import torch
    import io_aware_attention_fwd_gb300 as attn
    assert attn.attn_fwd_schedule(1, H, S, S, D, 2, 152) is not None
    q, k, v = (parity.to_device(x, dev) for x in qkv(970 + D, 1, H, S, S, D))
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty((1, H, S), dtype=torch.float32, device=dev)
    l2 = torch.empty_like(l1)
    full = torch.tensor([S], dtype=torch.int32, device=dev)
    attn.attn_fwd(q, k, v, o1, l1, 1, H, S, S, D, 1 / math.sqrt(D), True, None)
    attn.attn_fwd(q, k, v, o2, l2, 1, H, S, S, D, 1 / math.sqrt(D), True, full)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)



def test_host_schedule_is_bit_identical_to_the_formula_order_e4m3(dev):
    # The same check for the e4m3 kernel (its K + V here: 98 MB > 64 MiB).
    import torch
    import io_aware_attention_fwd_gb300 as attn
    B, H, S, D = 1, 32, 12000, 128
    assert attn.attn_fwd_schedule(B, H, S, S, D, 1, 152) is not None
    q, k, v = (si.normal_e4m3_torch(980, tid, B * H * S * D, 16.0, device=dev).view(B, H, S, D)
               for tid in (si.TID_Q, si.TID_K, si.TID_V))
    o1 = torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev)
    o2 = torch.empty_like(o1)
    l1 = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    l2 = torch.empty_like(l1)
    full = torch.tensor([S], dtype=torch.int32, device=dev)
    ds = 1.0 / 16.0
    attn.attn_fwd_fp8(q, k, v, o1, l1, B, H, S, S, D, 1 / math.sqrt(D), ds, ds, ds, True, None)
    attn.attn_fwd_fp8(q, k, v, o2, l2, B, H, S, S, D, 1 / math.sqrt(D), ds, ds, ds, True, full)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


# --- edge cases ----------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 127, 129, 200, 255, 257, 383, 640])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(dev, D, S, causal):
    q, k, v = qkv(100 + S, 1, 3, S, S, D)
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(D), causal)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S_q,S_kv", [(100, 300), (300, 100), (1, 513), (513, 1), (256, 640)])
@pytest.mark.parametrize("causal", [False, True])
def test_unequal_query_and_key_lengths(dev, D, S_q, S_kv, causal):
    q, k, v = qkv(200 + S_q + S_kv, 2, 2, S_q, S_kv, D)
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(D), causal)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_around_tile_edges(dev, D, causal):
    valid = [0, 1, 127, 128, 129, 300, 500]
    q, k, v = qkv(300, len(valid), 2, 300, 300, D)
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(D), causal, kv_valid_len=valid)


def test_padding_length_out_of_range_is_clamped(dev):
    q, k, v = qkv(301, 3, 1, 64, 200, 64)
    o1, l1 = parity.run_cuda(q, k, v, 0.125, False, kv_valid_len=[-7, 10**6, 200])
    o2, l2 = parity.run_cuda(q, k, v, 0.125, False, kv_valid_len=[0, 200, 200])
    import torch
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("D", [64, 128])
def test_peaked_softmax_rescaling(dev, D):
    # Q x 8 makes every row nearly one-hot; Q, K x 2 stresses the max-growth path.
    q, k, v = qkv(400, 2, 4, 700, 700, D, q_mult=8.0)
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(D), False)
    q, k, v = qkv(401, 2, 4, 700, 700, D, q_mult=2.0, k_mult=2.0)
    parity.check_against_oracle(q, k, v, 1 / math.sqrt(D), True)


def test_increasing_scores_force_every_rescale(dev):
    # Scores grow with the key index, so the running max rises on every tile.
    S, D = 1024, 64
    q = np.zeros((1, 1, S, D), np.uint16)
    q[..., 0] = 0x3F80  # 1.0
    keys = si.f32_to_bf16_bits(np.linspace(0.0, 60.0, S, dtype=np.float32))
    k = np.zeros((1, 1, S, D), np.uint16)
    k[0, 0, :, 0] = keys
    v = si.normal_bf16(402, si.TID_V, S * D).reshape(1, 1, S, D)
    for causal in (False, True):
        parity.check_against_oracle(q, k, v, 1.0, causal)


def test_large_head_count_small_sequence(dev):
    q, k, v = qkv(500, 8, 64, 64, 64, 64)
    parity.check_against_oracle(q, k, v, 0.125, True)


def test_empty_keys_and_queries(dev):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    q, _, _ = qkv(600, 2, 2, 50, 1, 64)
    e = np.zeros((2, 2, 0, 64), np.uint16)
    parity.check_against_oracle(q, e, e, 0.125, False)
    # S_q == 0: nothing is written
    z = torch.zeros((1, 1, 0, 64), dtype=torch.bfloat16, device=dev)
    kk = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1,), dtype=torch.float32, device=dev)
    attn.attn_fwd(kk, kk, kk, kk, lse, 1, 1, 0, 8, 64, 0.125, False)
    torch.cuda.synchronize()


def test_deterministic(dev):
    q, k, v = qkv(700, 2, 8, 1000, 1000, 128)
    t = tuple(parity.to_device(x, dev) for x in (q, k, v))
    o1, l1 = parity.run_cuda(q, k, v, 0.1, True, tensors=t)
    o2, l2 = parity.run_cuda(q, k, v, 0.1, True, tensors=t)
    import torch
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("B,H,S,graph", [(4, 16, 640, True), (1, 32, 640, True), (2, 8, 640, False),
                                         (1, 32, 8192, True)])
def test_host_forward_equals_one_launch(dev, B, H, S, graph):
    # HostForward runs a step as attn_fwd calls on contiguous pieces of the
    # batch, with pinned copies on side streams (captured as a CUDA graph or
    # eager): each row's O and LSE must equal one launch over the whole batch
    import torch
    import io_aware_attention_fwd_gb300 as attn
    D = 64 if B == 4 else 128
    if S > 640:  # long enough for tapered pieces (small first and last ones)
        from io_aware_attention_fwd_gb300.host import plan_tapered
        assert plan_tapered(B, H, S, D) is not None
    q, k, v = (parity.to_device(x, dev) for x in qkv(900 + B, B, H, S, S, D))
    kvl = torch.tensor([640, 333], dtype=torch.int32, device=dev) if B == 2 else None
    hf = attn.HostForward(B, H, S, S, D, modes=(False, True), scale=0.1, kv_valid_len=kvl, device=dev, graph=graph)
    for dst, src in zip(hf.host_inputs, (q, k, v)):
        dst.copy_(src.cpu())
    for _ in range(2):  # a replay reuses every buffer
        hf.run()
    torch.cuda.synchronize()
    for causal in (False, True):
        o1, l1 = torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device=dev)
        attn.attn_fwd(q, k, v, o1, l1, B, H, S, S, D, 0.1, causal, kvl)
        torch.cuda.synchronize()
        ho, hl = hf.host_outputs[causal]
        assert torch.equal(o1.cpu(), ho) and torch.equal(l1.cpu(), hl)


def test_side_stream_and_api_wrapper(dev):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    q, k, v = qkv(800, 1, 4, 300, 300, 128)
    t = [parity.to_device(x, dev) for x in (q, k, v)]
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        o, lse = attn.attention_forward(*t, causal=True)
    s.synchronize()
    o_gpu, l_gpu = parity.gather_rows(o, lse)
    import oracle
    o_ref, l_ref = oracle.attention_f64(q, k, v, 1 / math.sqrt(128), True)
    parity.compare(o_gpu, l_gpu, o_ref, l_ref)


def test_library_allocates_no_device_memory(dev):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    q, k, v = qkv(900, 1, 8, 4096, 4096, 128)
    t = [parity.to_device(x, dev) for x in (q, k, v)]
    o = torch.empty_like(t[0])
    lse = torch.empty((1, 8, 4096), dtype=torch.float32, device=dev)
    # The first call loads the module.  Its device image carries the fixed
    # 32 MiB scratch array of attn_fwd_splitkv_static on every device that
    # loads it, so device memory is measured only after that first call.
    attn.attn_fwd(*t, o, lse, 1, 8, 4096, 4096, 128, 0.1, True)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for causal in (False, True):
        attn.attn_fwd(*t, o, lse, 1, 8, 4096, 4096, 128, 0.1, causal)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    # nothing was allocated: 8 heads x 4096^2 fp32 scores alone would be 512 MiB
    assert free1 == free0
    assert torch.cuda.memory_allocated(dev) == alloc0


def test_watchdog_gives_up_and_context_survives(dev):
    import torch
    import io_aware_attention_fwd_gb300 as attn
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK
    assert attn.attn_watchdog_selftest(2_000_000) == attn.ATTN_ERR_TIMEOUT  # 2 ms limit
    assert attn.attn_fwd_debug_status() == attn.ATTN_OK  # the word was cleared
    # the context is still usable
    q, k, v = qkv(1000, 1, 2, 256, 256, 64)
    parity.check_against_oracle(q, k, v, 0.125, True)
    torch.cuda.synchronize()
