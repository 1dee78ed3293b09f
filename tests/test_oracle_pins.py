"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks a value the pages print, a closed form, an invariant, or an
independent library routine (torch's float64 CPU scaled_dot_product_attention).
"""
from __future__ import annotations

import math
from pathlib import Path

import numpy as np
import pytest

import oracle
import seeded_inputs as si

GOLDEN = Path(__file__).resolve().parent / "golden"
BF16_ONE = 0x3F80


def bits(seed, shape, tid=si.TID_Q, mult=1.0):
    n = int(np.prod(shape))
    return si.normal_bf16(seed, tid, n, mult).reshape(shape)


def f64(b):
    return si.bf16_bits_to_f32(b).astype(np.float64)


def allowed_mask(S_q, S_kv, causal, valid):
    j = np.arange(S_kv)[None, :]
    i = np.arange(S_q)[:, None]
    m = np.broadcast_to(j < valid, (S_q, S_kv))
    if causal:
        m = m & (j <= i)
    return m


# --- "Attention memory" page, "Formula" + "Worked example" -------------------

def test_score_buffer_worked_example():
    rows = [l.split() for l in (GOLDEN / "score_buffer_worked_example.txt").read_text().splitlines()
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    sizes = []
    for B, H, s, e, printed in rows:
        nbytes = oracle.score_buffer_bytes(int(B), int(H), int(s), int(e))
        sizes.append(nbytes)
        assert f"{nbytes / 1e9:.2f}" == printed
        # a binary (GiB) divisor would not reproduce the printed figure
        assert f"{nbytes / 2**30:.2f}" != printed
    assert sizes == [1_073_741_824, 4_294_967_296]
    assert sizes[1] == 4 * sizes[0]  # "four times as much for twice the length"


def test_score_buffer_linear_in_batch_and_heads():
    base = oracle.score_buffer_bytes(1, 1, 1000, 2)
    assert base == 2_000_000
    assert oracle.score_buffer_bytes(3, 5, 1000, 2) == 15 * base
    assert oracle.score_buffer_bytes(1, 1, 1000, 4) == 2 * base


# --- softmax and masking invariants -------------------------------------------

@pytest.mark.parametrize("causal,valid", [(False, 8), (True, 8), (False, 5), (True, 3)])
def test_probabilities_sum_to_one(causal, valid):
    # With V = identity (D = S_kv), output row i is the probability row of i.
    S = 8
    q = bits(11, (1, 1, S, S))
    k = bits(11, (1, 1, S, S), si.TID_K)
    v = np.zeros((1, 1, S, S), np.uint16)
    v[0, 0, np.arange(S), np.arange(S)] = BF16_ONE
    o, _ = oracle.attention_f64(q, k, v, 0.5, causal, kv_valid_len=[valid])
    mask = allowed_mask(S, S, causal, valid)
    assert np.all(o >= 0)
    np.testing.assert_allclose(o.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(o[~mask] == 0.0)          # masked keys get exactly zero weight
    assert np.all(o[mask] > 0.0)


def test_constant_v_gives_constant_o():
    B, H, S, D = 2, 3, 17, 8
    q, k = bits(12, (B, H, S, D)), bits(12, (B, H, S, D), si.TID_K)
    row = si.f32_to_bf16_bits(np.linspace(-3, 3, D).astype(np.float32))
    v = np.broadcast_to(row, (B, H, S, D)).copy()
    for causal in (False, True):
        o, _ = oracle.attention_f64(q, k, v, 0.3, causal, kv_valid_len=[17, 4])
        np.testing.assert_allclose(o, np.broadcast_to(f64(row), o.shape), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_is_mean_of_allowed_v(causal):
    B, H, S_q, S_kv, D = 2, 2, 9, 12, 8
    q = np.zeros((B, H, S_q, D), np.uint16)
    k, v = bits(13, (B, H, S_kv, D), si.TID_K), bits(13, (B, H, S_kv, D), si.TID_V)
    valid = [12, 5]
    o, lse = oracle.attention_f64(q, k, v, 0.125, causal, kv_valid_len=valid)
    o = o.reshape(B, H, S_q, D)
    lse = lse.reshape(B, H, S_q)
    for b in range(B):
        m = allowed_mask(S_q, S_kv, causal, valid[b])
        for h in range(H):
            for i in range(S_q):
                sel = f64(v[b, h])[m[i]]
                np.testing.assert_allclose(o[b, h, i], sel.mean(axis=0), rtol=1e-12, atol=1e-14)
                assert lse[b, h, i] == pytest.approx(math.log(m[i].sum()), abs=1e-14)


def test_causal_row0_is_v0():
    B, H, S, D = 1, 4, 10, 16
    q, k, v = (bits(14, (B, H, S, D), t) for t in (si.TID_Q, si.TID_K, si.TID_V))
    scale = 0.25
    o, lse = oracle.attention_f64(q, k, v, scale, True)
    o = o.reshape(B, H, S, D)
    lse = lse.reshape(B, H, S)
    for h in range(H):
        np.testing.assert_array_equal(o[0, h, 0], f64(v[0, h, 0]))
        exact = scale * float(np.dot(f64(q[0, h, 0]), f64(k[0, h, 0])))
        assert lse[0, h, 0] == pytest.approx(exact, rel=1e-15, abs=1e-15)


def test_key_permutation_equivariance():
    B, H, S_q, S_kv, D = 1, 2, 7, 13, 8
    q, k, v = (bits(15, (B, H, n, D), t) for n, t in
               ((S_q, si.TID_Q), (S_kv, si.TID_K), (S_kv, si.TID_V)))
    perm = np.random.default_rng(0).permutation(S_kv)
    o1, l1 = oracle.attention_f64(q, k, v, 0.4, False)
    o2, l2 = oracle.attention_f64(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14, atol=1e-14)
    # and a permutation is not the identity on the output of a causal call
    o3, _ = oracle.attention_f64(q, k[:, :, perm], v[:, :, perm], 0.4, True)
    o4, _ = oracle.attention_f64(q, k, v, 0.4, True)
    assert not np.allclose(o3, o4)


@pytest.mark.parametrize("causal", [False, True])
def test_padding_equals_truncation(causal):
    B, H, S, D = 1, 2, 16, 8
    q, k, v = (bits(16, (B, H, S, D), t) for t in (si.TID_Q, si.TID_K, si.TID_V))
    n = 11
    o1, l1 = oracle.attention_f64(q, k, v, 0.3, causal, kv_valid_len=[n])
    o2, l2 = oracle.attention_f64(q, k[:, :, :n].copy(), v[:, :, :n].copy(), 0.3, causal)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_one_hot_peak_selects_value_row():
    # q_0 = 8 * e_0 and k_5 = 8 * e_0: score 64*scale on key 5, 0 elsewhere.
    S, D = 12, 8
    q = np.zeros((1, 1, 1, D), np.uint16)
    k = np.zeros((1, 1, S, D), np.uint16)
    q[0, 0, 0, 0] = 0x4100  # 8.0
    k[0, 0, 5, 0] = 0x4100
    v = bits(17, (1, 1, S, D), si.TID_V)
    o, lse = oracle.attention_f64(q, k, v, 1.0, False)
    w5 = 1.0 / (1.0 + (S - 1) * math.exp(-64.0))
    expect = w5 * f64(v[0, 0, 5]) + (1 - w5) / (S - 1) * np.delete(f64(v[0, 0]), 5, axis=0).sum(0)
    np.testing.assert_allclose(o[0], expect, rtol=1e-13, atol=1e-15)
    assert lse[0] == pytest.approx(64.0 + math.log1p((S - 1) * math.exp(-64.0)), abs=1e-13)


def test_logit_shift_moves_lse_only():
    # Append a column of ones to q and a column of alpha to k: every score gains
    # scale*alpha, so O is unchanged and LSE moves by exactly scale*alpha.
    B, H, S, D = 1, 2, 9, 7
    q, k, v = (bits(18, (B, H, S, D), t) for t in (si.TID_Q, si.TID_K, si.TID_V))
    alpha_bits, alpha = 0x4040, 3.0  # 3.0 in bf16
    q2 = np.concatenate([q, np.full((B, H, S, 1), BF16_ONE, np.uint16)], axis=-1)
    k2 = np.concatenate([k, np.full((B, H, S, 1), alpha_bits, np.uint16)], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, S, 1), np.uint16)], axis=-1)
    for causal in (False, True):
        o1, l1 = oracle.attention_f64(q, k, v, 0.5, causal)
        o2, l2 = oracle.attention_f64(q2, k2, v2, 0.5, causal)
        np.testing.assert_allclose(o2[:, :D], o1, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(l2, l1 + 0.5 * alpha, rtol=0, atol=1e-12)


def test_single_key_is_exact_for_bf16_extremes():
    # One allowed key: weight 1, so O is that value row bit for bit, and LSE is
    # the single score.  Covers subnormal, large and negative bf16 patterns.
    pats = np.array([0x0001, 0x8001, 0x7F7F, 0xFF7F, 0x3F80, 0xBF80, 0x0080, 0x4049], np.uint16)
    D = pats.size
    q = np.zeros((1, 1, 1, D), np.uint16)
    q[0, 0, 0, 0] = BF16_ONE
    k = np.zeros((1, 1, 1, D), np.uint16)
    k[0, 0, 0, 0] = 0x4000  # 2.0
    v = pats.reshape(1, 1, 1, D)
    o, lse = oracle.attention_f64(q, k, v, 0.75, False)
    np.testing.assert_array_equal(o[0], f64(pats))
    assert lse[0] == 1.5


def test_rows_with_no_allowed_key():
    B, H, S, D = 2, 1, 6, 4
    q, k, v = (bits(19, (B, H, S, D), t) for t in (si.TID_Q, si.TID_K, si.TID_V))
    o, lse = oracle.attention_f64(q, k, v, 0.5, True, kv_valid_len=[0, 6])
    o = o.reshape(B, H, S, D)
    lse = lse.reshape(B, H, S)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))
    # no keys at all
    e = np.zeros((B, H, 0, D), np.uint16)
    o, lse = oracle.attention_f64(q, e, e, 0.5, False)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_row_subset_and_threads_match_full():
    B, H, S, D = 2, 3, 33, 16
    q, k, v = (bits(20, (B, H, S, D), t) for t in (si.TID_Q, si.TID_K, si.TID_V))
    o, lse = oracle.attention_f64(q, k, v, 0.25, True, kv_valid_len=[33, 20], threads=1)
    rows = np.array([0, 5, 32, 33, 100, B * H * S - 1])
    o2, l2 = oracle.attention_f64(q, k, v, 0.25, True, kv_valid_len=[33, 20], rows=rows, threads=4)
    np.testing.assert_array_equal(o2, o[rows])
    np.testing.assert_array_equal(l2, lse[rows])


def test_rejects_bad_rows():
    q = np.zeros((1, 1, 4, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle.attention_f64(q, q, q, 1.0, False, rows=[4])


# --- an independent library routine ------------------------------------------

@pytest.mark.parametrize("B,H,S_q,S_kv,D,causal,valid", [
    (1, 2, 16, 16, 64, False, None),
    (2, 2, 19, 19, 64, True, None),
    (2, 1, 13, 21, 32, True, [21, 9]),     # S_q != S_kv, causal top-left
    (2, 3, 24, 17, 128, False, [17, 3]),
    (1, 1, 30, 12, 16, True, [7]),         # rows beyond the last key
])
def test_matches_torch_sdpa_float64(B, H, S_q, S_kv, D, causal, valid):
    torch = pytest.importorskip("torch")
    q = bits(21, (B, H, S_q, D), si.TID_Q, 2.0)
    k = bits(21, (B, H, S_kv, D), si.TID_K, 2.0)
    v = bits(21, (B, H, S_kv, D), si.TID_V)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attention_f64(q, k, v, scale, causal, kv_valid_len=valid)
    tq, tk, tv = (torch.from_numpy(f64(x)) for x in (q, k, v))
    vl = valid if valid is not None else [S_kv] * B
    mask = torch.stack([torch.from_numpy(np.array(allowed_mask(S_q, S_kv, causal, vl[b]))) for b in range(B)])
    mask = mask[:, None].expand(B, H, S_q, S_kv)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(o.reshape(B, H, S_q, D), ref.numpy(), rtol=1e-11, atol=1e-12)
    logits = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
    ref_lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
    np.testing.assert_allclose(lse.reshape(B, H, S_q), ref_lse.numpy(), rtol=1e-12, atol=1e-12)


# --- merge of results over disjoint key sets ----------------------------------

@pytest.mark.parametrize("cuts", [[0, 5, 17], [0, 1, 2, 17], [0, 16, 17]])
def test_merge_of_key_chunks_equals_full_attention(cuts):
    # Attention over keys [a, b) for consecutive chunks, merged, equals attention
    # over all keys (non-causal, so a chunk is a plain slice of K and V).
    B, H, S_q, S_kv, D = 2, 2, 9, 17, 8
    q, k, v = (bits(50, (B, H, n, D), t) for n, t in ((S_q, si.TID_Q), (S_kv, si.TID_K), (S_kv, si.TID_V)))
    o_full, l_full = oracle.attention_f64(q, k, v, 0.35, False)
    parts = [oracle.attention_f64(q, k[:, :, a:b].copy(), v[:, :, a:b].copy(), 0.35, False)
             for a, b in zip(cuts[:-1], cuts[1:])]
    o, l = oracle.merge_f64([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, o_full, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, l_full, rtol=1e-13, atol=1e-13)


def test_merge_closed_forms():
    o1 = np.array([[1.0, 2.0], [3.0, 4.0]])
    o2 = np.array([[5.0, 6.0], [7.0, 8.0]])
    # equal weights -> the average; LSE gains ln 2
    o, l = oracle.merge_f64([o1, o2], [[0.5, -1.0], [0.5, -1.0]])
    np.testing.assert_allclose(o, (o1 + o2) / 2)
    np.testing.assert_allclose(l, [0.5 + math.log(2), -1.0 + math.log(2)])
    # a part without keys (-inf) has no weight; all parts empty -> 0 / -inf
    o, l = oracle.merge_f64([o1, o2], [[-np.inf, -np.inf], [2.0, -np.inf]])
    np.testing.assert_array_equal(o[0], o2[0])
    assert l[0] == 2.0 and np.isneginf(l[1]) and np.all(o[1] == 0)
    # one part is the identity
    o, l = oracle.merge_f64([o1], [[0.25, 7.0]])
    np.testing.assert_array_equal(o, o1)
    np.testing.assert_array_equal(l, [0.25, 7.0])


@pytest.mark.parametrize("causal", [False, True])
def test_matches_extended_precision_brute_force(causal):
    """Tiny problems (S <= 16) evaluated directly in numpy's long double, one
    sum at a time: the score of every allowed pair, the row maximum, the
    exponentials, their sum and the weighted sum of value rows."""
    B, H, S_q, S_kv, D = 2, 2, 9, 13, 8
    q = bits(71, (B, H, S_q, D), si.TID_Q, 2.0)
    k = bits(71, (B, H, S_kv, D), si.TID_K, 2.0)
    v = bits(71, (B, H, S_kv, D), si.TID_V)
    valid = [13, 5]
    scale = 0.35
    o, lse = oracle.attention_f64(q, k, v, scale, causal, kv_valid_len=valid)
    o = o.reshape(B, H, S_q, D)
    lse = lse.reshape(B, H, S_q)
    ld = np.longdouble
    ql, kl, vl = (si.bf16_bits_to_f32(x).astype(ld) for x in (q, k, v))
    for b in range(B):
        for h in range(H):
            for i in range(S_q):
                allowed = [j for j in range(S_kv) if j < valid[b] and (not causal or j <= i)]
                s = {j: ld(scale) * sum(ql[b, h, i, d] * kl[b, h, j, d] for d in range(D)) for j in allowed}
                m = max(s.values())
                e = {j: np.exp(s[j] - m) for j in allowed}
                l = sum(e.values())
                ref_o = [sum(e[j] * vl[b, h, j, d] for j in allowed) / l for d in range(D)]
                ref_lse = m + np.log(l)
                assert np.allclose(o[b, h, i].astype(ld), ref_o, rtol=0, atol=1e-12), (b, h, i)
                assert abs(ld(lse[b, h, i]) - ref_lse) <= 1e-12, (b, h, i)
