"""Pins of the oracle's backward pass: central finite differences of the
oracle's own (C++) forward pass, and torch's float64 CPU autograd through
scaled_dot_product_attention."""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si


def draws(seed, shape, tid, mult=1.0):
    return si.normal_f64(seed, tid, int(np.prod(shape))).reshape(shape) * mult


@pytest.mark.parametrize("causal,valid", [(False, None), (True, None), (True, [9, 4]), (False, [0, 7])])
def test_backward_matches_finite_differences(causal, valid):
    B, H, S_q, S_kv, D = 2, 1, 7, 9, 5
    q = draws(60, (B, H, S_q, D), 1)
    k = draws(60, (B, H, S_kv, D), 2)
    v = draws(60, (B, H, S_kv, D), 3)
    g = draws(60, (B, H, S_q, D), 5)          # dL/dO for L = sum(O * g)
    scale = 0.6
    dq, dk, dv = oracle.attention_bwd_f64(q, k, v, g, scale, causal, kv_valid_len=valid)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_f64_dbl(q_, k_, v_, scale, causal, kv_valid_len=valid)
        return float((o.reshape(g.shape) * g).sum())

    eps = 1e-5
    rng = np.random.default_rng(0)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert fd == pytest.approx(grad[idx], rel=1e-6, abs=1e-9), (name, idx)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    torch = pytest.importorskip("torch")
    B, H, S_q, S_kv, D = 1, 2, 12, 16, 8
    bits = [si.normal_bf16(61, t, B * H * n * D, 2.0).reshape(B, H, n, D)
            for t, n in ((1, S_q), (2, S_kv), (3, S_kv), (5, S_q))]
    q, k, v, g = (si.bf16_bits_to_f32(x).astype(np.float64) for x in bits)
    scale = 1 / math.sqrt(D)
    dq, dk, dv = oracle.attention_bwd_f64(*bits, scale, causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    out.backward(torch.from_numpy(g))
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_float_and_bf16_inputs_agree():
    B, H, S, D = 1, 1, 6, 4
    bits = [si.normal_bf16(62, t, B * H * S * D).reshape(B, H, S, D) for t in (1, 2, 3, 5)]
    a = oracle.attention_bwd_f64(*bits, 0.5, True)
    b = oracle.attention_bwd_f64(*(si.bf16_bits_to_f32(x) for x in bits), 0.5, True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sums_and_masked_keys(causal):
    """Closed forms that hold for any inputs:
    * Adding one vector to every key shifts each row's logits by a constant,
      which the softmax ignores, so the key gradients of a head sum to zero.
    * Each row of P sums to one, so the value gradients of a head sum to the
      sum of dO over the rows that have at least one allowed key.
    * A key past its batch's valid length gets exactly zero gradient, and a
      batch with no valid key gets zero gradients everywhere."""
    B, H, S_q, S_kv, D = 3, 2, 9, 11, 6
    q = draws(63, (B, H, S_q, D), 1)
    k = draws(63, (B, H, S_kv, D), 2)
    v = draws(63, (B, H, S_kv, D), 3)
    g = draws(63, (B, H, S_q, D), 5)
    valid = [11, 4, 0]
    dq, dk, dv = oracle.attention_bwd_f64(q, k, v, g, 0.7, causal, kv_valid_len=valid)
    for b in range(B):
        n = valid[b]
        # with top-left causal alignment key 0 is allowed for every row
        has_key = np.full(S_q, n > 0)
        np.testing.assert_allclose(dk[b].sum(axis=1), 0.0, atol=1e-12)
        np.testing.assert_allclose(dv[b].sum(axis=1), g[b][:, has_key].sum(axis=1), atol=1e-12)
        assert np.all(dk[b, :, n:] == 0.0) and np.all(dv[b, :, n:] == 0.0)
    assert np.all(dq[2] == 0.0)


def test_backward_head_subset_matches_full():
    B, H, S, D = 2, 3, 10, 4
    args = [draws(64, (B, H, S, D), t) for t in (1, 2, 3, 5)]
    full = oracle.attention_bwd_f64(*args, 0.5, True, kv_valid_len=[10, 6])
    part = oracle.attention_bwd_f64(*args, 0.5, True, kv_valid_len=[10, 6], heads=[(0, 2), (1, 0)])
    for f, g in zip(full, part):
        for b in range(B):
            for h in range(H):
                if (b, h) in [(0, 2), (1, 0)]:
                    np.testing.assert_array_equal(g[b, h], f[b, h])
                else:
                    assert np.all(g[b, h] == 0.0)
