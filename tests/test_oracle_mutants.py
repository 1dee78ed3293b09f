"""Planted mistakes in the oracle must each break at least one pin.

Each case copies the oracle's C++ source, applies one textual mutation that a
plausible slip would make (a dropped term, a wrong sign or index, a swapped
operand), compiles the copy into a temporary library, and runs a battery of
pins (closed forms plus torch's float64 CPU SDPA) against it.  The unmutated
source passes the same battery.  Everything runs on the CPU.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si

MUTANTS = {
    "drop_scale": ("s_row[j] = p.scale * dot;", "s_row[j] = dot;"),
    "causal_excludes_diagonal": ("if (p.causal && j > i) return false;",
                                 "if (p.causal && j >= i) return false;"),
    "padding_off_by_one": ("if (j >= valid) return false;", "if (j > valid) return false;"),
    "q_dot_v_instead_of_k": ("q_at(p, qi + d) * k_at(p, kbh + j * p.D + d)",
                             "q_at(p, qi + d) * v_at(p, vbh + j * p.D + d)"),
    "no_normalisation": ("o_row[d] /= l;", "o_row[d] /= 1.0;"),
    "lse_without_max": ("*lse_out = m + std::log(l);", "*lse_out = std::log(l);"),
    "lse_base2": ("*lse_out = m + std::log(l);", "*lse_out = m + std::log2(l);"),
    "valid_len_of_batch0": ("std::max<int64_t>(p.kv_valid_len[b], 0)",
                            "std::max<int64_t>(p.kv_valid_len[0], 0)"),
    "k_head_index_dropped": ("const int64_t kbh = (b * p.H + h) * p.S_kv * p.D;",
                             "const int64_t kbh = (b * p.H + 0) * p.S_kv * p.D;"),
    "v_row_index_shifted": ("e * v_at(p, vbh + j * p.D + d)",
                            "e * v_at(p, vbh + ((j + 1) % p.S_kv) * p.D + d)"),
}


def _bits(seed, shape, tid, mult=1.0):
    return si.normal_bf16(seed, tid, int(np.prod(shape)), mult).reshape(shape)


def _f64(b):
    return si.bf16_bits_to_f32(b).astype(np.float64)


def pin_failures(lib) -> list[str]:
    """Names of the pins that ``lib`` violates (empty when all hold)."""
    torch = pytest.importorskip("torch")
    failed = []
    B, H, S_q, S_kv, D = 2, 2, 11, 14, 16
    q = _bits(31, (B, H, S_q, D), si.TID_Q, 2.0)
    k = _bits(31, (B, H, S_kv, D), si.TID_K, 2.0)
    v = _bits(31, (B, H, S_kv, D), si.TID_V)
    scale = 0.25
    valid = [14, 6]
    for causal in (False, True):
        o, lse = oracle.attention_f64(q, k, v, scale, causal, kv_valid_len=valid, lib=lib)
        j = np.arange(S_kv)[None, :]
        i = np.arange(S_q)[:, None]
        masks = []
        for b in range(B):
            m = np.broadcast_to(j < valid[b], (S_q, S_kv))
            masks.append(m & (j <= i) if causal else m)
        mask = torch.from_numpy(np.stack(masks))[:, None].expand(B, H, S_q, S_kv)
        tq, tk, tv = (torch.from_numpy(_f64(x)) for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
        if not np.allclose(o.reshape(ref.shape), ref.numpy(), rtol=1e-10, atol=1e-12):
            failed.append(f"torch_sdpa_o_causal{int(causal)}")
        logits = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1).numpy()
        if not np.allclose(lse.reshape(ref_lse.shape), ref_lse, rtol=1e-10, atol=1e-12):
            failed.append(f"torch_sdpa_lse_causal{int(causal)}")
    # Q = 0: O is the mean of the allowed value rows and LSE = ln(count)
    z = np.zeros_like(q)
    o, lse = oracle.attention_f64(z, k, v, scale, False, kv_valid_len=valid, lib=lib)
    o = o.reshape(B, H, S_q, D)
    for b in range(B):
        if not np.allclose(o[b], _f64(v[b, :, :valid[b]]).mean(axis=1, keepdims=True), atol=1e-12):
            failed.append("zero_q_mean")
            break
    if not np.allclose(lse.reshape(B, H, S_q)[1], math.log(valid[1]), atol=1e-12):
        failed.append("zero_q_lse")
    return failed


def test_unmutated_oracle_passes_battery():
    assert pin_failures(oracle.load_library()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    find, repl = MUTANTS[name]
    src = oracle.SOURCE.read_text()
    assert src.count(find) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "attn_ref_mutant.cpp"
    mutated.write_text(src.replace(find, repl, 1))
    lib_path = oracle.compile_library(mutated, tmp_path / f"libmutant_{name}.so", ("-O1",))
    lib = oracle.load_library(lib_path)
    assert pin_failures(lib), f"planted mistake {name} went unnoticed"
