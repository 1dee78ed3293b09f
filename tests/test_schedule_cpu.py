"""The host-built unit order of long causal launches (attn_fwd_schedule):
a valid table, balanced across the CTAs, with few heads in flight at once.

Host logic only: the library builds the table without a device.  The cost
model here is restated from the causal mask, not taken from the library: the
query pair p of a head covers rows [256 p, 256 p + 256), and its second query
tile, which sees the most keys, needs ceil(min(S_kv, rows seen) / 128) kv
tiles."""
from __future__ import annotations

import heapq
import math

import pytest

import io_aware_attention_fwd_gb300 as attn
from io_aware_attention_fwd_gb300 import build_ext

SMS = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()


def kv_tiles(p, S_q, S_kv):
    # the longest of the pair's two 128-row tiles under the causal mask
    n = 1
    for t in range(2):
        qs = p * 256 + t * 128
        if qs < S_q:
            n = max(n, math.ceil(min(S_kv, qs + 128, S_q) / 128))
    return n


def decode(u, BH, n_pairs):
    return u % BH, n_pairs - 1 - u // BH  # (head, query pair)


def simulate(off, unit, BH, n_pairs, S_q, S_kv):
    """Run the table with each unit costing its kv tiles plus one: returns
    the per-CTA finish times and the most heads any instant has in flight."""
    G = len(off) - 1
    events = []
    finish = []
    for c in range(G):
        t = 0
        for u in unit[off[c]:off[c + 1]]:
            bh, p = decode(u, BH, n_pairs)
            d = kv_tiles(p, S_q, S_kv) + 1
            events.append((t, 1, bh))
            events.append((t + d, -1, bh))
            t += d
        finish.append(t)
    events.sort(key=lambda e: (e[0], e[1]))  # ends before starts at the same instant
    live, most = {}, 0
    for _, delta, bh in events:
        live[bh] = live.get(bh, 0) + delta
        if live[bh] == 0:
            del live[bh]
        most = max(most, len(live))
    return finish, most


@pytest.mark.parametrize("B,H,S,D,eb", [
    (1, 32, 32768, 128, 2),   # the long-context shape: K + V = 512 MiB
    (1, 32, 8192, 128, 2),    # 128 MiB
    (1, 16, 9000, 128, 2),    # ragged last pair, 16 heads
    (1, 16, 17000, 64, 2),    # D = 64
    (2, 8, 16384, 128, 2),    # two sequences
    (1, 32, 32768, 128, 1),   # e4m3: 256 MiB
])
def test_table_is_a_balanced_permutation(B, H, S, D, eb):
    got = attn.attn_fwd_schedule(B, H, S, S, D, eb, SMS)
    assert got is not None
    off, unit = got
    BH, n_pairs = B * H, math.ceil(S / 256)
    n = BH * n_pairs
    G = min(n, SMS)
    assert len(off) == G + 1 and off[0] == 0 and off[-1] == n
    assert all(a <= b for a, b in zip(off, off[1:]))
    assert sorted(unit) == list(range(n))  # every unit exactly once
    finish, most = simulate(off, unit, BH, n_pairs, S, S)
    total = sum(kv_tiles(p, S, S) + 1 for _ in range(BH) for p in range(n_pairs))
    # greedy list scheduling is within one unit of the mean load
    longest = max(kv_tiles(p, S, S) for p in range(n_pairs)) + 1
    assert max(finish) <= total / G + longest
    assert total / G / max(finish) > 0.96
    # the L2 working set: the K and V of the heads in flight stay within
    # 96 MiB (the interleaved last heads' 64 MiB plus the head-major window),
    # under GB300's 129 MB L2, where every head's would be B*H*S*D*eb*2
    head_kv = S * D * eb * 2
    assert most * head_kv <= 96 << 20, (most, head_kv)


def test_heads_before_the_tail_run_in_order():
    # head-major part: a head's units are all handed out before the next head's
    B, H, S, D = 1, 32, 32768, 128
    off, unit = attn.attn_fwd_schedule(B, H, S, S, D, 2, SMS)
    n_pairs = math.ceil(S / 256)
    tail = (64 << 20) // (S * D * 2 * 2)
    starts = {}
    for c in range(len(off) - 1):
        t = 0
        for u in unit[off[c]:off[c + 1]]:
            bh, p = decode(u, H, n_pairs)
            starts.setdefault(bh, []).append(t)
            t += kv_tiles(p, S, S) + 1
    firsts = [min(starts[h]) for h in range(H - tail)]
    assert firsts == sorted(firsts)


@pytest.mark.parametrize("B,H,S,D,eb", [
    (1, 32, 4096, 128, 2),    # K + V = 64 MiB exactly: the longest-first order
    (4, 16, 1024, 64, 2),
    (1, 1, 32768, 128, 2),    # one head: 16 MiB
])
def test_short_launches_have_no_table(B, H, S, D, eb):
    assert attn.attn_fwd_schedule(B, H, S, S, D, eb, SMS) is None


@pytest.mark.parametrize("kw", [dict(B=0), dict(S_q=0), dict(D=96), dict(elem_bytes=4), dict(sms=0)])
def test_invalid_arguments(kw):
    args = dict(B=1, H=32, S_q=32768, S_kv=32768, D=128, elem_bytes=2, sms=SMS)
    args.update(kw)
    with pytest.raises(ValueError):
        attn.attn_fwd_schedule(**args)
