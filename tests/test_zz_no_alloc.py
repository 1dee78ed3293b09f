"""attn_fwd_splitkv_static: the key-split forward pass for callers that cannot
allocate device memory, using the library's fixed scratch array.

Its results must match the workspace-taking entry point (attn_fwd_splitkv)
within the parity tolerance, on two calls in a row (the second call finds the
first one's partials still in the shared array).  The file name makes pytest
collect it last, so a run that stops at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import seeded_inputs as si
from tests import parity


_REFUSALS = r"""
import re, sys
from pathlib import Path
import io_aware_attention_fwd_gb300 as attn
header = (Path(sys.argv[1]) / "include" / "attn_fwd.h").read_text()
m = re.search(r"#define ATTN_STATIC_SCRATCH_BYTES \((\d+)ull << (\d+)\)", header)
assert m and int(m.group(1)) << int(m.group(2)) == attn.STATIC_SCRATCH_BYTES
fake = 0x10000
# 64 splits x 8 heads x 4096 rows x 129 floats is over 32 MiB: refused before any launch
need = attn.attn_fwd_splitkv_workspace_bytes(1, 8, 4096, 128, 64)
assert need > attn.STATIC_SCRATCH_BYTES
st = attn.call_status(attn.attn_fwd_splitkv_static, fake, fake, fake, fake, fake, 1, 8, 4096, 4096,
                      128, 0.1, False, None, 64)
assert st == attn.ATTN_ERR_UNSUPPORTED, st
st = attn.call_status(attn.attn_fwd_splitkv_static, fake, fake, fake, fake, fake, 1, 8, 4096, 4096,
                      128, 0.1, False, None, 0)
assert st == attn.ATTN_ERR_INVALID_ARG, st
print("refusals ok")
"""


def test_static_entry_rejects_sizes_beyond_the_fixed_scratch():
    # The refusals are checked in a child process that sees no CUDA device:
    # the fake pointers below could never reach a kernel, and a refusal that
    # came only after a device call would show up as ATTN_ERR_DEVICE instead.
    import os
    import subprocess
    import sys
    from pathlib import Path
    import io_aware_attention_fwd_gb300 as attn
    attn.build()
    root = Path(__file__).resolve().parent.parent
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", PYTHONPATH=str(root))
    res = subprocess.run([sys.executable, "-c", _REFUSALS, str(root)], capture_output=True, text=True,
                         timeout=300, env=env, cwd=root)
    assert res.returncode == 0 and "refusals ok" in res.stdout, res.stderr[-2000:]


@pytest.mark.gpu
def test_static_entry_matches_workspace_entry_twice():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import io_aware_attention_fwd_gb300 as attn
    attn.build()
    dev = torch.device("cuda:0")
    cases = [  # (seed, B, H, S_q, S_kv, D, causal, n_splits, kv_valid_len)
        (1001, 1, 8, 256, 8192, 128, False, 9, None),
        (1002, 2, 2, 300, 3000, 64, True, 5, [3000, 1234]),
    ]
    for seed, B, H, S_q, S_kv, D, causal, n_splits, valid in cases:
        assert attn.attn_fwd_splitkv_workspace_bytes(B, H, S_q, D, n_splits) <= attn.STATIC_SCRATCH_BYTES
        q, k, v = si.qkv_bf16(seed, B, H, S_q, S_kv, D)
        tq, tk, tv = (parity.to_device(x, dev) for x in (q, k, v))
        kvl = None if valid is None else torch.tensor(valid, dtype=torch.int32, device=dev)
        scale = 1 / math.sqrt(D)
        # reference: the entry point that takes a caller workspace
        o_ref = torch.empty_like(tq)
        l_ref = torch.empty((B, H, S_q), dtype=torch.float32, device=dev)
        nbytes = attn.attn_fwd_splitkv_workspace_bytes(B, H, S_q, D, n_splits)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        attn.attn_fwd_splitkv(tq, tk, tv, o_ref, l_ref, B, H, S_q, S_kv, D, scale, causal, kvl, n_splits,
                              ws, nbytes)
        # the fixed-scratch entry point, through the C ABI
        o = torch.full_like(tq, float("nan"))
        lse = torch.full((B, H, S_q), float("nan"), dtype=torch.float32, device=dev)
        attn.attn_fwd_splitkv_static(tq, tk, tv, o, lse, B, H, S_q, S_kv, D, scale, causal, kvl, n_splits)
        torch.cuda.synchronize()
        assert attn.attn_fwd_debug_status() == attn.ATTN_OK
        o_a, l_a = parity.gather_rows(o, lse)
        o_b, l_b = parity.gather_rows(o_ref, l_ref)
        parity.compare(o_a, l_a, o_b, l_b)
        # and both against the fp64 oracle on the same inputs
        o_or, l_or = oracle.attention_f64(q, k, v, scale, causal, kv_valid_len=valid)
        parity.compare(o_a, l_a, o_or, l_or)
        parity.compare(o_b, l_b, o_or, l_or)
