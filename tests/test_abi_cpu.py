"""The C-ABI library builds, loads without a GPU, exports what its header
declares, and rejects bad arguments before touching the device."""
from __future__ import annotations

import re
from pathlib import Path

import pytest

import io_aware_attention_fwd_gb300 as attn
from io_aware_attention_fwd_gb300 import build_ext

HEADER = Path(__file__).resolve().parent.parent / "include" / "attn_fwd.h"
FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced on these paths


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(attn.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = attn.load()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_is_sm103a_only():
    # the fatbin is built for sm_103a alone (no PTX fallback, no other arch)
    assert "arch=compute_103a,code=sm_103a" in " ".join(build_ext.NVCC_FLAGS)
    assert build_ext.NVCC_FLAGS.count("-gencode") == 1


def test_abi_version_and_status_strings():
    assert attn.attn_fwd_abi_version() == 1
    names = {s: attn.attn_status_str(s) for s in range(7)}
    assert names[0] == "ok" and len(set(names.values())) == 7
    assert attn.attn_status_str(99) == "unknown status"


def call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, S_q=128, S_kv=128, D=64,
                scale=0.125, causal=False, kv_valid_len=None)
    args.update(kw)
    return attn.attn_fwd_status(**args)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(k=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(v=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(H=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(S_q=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(S_kv=-5), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.5), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q=FAKE + 8), attn.ATTN_ERR_ALIGNMENT),
    (dict(k=FAKE + 2), attn.ATTN_ERR_ALIGNMENT),
    (dict(o=FAKE + 4), attn.ATTN_ERR_ALIGNMENT),
    (dict(lse=FAKE + 2), attn.ATTN_ERR_ALIGNMENT),
    (dict(kv_valid_len=FAKE + 1), attn.ATTN_ERR_ALIGNMENT),
    (dict(B=1 << 16, H=1 << 16), attn.ATTN_ERR_UNSUPPORTED),          # B*H overflows int32
    (dict(B=1 << 15, H=1 << 10, S_q=1 << 20), attn.ATTN_ERR_UNSUPPORTED),  # grid too large
    (dict(S_q=0), attn.ATTN_OK),                                      # empty query set: no-op
    (dict(S_q=0, q=None, o=None, lse=None), attn.ATTN_OK),            # empty tensors may be null
])
def test_argument_checks_before_launch(kw, expect):
    assert call(**kw) == expect


def test_causal_flag_must_be_boolean():
    lib = attn.load()
    st = lib.attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 8, 64, 0.125, 2, None, None)
    assert st == attn.ATTN_ERR_INVALID_ARG


def test_watchdog_selftest_rejects_bad_limits():
    assert attn.attn_watchdog_selftest(10) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_watchdog_selftest(10**11) == attn.ATTN_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    from io_aware_attention_fwd_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", tmp_path / "absent.so")
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()


def split_call(**kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, S_q=128, S_kv=4096, D=128,
                scale=0.1, causal=False, kv_valid_len=None, n_splits=4, workspace=FAKE,
                workspace_bytes=attn.attn_fwd_splitkv_workspace_bytes(1, 2, 128, 128, 4))
    args.update(kw)
    return attn.call_status(attn.attn_fwd_splitkv, **args)


def test_splitkv_workspace_size():
    # fp32 partial O and LSE per split: n_splits * rows * (D + 1) * 4 bytes
    assert attn.attn_fwd_splitkv_workspace_bytes(2, 3, 100, 64, 5) == 5 * 600 * 65 * 4
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 96, 2) == 0      # bad D
    assert attn.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 64, 65) == 0     # too many splits


@pytest.mark.parametrize("kw,expect", [
    (dict(n_splits=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(n_splits=65), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace=FAKE + 8), attn.ATTN_ERR_ALIGNMENT),
    (dict(workspace_bytes=1000), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=80), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(S_q=0), attn.ATTN_OK),
])
def test_splitkv_argument_checks(kw, expect):
    assert split_call(**kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(n_parts=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(rows=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(D=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(o_parts=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o_parts=FAKE + 4), attn.ATTN_ERR_ALIGNMENT),
    (dict(o=FAKE + 2), attn.ATTN_ERR_ALIGNMENT),
    (dict(rows=0), attn.ATTN_OK),
])
def test_merge_argument_checks(kw, expect):
    args = dict(o_parts=FAKE, lse_parts=FAKE, n_parts=3, rows=100, D=64, o=FAKE, lse=FAKE)
    args.update(kw)
    assert attn.call_status(attn.attn_merge, **args) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(D=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q_descale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(k_descale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(v_descale=-1.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=1e-30, q_descale=1e-30, k_descale=1e-30), attn.ATTN_ERR_INVALID_ARG),  # underflows
    (dict(q=FAKE + 4), attn.ATTN_ERR_ALIGNMENT),
    (dict(S_q=0), attn.ATTN_OK),
])
def test_fp8_argument_checks(kw, expect):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=2, S_q=128, S_kv=128, D=128,
                scale=0.1, q_descale=1.0, k_descale=1.0, v_descale=1.0, causal=False)
    args.update(kw)
    assert attn.call_status(attn.attn_fwd_fp8, **args) == expect


def test_bwd_workspace_size():
    # lse2 and delta padded to whole 128-row tiles, plus the fp32 dQ accumulator
    assert attn.attn_bwd_workspace_bytes(2, 3, 200, 64) == (2 * 6 * 256 + 6 * 200 * 64) * 4
    assert attn.attn_bwd_workspace_bytes(1, 1, 10, 96) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(d_o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(dq=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(dk=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace_bytes=100), attn.ATTN_ERR_INVALID_ARG),
    (dict(workspace=FAKE + 4), attn.ATTN_ERR_ALIGNMENT),
    (dict(dv=FAKE + 2), attn.ATTN_ERR_ALIGNMENT),
    (dict(D=32), attn.ATTN_ERR_UNSUPPORTED),
    (dict(scale=-1.0), attn.ATTN_ERR_INVALID_ARG),
])
def test_bwd_argument_checks(kw, expect):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, d_o=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=1, H=2,
                S_q=128, S_kv=128, D=64, scale=0.125, causal=False, kv_valid_len=None, workspace=FAKE,
                workspace_bytes=attn.attn_bwd_workspace_bytes(1, 2, 128, 64))
    args.update(kw)
    assert attn.call_status(attn.attn_bwd, **args) == expect
