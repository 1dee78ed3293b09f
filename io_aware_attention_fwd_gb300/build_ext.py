"""Builds the CUDA library in-tree: ``_build/libattn_fwd.so`` for sm_103a.

The library is the product's only compute path; nothing falls back to the
CPU.  Run ``python -m io_aware_attention_fwd_gb300.build_ext`` or call
``build()``.
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
SOURCES = [PKG / "csrc" / "attn_fwd.cu"]
HEADERS = [ROOT / "include" / "attn_fwd.h", *sorted((PKG / "csrc").glob("*.cuh"))]
BUILD_DIR = PKG / "_build"
LIB_PATH = BUILD_DIR / "libattn_fwd.so"

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = Path(cuda_home) / "bin" / "nvcc"
    return str(cand) if cand.exists() else "nvcc"


def is_stale() -> bool:
    if not LIB_PATH.exists():
        return True
    t = LIB_PATH.stat().st_mtime
    return any(p.stat().st_mtime > t for p in SOURCES + HEADERS + [Path(__file__)])


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile the library if it is missing or stale; returns its path."""
    if not force and not is_stale():
        return LIB_PATH
    BUILD_DIR.mkdir(parents=True, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=str(BUILD_DIR))
    os.close(fd)
    cmd = [nvcc(), *NVCC_FLAGS, "-I", str(ROOT / "include"), *map(str, SOURCES), "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{res.stderr}")
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
