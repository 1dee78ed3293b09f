"""Host logic of bench.py: FLOP accounting, rank aggregation over gloo
(world size 2, CPU), and the reference arm under torchrun."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest

import bench

ROOT = Path(__file__).resolve().parent.parent


def test_flop_accounting_matches_closed_forms():
    w = bench.WORKLOADS["b1_h32_s4096_d128"]
    assert bench.alg_flops(w, True) == 4 * 32 * 128 * 4096 * 4097 // 2
    assert bench.alg_flops(w, False) == 4 * 32 * 128 * 4096 * 4096
    w = bench.WORKLOADS["b2_h32_s8192_d128_padded"]
    assert bench.alg_flops(w, False) == 4 * 32 * 128 * 8192 * (8192 + 5000)
    # causal with padding: row i sees min(valid, i + 1) keys
    assert bench.allowed_pairs(1, 1, 6, 6, True, [3]) == 1 + 2 + 3 + 3 + 3 + 3
    assert bench.allowed_pairs(1, 1, 4, 9, True) == 1 + 2 + 3 + 4
    assert bench.allowed_pairs(1, 1, 9, 4, True) == 1 + 2 + 3 + 4 * 6
    assert bench.allowed_pairs(2, 1, 5, 5, False, [0, 2]) == 0 + 10


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r: 1e12 * (r + 1) FLOPs per step in (10 + r) ms, e2e (20 + 5 r) ms
    res = bench.aggregate_ranks(1e12 * (rank + 1), 10.0 + rank, 20.0 + 5 * rank, dist, "cpu")
    out.put((rank, res))
    dist.destroy_process_group()


@pytest.mark.parametrize("B,H", [(4, 16), (1, 32), (2, 32), (1, 2), (1, 1), (3, 5), (8, 2)])
def test_e2e_pieces_cover_the_grid_once_contiguously(B, H):
    # the end-to-end leg moves each piece with one copy per tensor and runs it
    # as one attn_fwd call: whole batches, or a head range of one batch
    from io_aware_attention_fwd_gb300.host import plan_pieces
    seen = set()
    pieces = plan_pieces(B, H)
    for b0, nb, h0, nh in pieces:
        assert nb >= 1 and nh >= 1
        assert nb == 1 or (h0 == 0 and nh == H)
        for b in range(b0, b0 + nb):
            for h in range(h0, h0 + nh):
                assert (b, h) not in seen
                seen.add((b, h))
    assert len(seen) == B * H
    assert len(pieces) <= max(4, B * 2)


def test_auto_piece_count_follows_the_copy_size_rule():
    # each piece's Q copy stays at 4 MiB or more, with at most 4 pieces
    from io_aware_attention_fwd_gb300.host import MAX_PIECES, MIN_PIECE_BYTES, auto_pieces
    assert auto_pieces(1) == 1 and auto_pieces(MIN_PIECE_BYTES - 1) == 1
    assert auto_pieces(4 * 16 * 1024 * 64 * 2) == 2        # 1k, D=64 batch: 8 MiB of Q
    assert auto_pieces(32 * 4096 * 128 * 2) == MAX_PIECES  # 4k worked example: 32 MiB of Q
    assert auto_pieces(32 * 32768 * 128 * 2) == MAX_PIECES
    for n in range(MIN_PIECE_BYTES, 64 * MIN_PIECE_BYTES, MIN_PIECE_BYTES // 3):
        assert n // auto_pieces(n) >= MIN_PIECE_BYTES


def test_tapered_pieces_for_one_long_batch():
    from io_aware_attention_fwd_gb300.host import plan_tapered
    # 32k tokens, 32 heads: two-head end pieces (256 units each fill 152 SMs), three middle pieces
    pl = plan_tapered(1, 32, 32768, 128)
    assert [nh for _, _, _, nh in pl] == [2, 10, 9, 9, 2]
    assert [h0 for _, _, h0, _ in pl] == [0, 2, 12, 21, 30]
    # 4k tokens: an end piece would need 10 heads, too many for a taper; several batches: none
    assert plan_tapered(1, 32, 4096, 128) is None
    assert plan_tapered(4, 16, 1024, 64) is None
    for S in (8192, 16384, 32768, 65536):
        for H in (8, 16, 32, 64):
            pl = plan_tapered(1, H, S, 128)
            if pl is not None:
                assert sum(nh for *_, nh in pl) == H and pl[0][3] == pl[-1][3]
                assert all(a[2] + a[3] == b[2] for a, b in zip(pl, pl[1:]))


def test_profiled_traffic_needs_the_current_kernel_source(tmp_path, monkeypatch):
    # a profile summary supplies the roofline's DRAM traffic only while its
    # kernel-source hash matches the sources the bench runs
    current = bench.kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "x.md").write_text(f"# x\n\nbench_workload: wl_a\nkernel_source_sha256_16: {current}\n"
                               "dram_bytes_per_launch: 12345\n")
    (prof / "y.md").write_text("# y\n\nbench_workload: wl_b\nkernel_source_sha256_16: 0000000000000000\n"
                               "dram_bytes_per_launch: 999\n")
    monkeypatch.setattr(bench, "ROOT", tmp_path)  # the lookup reads tmp_path/profiles
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: current)
    assert bench.profiled_traffic("wl_a") == 12345.0
    assert bench.profiled_traffic("wl_b") is None       # stale hash
    assert bench.profiled_traffic("wl_c") is None       # no summary


def test_committed_profiles_name_bench_workloads():
    # every committed summary names a workload the bench knows and carries
    # the three fields the lookup reads
    import re
    files = sorted((Path(bench.__file__).resolve().parent / "profiles").glob("*.md"))
    assert files
    for f in files:
        text = f.read_text()
        w = re.search(r"^bench_workload:\s*(\S+)", text, re.M)
        assert w and w.group(1) in bench.WORKLOADS, f.name
        assert re.search(r"^kernel_source_sha256_16:\s*[0-9a-f]{16}$", text, re.M), f.name
        assert re.search(r"^dram_bytes_per_launch:\s*[0-9]+$", text, re.M), f.name


def test_rank_aggregation_gloo_world2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        value, e2e, t, te = got[r]
        assert t == 11.0 and te == 25.0                    # slowest rank
        assert value == pytest.approx(3e12 / 11e-3 / 1e12)  # summed work / max time
        assert e2e == pytest.approx(3e12 / 25e-3 / 1e12)


def test_single_rank_aggregation():
    value, e2e, t, te = bench.aggregate_ranks(2e12, 4.0, 8.0)
    assert (value, e2e, t, te) == (500.0, 250.0, 4.0, 8.0)


def test_reference_arm_under_torchrun_world2():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(ROOT / "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-seconds", "0.3",
           "--workload", "b4_h16_s1024_d64"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the whole step at the sampled rate, labelled as an extrapolation
    w = bench.WORKLOADS["b4_h16_s1024_d64"]
    full = sum(bench.alg_flops(w, c) for c in w["modes"])
    assert d["cpu_baseline"]["extrapolated_full_step_s"] == pytest.approx(full / (d["value"] * 1e12))
    # the same config object the GPU arm prints for this workload
    assert d["config"] == bench.workload_config("b4_h16_s1024_d64", bench.WORKLOADS["b4_h16_s1024_d64"], 2)


def test_default_workload_is_the_long_context_target():
    # the headline runs the 32k, D = 128 shape in both modes; the other
    # forward shapes are timed beside it
    w = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    assert (w["B"], w["H"], w["S"], w["D"]) == (1, 32, 32768, 128)
    assert set(w["modes"]) == {True, False}
    assert all(n in bench.WORKLOADS and n != bench.DEFAULT_WORKLOAD for n in bench.PER_CONFIG)
    cfg = bench.workload_config(bench.DEFAULT_WORKLOAD, w, 1)
    assert cfg["l2"].startswith("inputs larger than L2")
    assert bench.workload_config("b4_h16_s1024_d64", bench.WORKLOADS["b4_h16_s1024_d64"], 1)["l2"].startswith(
        "flushed")
