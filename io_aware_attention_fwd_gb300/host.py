"""Attention forward on host-resident inputs, with the copies overlapped.

``HostForward`` owns pinned host buffers for Q, K, V (which the caller
fills) and for O and LSE of each mask mode, plus their device copies.  One
``run()`` moves the inputs in, runs ``attn_fwd`` for every mode and moves the
results out.  The batch goes through in contiguous pieces, either whole
batches or a head range of one batch, so that the copy-in of one piece, the
kernels of another and the copy-out of a third run at the same time on three
streams.  Every piece is an ordinary ``attn_fwd`` call on contiguous slices,
and each row's result does not depend on the piece it was computed in.  The
whole step is captured once as a CUDA graph and replayed, so the host only
issues one launch per step.

PyTorch provides the memory, the streams and the graph; all attention
arithmetic runs in the CUDA library.
"""
from __future__ import annotations

import math

from . import _lib


# Piece-count rule, from pinned-copy bandwidth measured against copy size on
# GB300 (NVLink-C2C host link): one copy reaches about 90% of the ~205 GB/s
# host-to-device plateau from 4 MiB up, while 1-2 MiB copies run at 45-100
# GB/s; and beyond 4 pieces the per-piece kernel tails cost more than the
# shorter exposed first copy-in and last copy-out save.
MIN_PIECE_BYTES = 4 << 20
MAX_PIECES = 4


def auto_pieces(q_bytes: int) -> int:
    """Pieces for a step whose Q tensor has ``q_bytes``: as many as keep each
    piece's Q copy at MIN_PIECE_BYTES or more, at most MAX_PIECES."""
    return max(1, min(MAX_PIECES, int(q_bytes) // MIN_PIECE_BYTES))


def plan_tapered(B: int, H: int, S_q: int, D: int, sms: int = 152):
    """Pieces for one long batch: small first and last pieces, so that only
    their copies (the first copy-in, the last copy-out) are exposed, with
    larger ones between.  An end piece has the fewest heads whose work units
    (pairs of 128-row query tiles) still fill every SM once and whose Q copy
    is MIN_PIECE_BYTES or more; the heads between go into up to three equal
    pieces.  Returns None where that does not apply (B > 1, or too few heads
    for small end pieces); measured on GB300 at 32k tokens, 32 heads: heads
    [2, 10, 10, 8, 2] per piece ran the step 3% faster than four equal pieces,
    while at 4k tokens (copy-bound) equal pieces were as fast."""
    if B != 1 or H < 4:
        return None
    units_per_head = -(-S_q // 256)
    head_bytes = S_q * D * 2
    h_end = max(-(-sms // units_per_head), -(-MIN_PIECE_BYTES // head_bytes))
    if 4 * h_end > H:
        return None
    mid = H - 2 * h_end
    n_mid = max(1, min(3, auto_pieces(mid * head_bytes)))
    sizes = [h_end] + [mid // n_mid + (1 if i < mid % n_mid else 0) for i in range(n_mid)] + [h_end]
    out, h0 = [], 0
    for nh in sizes:
        out.append((0, 1, h0, nh))
        h0 += nh
    return out


def plan_pieces(B: int, H: int, target: int = 4):
    """About ``target`` pieces (b0, nb, h0, nh) of the [B][H] grid, each either
    whole batches (h0 = 0, nh = H) or a head range of one batch (nb = 1), so
    every piece of a [B][H][S][D] tensor is one contiguous block."""
    if B < 1 or H < 1 or target < 1:
        raise ValueError("B, H and target must be positive")
    if B >= target:
        nb = -(-B // target)
        return [(b0, min(nb, B - b0), 0, H) for b0 in range(0, B, nb)]
    per_b = -(-target // B)  # head pieces per batch
    nh = -(-H // per_b)
    return [(b, 1, h0, min(nh, H - h0)) for b in range(B) for h0 in range(0, H, nh)]


class HostForward:
    """Forward pass for fixed shapes on pinned host buffers (see module doc).

    B, H, S_q, S_kv, D: shapes as for ``attn_fwd``.  modes: the mask modes run
    per step (False = non-causal, True = causal), each with its own outputs.
    kv_valid_len: int32 CUDA tensor [B] or None, fixed for the executor's
    life.  pieces: target number of pieces (None: ``plan_tapered`` where it
    applies, else ``auto_pieces`` of the Q tensor's size).  graph: capture the
    step as a CUDA graph (else every ``run`` issues the launches and copies
    eagerly).

    Fill ``host_inputs`` (q, k, v: pinned bf16 [B,H,S,D]) before ``run()``;
    after the stream has reached the end of a step, ``host_outputs[mode]``
    holds (o bf16 [B,H,S_q,D], lse fp32 [B,H,S_q]).
    """

    def __init__(self, B: int, H: int, S_q: int, S_kv: int, D: int, modes=(False,),
                 scale: float | None = None, kv_valid_len=None, device="cuda", pieces: int | None = None,
                 graph: bool = True):
        import torch

        self.shape = (B, H, S_q, S_kv, D)
        self.modes = tuple(bool(m) for m in modes)
        if not self.modes:
            raise ValueError("at least one mode")
        self.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
        self.device = torch.device(device)
        self.kv_valid_len = kv_valid_len
        plan = None
        if pieces is None:
            plan = plan_tapered(B, H, S_q, D, torch.cuda.get_device_properties(self.device).multi_processor_count)
            pieces = auto_pieces(B * H * S_q * D * 2)
        self.pieces = plan if plan is not None else plan_pieces(B, H, pieces)
        bf = torch.bfloat16
        dev = self.device
        self._q = torch.empty((B, H, S_q, D), dtype=bf, device=dev)
        self._k = torch.empty((B, H, S_kv, D), dtype=bf, device=dev)
        self._v = torch.empty((B, H, S_kv, D), dtype=bf, device=dev)
        self._outs = {m: (torch.empty((B, H, S_q, D), dtype=bf, device=dev),
                          torch.empty((B, H, S_q), dtype=torch.float32, device=dev)) for m in self.modes}
        self.host_inputs = tuple(torch.empty(x.shape, dtype=bf).pin_memory() for x in (self._q, self._k, self._v))
        self.host_outputs = {m: (torch.empty(o.shape, dtype=bf).pin_memory(),
                                 torch.empty(lse.shape, dtype=torch.float32).pin_memory())
                             for m, (o, lse) in self._outs.items()}
        self.h2d_bytes = sum(x.numel() * x.element_size() for x in self.host_inputs)
        self.d2h_bytes = sum(x.numel() * x.element_size() for pair in self.host_outputs.values() for x in pair)
        self._s_in = torch.cuda.Stream(dev)
        self._s_out = torch.cuda.Stream(dev)
        self._graph = None
        # one eager step warms every piece's launch path before any capture
        self._step(torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._step(torch.cuda.current_stream(dev))
            torch.cuda.synchronize(dev)
            self._graph = g

    def _step(self, main) -> None:
        import torch

        B, H, S_q, S_kv, D = self.shape
        begin = torch.cuda.Event()
        begin.record(main)
        self._s_in.wait_event(begin)  # earlier work on the stream has read the device inputs
        dev_in = (self._q, self._k, self._v)
        for b0, nb, h0, nh in self.pieces:
            sl = (slice(b0, b0 + nb), slice(h0, h0 + nh))
            with torch.cuda.stream(self._s_in):
                for dst, src in zip(dev_in, self.host_inputs):
                    dst[sl].copy_(src[sl], non_blocking=True)
                arrived = torch.cuda.Event()
                arrived.record(self._s_in)
            main.wait_event(arrived)
            kvl = self.kv_valid_len[b0:b0 + nb] if self.kv_valid_len is not None else None
            for m in self.modes:
                o, lse = self._outs[m]
                _lib.attn_fwd(self._q[sl], self._k[sl], self._v[sl], o[sl], lse[sl], nb, nh, S_q, S_kv, D,
                              self.scale, m, kvl, main)
            computed = torch.cuda.Event()
            computed.record(main)
            self._s_out.wait_event(computed)
            with torch.cuda.stream(self._s_out):
                for m in self.modes:
                    for dst, src in zip(self.host_outputs[m], self._outs[m]):
                        dst[sl].copy_(src[sl], non_blocking=True)
        copied = torch.cuda.Event()
        copied.record(self._s_out)
        main.wait_event(copied)  # the step ends when its last result is on the host

    def run(self) -> None:
        """Enqueue one step on the current stream."""
        import torch

        if self._graph is not None:
            self._graph.replay()
        else:
            self._step(torch.cuda.current_stream(self.device))

    @property
    def launches_per_step(self) -> int:
        return len(self.pieces) * len(self.modes)
