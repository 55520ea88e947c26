"""Hybrid CSA / HCA decoding, one token per step, through the C ABI.

"DeepSeek-V4 详解" section 2.4: the attention layers alternate, CSA in the
even layers and HCA in the odd ones.  The hongke120.com page, section 4.1,
lists the cache entries such a model keeps: uncompressed tail tokens, CSA
compressed blocks, HCA summaries and indexer keys.  ``HybridDecoder`` holds
one CSA layer and one HCA layer over a batch of sequences and keeps those
four caches as tokens arrive:

* raw rows of the recent tokens (KV rows and gate logits of both layers and
  the CSA indexer-key rows and gates): one sliding buffer per tensor, row j
  holding position ``p0 + j``.  It keeps every row that a pending block or a
  window still needs; when it fills up, the rows still needed move to the
  front (one contiguous device copy per sequence and tensor);
* CSA entries and indexer keys: the block of m = 4 tokens that a token
  completes is pooled into both caches by that token's ``csa_forward``
  (which compresses every entry from the last cached one on);
* HCA entries: the block of m' = 128 tokens that a token completes is pooled
  by ``csa_compress`` before that token's ``hca_attend``.

The projections that produce a token's rows and queries are upstream, as in
the single-layer calls: the caller writes the new token's raw rows into
``slot(name)`` (the projection's output buffer) and passes its queries to
``step``.  ``step`` only launches the library's kernels; the host keeps the
bookkeeping (position, cached counts, buffer origin).
"""

from __future__ import annotations

import torch

from . import csa

RAW_NAMES = ("x0", "g0", "xi0", "gi0", "x1", "g1")


class SlidingRows:
    """Sliding buffers of raw rows ([B, R, width] each): row j of every buffer
    holds position ``p0 + j``; positions ``p0 .. t_next - 1`` are filled."""

    def __init__(self, bufs: dict, p0: int, t_next: int):
        self.bufs = bufs
        self.R = next(iter(bufs.values())).shape[1]
        self.B = next(iter(bufs.values())).shape[0]
        if not 0 <= t_next - p0 <= self.R:
            raise ValueError(f"{t_next - p0} rows held, the buffers have {self.R}")
        self.p0, self.t_next = p0, t_next

    def room(self, keep_from: int):
        """Make row ``t_next`` free: when the buffers are full, move the rows of
        positions keep_from .. t_next-1 to the front.  keep_from must leave
        the source and destination apart (t_next - keep_from <= R / 2 does)."""
        t = self.t_next
        if t - self.p0 < self.R:
            return
        lo = max(keep_from, self.p0)
        n, a = t - lo, lo - self.p0
        if a < n:
            raise ValueError(f"keeping {n} of {self.R} rows would overlap the move")
        for buf in self.bufs.values():
            for b in range(self.B):  # contiguous rows: one device copy each
                buf[b, :n].copy_(buf[b, a:a + n])
        self.p0 = lo

    def slot(self, name: str) -> torch.Tensor:
        j = self.t_next - self.p0
        return self.bufs[name][:, j:j + 1]

    def advance(self):
        self.t_next += 1


class HybridDecoder:
    """One CSA layer (``p_csa``, m = 4) and one HCA layer (``p_hca``, m' =
    128) over B sequences, advanced one token per ``step``.

    ``t0`` is the position of the first token ``step`` takes.  Before it, the
    caches must hold the entries of the blocks completed before ``t0``
    (``kv``, ``keys``: ``t0 // m`` entries; ``ent``: ``t0 // m'``) and the raw
    buffers the rows of positions ``p0 .. t0 - 1`` (``seed``).  ``max_len``
    bounds the positions (cache capacity); ``raw_rows`` is the length of the
    sliding buffers and ``held`` how many rows before ``t0`` they start with
    (at least what the first step needs)."""

    def __init__(self, p_csa: csa.Params, p_hca: csa.Params, t0: int, max_len: int, device,
                 bias0, bias_i0, bias1, raw_rows: int = 512, held: int | None = None):
        pc, ph = p_csa, p_hca
        if pc.B != ph.B:
            raise ValueError("both layers decode the same batch")
        if not 0 <= t0 < max_len:
            raise ValueError(f"t0 {t0} not in [0, {max_len})")
        self.pc, self.ph, self.B = pc, ph, pc.B
        B = pc.B
        self.t = t0 - 1  # last position whose rows are in the buffers
        self.max_len = max_len
        self.need = max(pc.window, ph.window) + max(pc.m, ph.m)
        if raw_rows < 2 * self.need:
            raise ValueError(f"raw_rows {raw_rows} < {2 * self.need}")
        held = self.need if held is None else held
        if not self.need <= held < raw_rows:
            raise ValueError(f"held {held} not in [{self.need}, {raw_rows})")
        p0 = max(0, t0 - held)
        bf = torch.bfloat16
        self.n_max, self.n1_max = max_len // pc.m, max_len // ph.m
        self.kv = torch.zeros((B, self.n_max, pc.D_qk), dtype=bf, device=device)
        self.keys = torch.zeros((B, self.n_max, pc.d_I), dtype=bf, device=device)
        self.ent = torch.zeros((B, self.n1_max, ph.D_qk), dtype=bf, device=device)
        self.n_csa, self.n_hca = t0 // pc.m, t0 // ph.m
        width = {"x0": pc.D_qk, "g0": pc.D_qk, "xi0": pc.d_I, "gi0": pc.d_I, "x1": ph.D_qk,
                 "g1": ph.D_qk}
        self.raw = {k: torch.zeros((B, raw_rows, w), dtype=bf, device=device)
                    for k, w in width.items()}
        self.rows = SlidingRows(self.raw, p0, t0)
        self.bias0, self.bias_i0, self.bias1 = bias0, bias_i0, bias1
        self.out0 = torch.empty((B, 1, pc.H, pc.D_v), dtype=bf, device=device)
        self.out1 = torch.empty((B, 1, ph.H, ph.D_v), dtype=bf, device=device)
        nb = csa.workspace_size(pc, csa.WS_FORWARD, 1, self.n_max)
        self.ws0 = torch.empty(max(nb, 16), dtype=torch.uint8, device=device)
        nb = csa.workspace_size(ph, csa.WS_HCA, 1, self.n1_max)
        self.ws1 = torch.empty(max(nb, 16), dtype=torch.uint8, device=device)
        self.kv_rows, self.key_rows = csa.rows(self.kv), csa.rows(self.keys)
        self.ent_rows = csa.rows(self.ent)
        self.x1_rows = csa.rows(self.raw["x1"])

    # ------------------------------------------------------------ buffers
    @property
    def p0(self) -> int:
        """Position held in row 0 of the raw buffers."""
        return self.rows.p0

    @property
    def position(self) -> int:
        """Position of the token the next ``step`` takes."""
        return self.t + 1

    def seed(self, name: str, rows: torch.Tensor):
        """Rows of positions p0 .. t0-1 of one raw tensor ([B, t0 - p0, w])."""
        n = self.t + 1 - self.p0
        if rows.shape[1] != n:
            raise ValueError(f"{name}: {rows.shape[1]} rows, the buffer holds {n} before t0")
        self.raw[name][:, :n].copy_(rows)

    def _keep_from(self) -> int:
        """First position the next token still needs: the pending (not yet
        cached) block of each layer and both windows."""
        t = self.t + 1
        return min(self.n_csa * self.pc.m, self.n_hca * self.ph.m, t - self.pc.window + 1,
                   t - self.ph.window + 1)

    def slot(self, name: str) -> torch.Tensor:
        """Where the next token's row of raw tensor ``name`` goes ([B, 1, w]);
        valid until the next ``step``."""
        self.rows.room(self._keep_from())
        return self.rows.slot(name)

    def rewind(self, t0: int):
        """Drop the tokens from position t0 on: the next ``step`` takes t0
        again.  The rows of positions p0 .. t0-1 must still be in the buffers
        (p0 <= max(0, t0 - need)); the cache entries of blocks that end at or
        after t0 are rewritten by the steps that complete them."""
        if not (self.p0 <= max(0, t0 - self.need) and t0 <= self.t + 1):
            raise ValueError(f"cannot rewind to {t0}: the buffers hold {self.p0} .. {self.t}")
        self.t = t0 - 1
        self.n_csa, self.n_hca = t0 // self.pc.m, t0 // self.ph.m
        self.rows.t_next = t0

    # ---------------------------------------------------------- one token
    def step(self, q0, q_idx0, w0, q1, stream=None):
        """Run both layers for the next token, whose raw rows are in its
        slots.  q0 [B, 1, H, D_qk], q_idx0 [B, 1, H_I, d_I], w0 [B, 1, H_I]
        (CSA layer); q1 [B, 1, H', D_qk'] (HCA layer).  Returns the two
        outputs [B, 1, H, D_v] (owned by the decoder, overwritten by the next
        step)."""
        t = self.t + 1
        if t >= self.max_len:
            raise ValueError(f"position {t} beyond max_len {self.max_len}")
        self.rows.room(self._keep_from())
        self.rows.advance()
        self.t = t
        pc, ph, raw = self.pc, self.ph, self.raw
        # CSA layer: compress the block t completes (if any), index, top-k,
        # attend over the selected entries and the window
        args = csa.forward_args(x=raw["x0"], gate=raw["g0"], bias=self.bias0, xi=raw["xi0"],
                                gate_i=raw["gi0"], bias_i=self.bias_i0, raw_pos0=self.p0, q=q0,
                                q_idx=q_idx0, w=w0, q_pos0=t, kv=self.kv_rows,
                                keys=self.key_rows, n_cached=self.n_csa, out=self.out0)
        csa.forward(pc, args, self.ws0, stream=stream)
        self.n_csa = (t + 1) // pc.m
        # HCA layer: pool the 128-token block t completes, attend over every
        # entry and the window
        n1 = (t + 1) // ph.m
        if n1 > self.n_hca:
            csa.compress(raw["x1"], raw["g1"], self.bias1, ph.m, self.n_hca, n1, self.ent_rows,
                         x_pos0=self.p0, stream=stream)
            self.n_hca = n1
        csa.hca(ph, q1, self.ent_rows, self.x1_rows, self.p0, t, n1, self.out1,
                ws=self.ws1, stream=stream)
        return self.out0, self.out1

    def selected(self) -> torch.Tensor:
        """The CSA layer's selected entry indices of the last step ([B, k],
        ascending, -1 padded): the forward workspace holds the scores
        [B, 1, N] then, 256-byte aligned, the index lists."""
        N = (self.t + 1) // self.pc.m
        off = (self.B * N * 4 + 255) // 256 * 256
        n = self.B * self.pc.k
        return self.ws0[off: off + n * 4].view(torch.int32).view(self.B, self.pc.k)
