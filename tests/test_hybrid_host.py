"""Host bookkeeping of the hybrid decoder, on the CPU: the sliding raw-row
buffers keep every row a step reads, and the decoder hands the library the
right positions, cached counts and block ranges.  The library's compute calls
are replaced by recorders that check the buffers they would read."""

import numpy as np
import pytest
import torch

from long_context_sparse_25_b300 import csa, hybrid


def _pos_row(t: int, width: int) -> torch.Tensor:
    """A row that encodes position t exactly in bf16 (two base-256 digits)."""
    r = torch.zeros(width)
    r[0], r[1] = t // 256, t % 256
    return r


def _held(buf: torch.Tensor, p0: int, lo: int, hi: int):
    """Every row of positions lo .. hi-1 (all sequences) encodes its position."""
    assert lo >= p0 and hi - p0 <= buf.shape[1], (lo, hi, p0, buf.shape[1])
    v = buf[:, lo - p0: hi - p0, :2].float()
    got = (v[..., 0] * 256 + v[..., 1]).numpy()
    want = np.arange(lo, hi)[None, :].repeat(buf.shape[0], 0)
    assert np.array_equal(got, want), f"rows [{lo}, {hi}) do not hold their positions"


def test_sliding_rows_keep_what_is_asked():
    rng = np.random.default_rng(0)
    bufs = {"a": torch.zeros((2, 40, 2), dtype=torch.bfloat16),
            "b": torch.zeros((2, 40, 3), dtype=torch.bfloat16)}
    sr = hybrid.SlidingRows(bufs, p0=100, t_next=100)
    moved = 0
    for t in range(100, 1500):
        keep = t - int(rng.integers(0, 21))
        p_before = sr.p0
        sr.room(keep)
        moved += sr.p0 != p_before
        for name, buf in bufs.items():
            sr.slot(name).copy_(_pos_row(t, buf.shape[2]).expand(2, 1, -1))
        sr.advance()
        for buf in bufs.values():
            _held(buf, sr.p0, max(keep, sr.p0), t + 1)
    assert moved > 30


def test_sliding_rows_refuse_an_overlapping_move():
    bufs = {"a": torch.zeros((1, 8, 2), dtype=torch.bfloat16)}
    sr = hybrid.SlidingRows(bufs, p0=0, t_next=8)
    with pytest.raises(ValueError):
        sr.room(2)  # 6 rows kept of 8: source and destination overlap
    sr.room(4)
    assert sr.p0 == 4


class _Recorder:
    """Stands in for the library's compute calls and checks what they read."""

    def __init__(self, dec):
        self.dec = dec
        self.forward_calls, self.compress_calls, self.hca_calls = [], [], []

    def forward_args(self, **kw):
        return kw

    def forward(self, p, a, ws, stream=None):
        dec, m, W = self.dec, p.m, p.window
        t, p0 = a["q_pos0"], a["raw_pos0"]
        n = (t + 1) // m
        assert a["n_cached"] in (n, n - 1), "more than one block pending"
        # the window and the rows of the blocks the call compresses
        for name in ("x0", "g0", "xi0", "gi0"):
            _held(dec.raw[name], p0, max(0, t - W + 1), t + 1)
            if n > a["n_cached"]:
                _held(dec.raw[name], p0, a["n_cached"] * m, n * m)
        self.forward_calls.append((t, a["n_cached"]))

    def compress(self, x, gate, bias, m, s_begin, s_end, out, x_pos0=0, stream=None):
        _held(x, x_pos0, s_begin * m, s_end * m)
        _held(gate, x_pos0, s_begin * m, s_end * m)
        self.compress_calls.append((s_begin, s_end))

    def hca(self, p, q, kv, raw, raw_pos0, q_pos0, N, out, ws=None, stream=None):
        t = q_pos0
        assert N == (t + 1) // p.m
        _held(self.dec.raw["x1"], raw_pos0, max(0, t - p.window + 1), t + 1)
        self.hca_calls.append((t, N))


@pytest.mark.parametrize("t0", [0, 5, 130, 1000])
def test_decoder_bookkeeping(monkeypatch, t0):
    pc = csa.params(2, 4, 1, 8, 8, 1, 8, 4, 8, 1.0)
    ph = csa.params(2, 16, 1, 8, 8, 0, 0, 0, 12, 1.0)
    monkeypatch.setattr(csa, "workspace_size", lambda *a: 16)
    dec = hybrid.HybridDecoder(pc, ph, t0=t0, max_len=4096, device="cpu",
                               bias0=None, bias_i0=None, bias1=None, raw_rows=60,
                               held=min(40, max(t0, 28)) if t0 else 28)
    rec = _Recorder(dec)
    for name in ("forward_args", "forward", "compress", "hca"):
        monkeypatch.setattr(csa, name, getattr(rec, name))
    for name in hybrid.RAW_NAMES:
        n = t0 - dec.p0
        rows = torch.stack([_pos_row(p, dec.raw[name].shape[2]) for p in range(dec.p0, t0)]) \
            if n else torch.zeros((0, dec.raw[name].shape[2]))
        dec.seed(name, rows.unsqueeze(0).expand(2, -1, -1))
    S = 400
    for s in range(S):
        t = dec.position
        for name in hybrid.RAW_NAMES:
            dec.slot(name).copy_(_pos_row(t, dec.raw[name].shape[2]).expand(2, 1, -1))
        dec.step(None, None, None, None)
    ts = list(range(t0, t0 + S))
    assert [c[0] for c in rec.forward_calls] == ts
    assert [c[1] for c in rec.forward_calls] == [t // 4 for t in ts]
    assert rec.compress_calls == [((t + 1) // 16 - 1, (t + 1) // 16) for t in ts
                                  if (t + 1) % 16 == 0]
    assert rec.hca_calls == [(t, (t + 1) // 16) for t in ts]
    assert dec.n_csa == (t0 + S) // 4 and dec.n_hca == (t0 + S) // 16
    assert dec.p0 > t0  # the buffers moved


def test_decoder_rewind(monkeypatch):
    pc = csa.params(1, 4, 1, 8, 8, 1, 8, 4, 8, 1.0)
    ph = csa.params(1, 16, 1, 8, 8, 0, 0, 0, 8, 1.0)
    monkeypatch.setattr(csa, "workspace_size", lambda *a: 16)
    t0 = 100
    dec = hybrid.HybridDecoder(pc, ph, t0=t0, max_len=4096, device="cpu", bias0=None,
                               bias_i0=None, bias1=None, raw_rows=200, held=24)
    rec = _Recorder(dec)
    for name in ("forward_args", "forward", "compress", "hca"):
        monkeypatch.setattr(csa, name, getattr(rec, name))
    for name in hybrid.RAW_NAMES:
        w = dec.raw[name].shape[2]
        dec.seed(name, torch.stack([_pos_row(p, w) for p in range(dec.p0, t0)]).unsqueeze(0))

    def run(n):
        for _ in range(n):
            t = dec.position
            for name in hybrid.RAW_NAMES:
                dec.slot(name).copy_(_pos_row(t, dec.raw[name].shape[2]).expand(1, 1, -1))
            dec.step(None, None, None, None)

    run(40)
    first = (list(rec.forward_calls), list(rec.compress_calls), list(rec.hca_calls))
    dec.rewind(t0)
    rec.forward_calls, rec.compress_calls, rec.hca_calls = [], [], []
    run(40)
    assert (rec.forward_calls, rec.compress_calls, rec.hca_calls) == first
    with pytest.raises(ValueError):
        dec.rewind(dec.p0 + 3)  # rows before p0 are gone
