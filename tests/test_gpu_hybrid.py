"""Hybrid decoding on the GPU against the oracle recomputed from scratch.

A CSA layer and an HCA layer decode 12 consecutive tokens of 2 sequences
(production widths, k = 256) starting 5 tokens before a 128-token boundary:
the run crosses three CSA block boundaries and one HCA boundary, and the
sliding raw buffers move once.  The GPU caches before the first token are
filled by the library's own compression of the raw history; at every token
the oracle recomputes both layers from the raw rows of all positions 0 .. t
(compression, scores, top-k, attention), so a cache entry the decoder failed
to write, wrote twice or wrote at the wrong place shows up as an output or
selection mismatch.
"""

import numpy as np
import pytest
import torch

import oracle as O
from harness import check_out, check_selection, f64
from long_context_sparse_25_b300 import csa, hybrid, synth

pytestmark = pytest.mark.gpu

HW = synth.HYBRID["hybrid_decode_1m"].replace(B=2, t0=128 * 20 - 5, steps=12, k=256,
                                              history=True)


def _entries(x, g, bias, m, n):
    return O.store_rows(O.compress(x[: n * m], g[: n * m], bias, m), "bf16")


def test_hybrid_decode_matches_oracle(cuda_device):
    hw = HW
    dev = cuda_device
    inp = synth.make_hybrid_inputs(hw, dev)
    pc = csa.params(hw.B, hw.m, hw.H, hw.D_qk, hw.D_v, hw.H_I, hw.d_I, hw.k, hw.W, hw.scale)
    ph = csa.params(hw.B, hw.m1, hw.H, hw.D_qk, hw.D_v, 0, 0, 0, hw.W, hw.scale)
    t0, S = hw.t0, hw.steps
    dec = hybrid.HybridDecoder(pc, ph, t0=t0, max_len=t0 + S + 64, device=dev,
                               bias0=inp["bias0"], bias_i0=inp["bias_i0"], bias1=inp["bias1"],
                               raw_rows=518, held=512)
    # caches before t0: the library compresses the raw history
    n, n1 = t0 // hw.m, t0 // hw.m1
    csa.compress(inp["x0"][:, :t0].contiguous(), inp["g0"][:, :t0].contiguous(), inp["bias0"],
                 hw.m, 0, n, dec.kv_rows)
    csa.compress(inp["xi0"][:, :t0].contiguous(), inp["gi0"][:, :t0].contiguous(),
                 inp["bias_i0"], hw.m, 0, n, dec.key_rows)
    csa.compress(inp["x1"][:, :t0].contiguous(), inp["g1"][:, :t0].contiguous(), inp["bias1"],
                 hw.m1, 0, n1, dec.ent_rows)
    for name in hybrid.RAW_NAMES:
        dec.seed(name, inp[name][:, dec.p0:t0])
    torch.cuda.synchronize()

    raw = {name: [f64(inp[name][b]) for b in range(hw.B)] for name in hybrid.RAW_NAMES}
    bias = {k: f64(inp[k]) for k in ("bias0", "bias_i0", "bias1")}
    p0s = []
    for s in range(S):
        t = dec.position
        for name in hybrid.RAW_NAMES:
            dec.slot(name).copy_(inp[name][:, t:t + 1])
        out0, out1 = dec.step(inp["q0"][s], inp["q_idx0"][s], inp["w0"][s], inp["q1"][s])
        csa.device_status()
        p0s.append(dec.p0)
        sel = dec.selected().cpu().numpy()
        g0, g1 = f64(out0), f64(out1)
        nv, nv1 = (t + 1) // hw.m, (t + 1) // hw.m1
        for b in range(hw.B):
            kv = _entries(raw["x0"][b], raw["g0"][b], bias["bias0"], hw.m, nv)
            keys = _entries(raw["xi0"][b], raw["gi0"][b], bias["bias_i0"], hw.m, nv)
            qi, w = f64(inp["q_idx0"][s][b]), f64(inp["w0"][s][b])
            scores = O.index_scores(qi, w, keys, np.array([t]), hw.m)
            check_selection(sel[b:b + 1], scores, np.array([nv]), hw.k)
            ref0 = O.csa_attend(f64(inp["q0"][s][b]), kv, raw["x0"][b], 0, sel[b:b + 1],
                                np.array([t]), hw.W, hw.D_v, hw.scale)
            check_out(g0[b], ref0, f32=False)
            ent = _entries(raw["x1"][b], raw["g1"][b], bias["bias1"], hw.m1, nv1)
            ref1 = O.hca_attend(f64(inp["q1"][s][b]), ent, raw["x1"][b], 0, np.array([t]),
                                hw.m1, hw.W, hw.D_v, hw.scale)
            check_out(g1[b], ref1, f32=False)
    # the run crossed an HCA boundary and the buffers moved
    assert dec.n_hca == n1 + 1 and dec.n_csa == (t0 + S) // hw.m
    assert p0s[0] != p0s[-1]
    # the caches hold what the oracle compresses: the CSA entries and keys
    # are the bf16 nearest to the exact pooled value (identical), the HCA
    # entries (128-term sums) within one bf16 ulp
    for b in range(hw.B):
        nv, nv1 = dec.n_csa, dec.n_hca
        kv = _entries(raw["x0"][b], raw["g0"][b], bias["bias0"], hw.m, nv)
        keys = _entries(raw["xi0"][b], raw["gi0"][b], bias["bias_i0"], hw.m, nv)
        assert np.array_equal(f64(dec.kv[b, :nv]), kv), "CSA entries differ"
        assert np.array_equal(f64(dec.keys[b, :nv]), keys), "indexer keys differ"
        ent = _entries(raw["x1"][b], raw["g1"][b], bias["bias1"], hw.m1, nv1)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ent), 1e-30))) - 7)
        assert np.all(np.abs(f64(dec.ent[b, :nv1]) - ent) <= ulp + 1e-6), "HCA entries"
