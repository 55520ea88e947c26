"""Parity at the full size of the timed workloads, in the launch configuration
bench.py times.  CSA decode at 1M-token context, B = 32 (262,144 entries per
sequence, one csa_forward per step) and mixed-precision CSA decode at 512K,
B = 64: every sequence's compressed tail entry and key bit-exact, every
visible score within 1e-5 of the row scale, the selection within the swap
rule; the attention output on a fixed sample of 8 sequences (the oracle
evaluates the 1152 keys each query keeps).  HCA decode at 1M, B = 32: every
sequence.  CSA prefill at 64K tokens and HCA prefill at 1M tokens on fixed
query samples."""

import numpy as np
import pytest
import torch

import oracle as O
from long_context_sparse_25_b300 import csa, synth
from long_context_sparse_25_b300.pipeline import Step

from harness import DeviceRows, check_out, check_scores, check_selection, f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _decode_parity(wl, dev, attn_seqs):
    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
    step.run()
    torch.cuda.synchronize()
    csa.device_status()  # no bounded device-side wait gave up
    N, m = wl.N, wl.m
    pos = np.array([wl.q_pos0])
    sel_all = step.selected().cpu().numpy()
    out = f64(step.out)
    mixed = wl.dtype == "mixed"
    for b in range(wl.B):
        x, g = f64(inp["x"][b]), f64(inp["g"][b])
        xi, gi = f64(inp["xi"][b]), f64(inp["gi"][b])
        a = (N - 1) * m - wl.raw_pos0
        new_key = O.store_rows(O.compress(xi[a:a + m], gi[a:a + m], f64(inp["bias_i"]), m),
                               "e4m3" if mixed else "bf16")
        new_kv = O.store_rows(O.compress(x[a:a + m], g[a:a + m], f64(inp["bias"]), m),
                              "e4m3" if mixed else "bf16", wl.D_v)
        if mixed:
            keys = O.dequantize_rows_e4m3(inp["keys"][b].cpu().view(torch.uint8).numpy(),
                                          inp["keys_scale"][b].cpu().numpy())
            qi = O.dequantize_rows_e4m3(inp["q_idx"][b].cpu().view(torch.uint8).numpy(),
                                        inp["q_idx_scale"][b].cpu().numpy())
        else:
            keys = f64(inp["keys"][b])
            qi = f64(inp["q_idx"][b])
        # the GPU's tail rows were written in place; they must equal the oracle's
        assert np.array_equal(keys[N - 1], new_key[0]), f"seq {b}: tail indexer key"
        keys = np.array(keys)
        keys[N - 1] = new_key[0]
        ref = O.index_scores(qi, f64(inp["w"][b]), keys, pos, m)
        check_scores(step.scores()[b].cpu().double().numpy(), ref)
        check_selection(sel_all[b], ref, O.n_vis(pos, m), wl.k)
        if b in attn_seqs and wl.attend == "raw":
            o = O.csa_attend_raw(f64(inp["q"][b]), DeviceRows(inp["x_all"][b]), 0, sel_all[b],
                                 pos, m, wl.W, wl.D_v, wl.scale)
            check_out(out[b], o, False)
        elif b in attn_seqs:
            s = sel_all[b, 0]
            s = s[s >= 0]
            rows = torch.from_numpy(s).to(dev).long()
            if mixed:
                ent = O.dequantize_rows_e4m3(inp["kv_nope"][b][rows].cpu().view(torch.uint8).numpy(),
                                             inp["kv_scale"][b][rows].cpu().numpy(),
                                             inp["kv_rope"][b][rows].cpu().view(torch.int16).numpy().view(np.uint16))
            else:
                ent = f64(inp["kv"][b][rows])
            last = np.flatnonzero(s == N - 1)
            if last.size:
                assert np.array_equal(ent[last[0]], new_kv[0]), f"seq {b}: tail entry"
            o = O.csa_attend(f64(inp["q"][b]), ent, x, wl.raw_pos0, np.arange(s.size)[None], pos,
                             wl.W, wl.D_v, wl.scale)
            check_out(out[b], o, False, unit_scale=wl.outliers == 0)


def test_decode_1m_full_size(cuda_device):
    wl = synth.WORKLOADS["csa_decode_1m"]
    _decode_parity(wl, cuda_device, attn_seqs={0, 5, 11, 16, 21, 26, 30, 31})


def test_decode_raw_1m_full_size(cuda_device):
    """The raw-token attention at the headline decode size (B = 32, 2^20
    positions, the raw KV rows of every position resident): per query the
    4 raw tokens of each of the 1024 selected blocks plus the 128-token window
    (4,224 keys, 33 tiles, split runs with the combine); scores and selection
    as for the entry path, attention on a fixed sample of 8 sequences."""
    wl = synth.WORKLOADS["csa_decode_raw_1m"]
    _decode_parity(wl, cuda_device, attn_seqs={0, 5, 11, 16, 21, 26, 30, 31})


def test_decode_fp8_512k_full_size(cuda_device):
    """Mixed-precision CSA decode at 512K context, B = 64 (131,072 entries per
    sequence, e4m3 nope dims with a row scale, bf16 RoPE dims, e4m3 indexer
    keys and queries, 1% x20 outliers), in the launch configuration bench.py
    times: rows above 16,384 entries take the multi-CTA top-k, and the e4m3
    indexer runs its full schedule.  Every sequence's tail entry and key equal
    the oracle's (quantised from float64), every visible score within 1e-5 of
    the row scale, the selection within the swap rule; attention on a fixed
    sample of 8 sequences."""
    wl = synth.WORKLOADS["csa_decode_fp8_512k"]
    _decode_parity(wl, cuda_device, attn_seqs={0, 9, 18, 27, 36, 45, 54, 63})


def test_hca_decode_1m_full_size(cuda_device):
    """HCA decode at 2^20 tokens, B = 32 (8,192 entries of m' = 128 raw rows per
    sequence), in the launch configuration bench.py times (csa_compress of the
    block the token completes, then hca_attend): the key list of 8,192 entries
    plus 128 window rows is 65 tiles, cut into split runs whose full tiles of
    consecutive entries load as TMA boxes, merged by the combine kernel.  Every
    sequence's tail entry within one bf16 ulp of the oracle's and every
    sequence's attention output checked."""
    wl = synth.WORKLOADS["hca_decode_1m"]
    dev = cuda_device
    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
    step.run()
    torch.cuda.synchronize()
    csa.device_status()  # no bounded device-side wait gave up
    N, m = wl.N, wl.m
    pos = np.array([wl.q_pos0])
    out = f64(step.out)
    bias = f64(inp["bias"])
    for b in range(wl.B):
        x, g = f64(inp["x"][b]), f64(inp["g"][b])
        a = (N - 1) * m - wl.raw_pos0
        tail = O.compress(x[a:a + m], g[a:a + m], bias, m)[0]
        kv = f64(inp["kv"][b])
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(tail), 1e-30))) - 7)
        assert np.all(np.abs(kv[N - 1] - tail) <= ulp + 1e-6), f"seq {b}: tail entry off by > 1 ulp"
        o = O.hca_attend(f64(inp["q"][b]), kv, x, wl.raw_pos0, pos, m, wl.W, wl.D_v, wl.scale)
        check_out(out[b], o, False)


def test_prefill_64k_full_size(cuda_device):
    """CSA prefill at 65,536 tokens (16,384 entries, k = 1024, 128 heads), in
    the launch configuration bench.py times (one csa_forward): every
    compressed entry and indexer key bit-exact; scores, selection and
    attention output on a fixed query sample (the first 128 queries, every
    256th, the last 128)."""
    wl = synth.WORKLOADS["csa_prefill_64k"]
    dev = cuda_device
    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
    step.run()
    torch.cuda.synchronize()
    csa.device_status()  # no bounded device-side wait gave up
    m, N = wl.m, wl.N
    qs = np.unique(np.concatenate([np.arange(128), np.arange(0, wl.Q, 256),
                                   np.arange(wl.Q - 128, wl.Q)]))
    x, g = f64(inp["x"][0]), f64(inp["g"][0])
    xi, gi = f64(inp["xi"][0]), f64(inp["gi"][0])
    kv = O.store_rows(O.compress(x, g, f64(inp["bias"]), m), "bf16")
    keys = O.store_rows(O.compress(xi, gi, f64(inp["bias_i"]), m), "bf16")
    assert np.array_equal(f64(step.kv_buf[0]), kv), "compressed entries differ"
    assert np.array_equal(f64(step.keys_buf[0]), keys), "indexer keys differ"
    pos = wl.q_pos0 + qs
    tq = torch.from_numpy(qs).to(dev).long()
    ref = O.index_scores(f64(inp["q_idx"][0][tq]), f64(inp["w"][0][tq]), keys, pos, m)
    check_scores(step.scores()[0][tq].cpu().double().numpy(), ref)
    sel = step.selected()[0][tq].cpu().numpy()
    check_selection(sel, ref, O.n_vis(pos, m), wl.k)
    o = O.csa_attend(f64(inp["q"][0][tq]), kv, x, wl.raw_pos0, sel, pos, wl.W, wl.D_v, wl.scale)
    check_out(f64(step.out[0][tq]), o, False)


def test_hca_prefill_1m_full_size(cuda_device):
    """HCA prefill at 2^20 tokens (8,192 entries of m' = 128 raw rows, the
    last 8,192 queries, 128 heads), in the launch configuration bench.py
    times (csa_compress, then hca_attend): every compressed entry within one
    bf16 ulp of the oracle's (fp32 pooling rounded once), and the attention
    output of a fixed query sample (the first 4, 8 spread over the rest, the
    last 4).  Late queries see all 8,192 entries, 64 full tiles of
    consecutive entry rows."""
    wl = synth.WORKLOADS["hca_prefill_1m"]
    dev = cuda_device
    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
    step.run()
    torch.cuda.synchronize()
    csa.device_status()  # no bounded device-side wait gave up
    m, N = wl.m, wl.N
    got = f64(step.kv_buf[0])
    ents = np.empty_like(got)
    bias = f64(inp["bias"])
    per = 512  # entries per oracle call (bounded host memory)
    for e0 in range(0, N, per):
        e1 = min(N, e0 + per)
        a, b_ = e0 * m - wl.raw_pos0, e1 * m - wl.raw_pos0
        ents[e0:e1] = O.compress(f64(inp["x"][0][a:b_]), f64(inp["g"][0][a:b_]), bias, m)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ents), 1e-30))) - 7)
    assert np.all(np.abs(got - ents) <= ulp + 1e-6), "HCA entries off by more than 1 ulp"
    stored = O.store_rows(ents, "bf16")
    qs = np.unique(np.concatenate([np.arange(4), np.linspace(0, wl.Q - 1, 8).astype(int),
                                   np.arange(wl.Q - 4, wl.Q)]))
    tq = torch.from_numpy(qs).to(dev).long()
    q = f64(inp["q"][0][tq])
    ref = np.empty((qs.size, wl.H, wl.D_v))
    for j, i in enumerate(qs):
        t = wl.q_pos0 + int(i)
        lo, hi = O.window_range(t, wl.W)
        raw = f64(inp["x"][0][lo - wl.raw_pos0: hi - wl.raw_pos0])  # the query's window rows
        ref[j] = O.hca_attend(q[j:j + 1], stored, raw, lo, np.array([t]), m, wl.W, wl.D_v,
                              wl.scale)[0]
    check_out(f64(step.out[0][tq]), ref, False)
