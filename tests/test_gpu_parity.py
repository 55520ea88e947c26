"""CUDA path vs the CPU oracle, element by element, on seeded inputs.

Sizes the oracle finishes in seconds that still span several tiles and a
ragged tail; the full-size workloads sit in test_gpu_fullsize.py."""

import numpy as np
import pytest
import torch

import oracle as O
from long_context_sparse_25_b300 import csa, synth
from long_context_sparse_25_b300.pipeline import Step

from harness import (SeqOracle, cached_keys_f64, check_out, check_scores, check_scores_bf16,
                     check_selection, check_selection_bf16, f64)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CSA_CASES = {
    # fp32 tiny workload at its full size: every query
    "tiny_f32": (W["csa_tiny_f32"], None),
    # bf16 prefill, ragged length (2051 tokens -> 512 entries + 3-token tail)
    "prefill_bf16_ragged": (W["csa_prefill_64k"].replace(L=2051, Q=2051, k=32), 160),
    # bf16 prefill with the real k=1024 and more entries than k
    "prefill_bf16_8k": (W["csa_prefill_64k"].replace(L=8192, Q=8192), 48),
    # bf16 decode, 5000 entries (ragged w.r.t. 128-key tiles), batch 3
    "decode_bf16": (W["csa_decode_1m"].replace(B=3, L=20000), None),
    # mixed e4m3 + bf16 decode, 5001 entries
    "decode_mixed": (W["csa_decode_fp8_512k"].replace(B=2, L=20004), None),
    # a decode step with two new tokens per sequence (the first sees one entry
    # fewer): the tensor-core indexer's causal schedule with one query per block
    "decode_bf16_q2": (W["csa_decode_1m"].replace(B=2, L=20000, Q=2), None),
    # raw-token attention (the 4 raw tokens of every selected block, then the
    # window): decode over 5000 entries, and an 8K prefill
    "decode_raw": (W["csa_decode_raw_1m"].replace(B=3, L=20000), None),
    # indexer scores stored in bf16: decode (multi-CTA top-k over 16-bit keys)
    # and a prefill (one CTA per row)
    "decode_bf16_scores": (W["csa_decode_1m_bf16s"].replace(B=3, L=80000), None),
    # FP4 indexer keys converted to FP8 in the indexer (a multi-CTA top-k row)
    "decode_fp4_keys": (W["csa_decode_fp4_512k"].replace(B=2, L=80004), None),
    "prefill_bf16_scores_ragged": (W["csa_prefill_64k"].replace(L=2051, Q=2051, k=32,
                                                                scores="bf16"), 160),
    "prefill_raw_8k": (W["csa_prefill_64k"].replace(L=8192, Q=8192, attend="raw"), 24),
    # raw-token attention through the CUDA-core path (fp32)
    "tiny_raw_f32": (W["csa_tiny_f32"].replace(L=1024, Q=1024, attend="raw"), None),
}


def _query_sample(wl, n):
    if n is None or n >= wl.Q:
        return np.arange(wl.Q)
    rng = np.random.default_rng(wl.seed + 17)
    head = np.arange(min(8, wl.Q))
    tail = np.arange(max(0, wl.Q - 8), wl.Q)
    mid = rng.choice(wl.Q, size=n, replace=False)
    return np.unique(np.concatenate([head, mid, tail]))


def _run(wl, dev):
    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
    step.run()
    torch.cuda.synchronize()
    csa.device_status()  # no bounded device-side wait gave up
    return inp, step


@pytest.mark.parametrize("case", list(CSA_CASES))
def test_csa_forward_matches_oracle(case, cuda_device):
    wl, nsample = CSA_CASES[case]
    inp, step = _run(wl, cuda_device)
    qs = _query_sample(wl, nsample)
    out = f64(step.out)
    sel = step.selected().cpu().numpy()
    scores = step.scores().cpu().double().numpy()
    decode = wl.mode.endswith("decode")
    for b in range(wl.B):
        o = SeqOracle(wl, inp, b)
        # step 1: compressed entries and indexer keys (new rows only)
        n0 = wl.N - 1 if decode else 0
        if wl.dtype == "mixed":
            got_kv = O.dequantize_rows_e4m3(inp["kv_nope"][b, n0:].cpu().view(torch.uint8).numpy(),
                                            inp["kv_scale"][b, n0:].cpu().numpy(),
                                            inp["kv_rope"][b, n0:].cpu().view(torch.int16).numpy().view(np.uint16))
            got_keys = cached_keys_f64(wl, inp, b, slice(n0, None))
        else:
            kvt = inp["kv"] if decode else step.kv_buf
            kt = inp["keys"] if decode else step.keys_buf
            got_kv, got_keys = f64(kvt[b, n0:]), f64(kt[b, n0:])
        if wl.dtype == "f32":
            np.testing.assert_allclose(got_kv, o.new_kv, rtol=2e-6, atol=2e-6)
            np.testing.assert_allclose(got_keys, o.new_keys, rtol=2e-6, atol=2e-6)
        else:
            # bf16 nearest to the exact value / e4m3 decided in float64: identical
            assert np.array_equal(got_keys, o.new_keys), "indexer keys differ from the oracle"
            assert np.array_equal(got_kv, o.new_kv), "entries differ from the oracle"
        # step 2: scores; step 3: selection; step 4: attention on the GPU's set
        ref_scores = o.scores(qs)
        if wl.scores == "bf16":
            nv = O.n_vis(o.positions(qs), wl.m)
            # the fused forward leaves the invisible part unwritten
            vis = np.arange(wl.N)[None, :] < nv[:, None]
            check_scores_bf16(np.where(vis, scores[b, qs], -np.inf), ref_scores)
            check_selection_bf16(sel[b, qs], ref_scores, nv, wl.k)
        else:
            check_scores(scores[b, qs], ref_scores)
            check_selection(sel[b, qs], ref_scores, O.n_vis(o.positions(qs), wl.m), wl.k)
        ref_out = o.attend(qs, sel[b, qs])
        check_out(out[b, qs], ref_out, wl.dtype == "f32", unit_scale=wl.outliers == 0)


HCA_CASES = {
    "hca_prefill_ragged": W["hca_prefill_1m"].replace(L=128 * 100 + 57, Q=300),
    "hca_decode": W["hca_decode_1m"].replace(B=3, L=128 * 300),
}


@pytest.mark.parametrize("case", list(HCA_CASES))
def test_hca_matches_oracle(case, cuda_device):
    wl = HCA_CASES[case]
    inp, step = _run(wl, cuda_device)
    out = f64(step.out)
    decode = wl.mode.endswith("decode")
    n0 = wl.N - 1 if decode else 0
    for b in range(wl.B):
        o = SeqOracle(wl, inp, b)
        got_kv = f64((inp["kv"] if decode else step.kv_buf)[b, n0:])
        # m' = 128 > 16: fp32 pooling rounded once to bf16 -> at most one bf16
        # ulp of the oracle's value away, plus the fp32 evaluation error (which
        # is relative to sum w|x| ~ 1, not to the possibly cancelled result)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(o.new_kv), 1e-30))) - 7)
        assert np.all(np.abs(got_kv - o.new_kv) <= ulp + 1e-6), "HCA entries off by more than 1 ulp"
        qs = np.arange(wl.Q)
        check_out(out[b], o.hca(qs), False)


def test_topk_bit_exact_on_oracle_scores(cuda_device):
    """csa_topk fed fp32 scores (with many exact ties, signed zeros, -inf
    beyond visibility) returns exactly the oracle's index lists."""
    rng = np.random.default_rng(5)
    # rows held in shared memory, long rows over several CTAs (16-byte score
    # loads; N % 4 != 0 takes the scalar filter; visible lengths that end
    # inside a 4-score group), rows shorter than k, and a row of all-equal
    # scores
    for (B, Q, N, k, m, q_pos0) in [(2, 37, 700, 64, 4, 2700), (1, 5, 20000, 1024, 4, 79999),
                                     (3, 9, 300, 1024, 4, 1000), (1, 300, 16384, 1024, 4, 65235),
                                     (2, 7, 1001, 256, 4, 3998), (1, 3, 20001, 1024, 4, 80003),
                                     (1, 4, 20000, 1024, 4, 70000)]:
        s = rng.standard_normal((B, Q, N))
        s = np.where(rng.uniform(size=s.shape) < 0.3, np.round(s, 1), s)  # ties
        s = np.where(rng.uniform(size=s.shape) < 0.05, 0.0, s)
        s = np.where(rng.uniform(size=s.shape) < 0.05, -0.0, s)
        s[0, 0, :] = 1.5  # one row of all-equal scores
        s32 = s.astype(np.float32)
        pos = q_pos0 + np.arange(Q)
        nv = O.n_vis(pos, m)
        s32 = np.where(np.arange(N)[None, None] < nv[None, :, None], s32, -np.inf).astype(np.float32)
        p = csa.params(B, m, k=k)
        idx = torch.empty((B, Q, k), dtype=torch.int32, device=cuda_device)
        csa.topk(p, torch.from_numpy(s32).to(cuda_device), q_pos0, idx)
        got = idx.cpu().numpy()
        for b in range(B):
            ref = O.topk(s32[b].astype(np.float64), pos, m, k)
            assert np.array_equal(got[b], ref)


def test_topk_bit_exact_on_oracle_bf16_scores(cuda_device):
    """csa_topk_ex fed the oracle's bf16 scores (csa.topk with a bf16 tensor)
    returns exactly the oracle's index lists: many ties (bf16 keeps 8 bits),
    signed zeros, -inf beyond visibility; rows in shared memory, long rows
    over several CTAs, rows shorter than k."""
    rng = np.random.default_rng(11)
    for (B, Q, N, k, m, q_pos0) in [(2, 37, 700, 64, 4, 2700), (1, 5, 20000, 1024, 4, 79999),
                                     (3, 9, 300, 1024, 4, 1000), (2, 3, 262144, 1024, 4, 1048575),
                                     (2, 7, 1001, 256, 4, 3998), (1, 3, 20003, 512, 4, 80011),
                                     (1, 4, 20000, 1024, 4, 70000)]:
        s = rng.standard_normal((B, Q, N))
        s = np.where(rng.uniform(size=s.shape) < 0.05, 0.0, s)
        s = np.where(rng.uniform(size=s.shape) < 0.05, -0.0, s)
        s16 = O.round_to_bf16(s)
        pos = q_pos0 + np.arange(Q)
        nv = O.n_vis(pos, m)
        s16 = np.where(np.arange(N)[None, None] < nv[None, :, None], s16, -np.inf)
        dev = torch.from_numpy(O.encode_bf16(s16).view(np.int16)).view(torch.bfloat16).to(cuda_device)
        p = csa.params(B, m, k=k)
        idx = torch.empty((B, Q, k), dtype=torch.int32, device=cuda_device)
        csa.topk(p, dev, q_pos0, idx)
        got = idx.cpu().numpy()
        for b in range(B):
            assert np.array_equal(got[b], O.topk(s16[b], pos, m, k)), (B, Q, N, b)


def test_topk_long_row_whose_sample_misleads(cuda_device):
    """A long row whose largest scores sit exactly at the evenly spaced
    positions the multi-CTA path samples (4096 of n): too few keys reach the
    sampled threshold, and the path must fall back to an exact select over
    the whole row.  Output must equal the oracle's index list."""
    rng = np.random.default_rng(9)
    N, k, m = 20000, 1024, 4
    q_pos0 = m * N - 1
    s = rng.standard_normal((1, 1, N)).astype(np.float32)
    ns = 4096
    pos = (np.arange(ns, dtype=np.int64) * N) // ns
    s[0, 0, pos] = 100.0 + np.arange(ns, dtype=np.float32) * 1e-3
    p = csa.params(1, m, k=k)
    idx = torch.empty((1, 1, k), dtype=torch.int32, device=cuda_device)
    csa.topk(p, torch.from_numpy(s).to(cuda_device), q_pos0, idx)
    ref = O.topk(s[0].astype(np.float64), np.array([q_pos0]), m, k)
    assert np.array_equal(idx[0].cpu().numpy(), ref)


@pytest.mark.parametrize("case", ["prefill_bf16_ragged", "decode_mixed", "tiny_f32"])
def test_index_call_matches_oracle_with_invisible_fill(case, cuda_device):
    """The public csa_index call: scores of visible entries within 1e-5 of the
    row scale and exactly -inf beyond each query's visibility."""
    wl, nsample = CSA_CASES[case]
    inp, step = _run(wl, cuda_device)  # fills the caches
    scores = torch.full((wl.B, wl.Q, wl.N), 7.0, device=cuda_device)
    csa.index(step.p, inp["q_idx"], inp["w"], step.keys, wl.q_pos0, wl.N, scores,
              q_scale=inp.get("q_idx_scale"))
    torch.cuda.synchronize()
    csa.device_status()
    qs = _query_sample(wl, nsample)
    got = scores.cpu().double().numpy()
    for b in range(wl.B):
        o = SeqOracle(wl, inp, b)
        check_scores(got[b, qs], o.scores(qs), check_invisible=True)


def test_batch_invariance_and_determinism(cuda_device):
    """A sequence gives bitwise the same output alone or at any batch slot,
    and two runs give bitwise the same output."""
    wl = W["csa_decode_1m"].replace(B=4, L=12000)
    inp, step = _run(wl, cuda_device)
    first = step.out.clone()
    step.run()
    torch.cuda.synchronize()
    assert torch.equal(first, step.out)
    for b in (0, 2):
        one = {k: (v if k in ("bias", "bias_i") else v[b: b + 1].contiguous()) for k, v in inp.items()}
        s1 = Step(wl.replace(B=1), one)
        s1.run()
        torch.cuda.synchronize()
        assert torch.equal(s1.out[0], first[b]), f"sequence {b} differs alone"


def test_empty_and_degenerate_cases(cuda_device):
    """Queries that see no entry (t < m-1) and W = 0 give zeros; Q = 0 and
    N = 0 launch nothing and succeed."""
    wl = W["csa_tiny_f32"].replace(L=16, Q=16, W=0, k=4)
    inp, step = _run(wl, cuda_device)
    out = step.out.cpu()
    assert torch.count_nonzero(out[0, :3]) == 0  # positions 0..2: no visible entry, no window
    o = SeqOracle(wl, inp, 0)
    qs = np.arange(wl.Q)
    check_out(f64(step.out[0]), o.attend(qs, step.selected()[0].cpu().numpy()), True)
    p = csa.params(1, 4, 16, 128, 128, 4, 64, 4, 0, 1.0)
    empty = torch.empty((1, 0, 4, 64), device=cuda_device)
    csa.index(p, empty, torch.empty((1, 0, 4), device=cuda_device), csa.rows(inp["xi"]), 0, 0,
              torch.empty((1, 0, 0), device=cuda_device))


@pytest.mark.parametrize("Q,dense", [(1, False), (3, False), (2, True)])
def test_attend_rescale_holes_and_order(Q, dense, cuda_device):
    """csa_attend / hca_attend called directly on crafted keys: logits that
    grow by several nats from one 128-key tile to the next (the running
    maximum must be raised and the partial output rescaled), -1 holes in the
    middle of an index list, an index list in descending order, and window
    rows; compared with the oracle on the same index lists."""
    rng = np.random.default_rng(11 + Q)
    B, H, D, Dv, W, m = 2, 128, 576, 512, 5, 4
    N, k = 700, 400
    L = N * m + 3
    q_pos0 = L - Q
    q = rng.standard_normal((B, Q, H, D)) / np.sqrt(D)
    kv = rng.standard_normal((B, N, D))
    # keys aligned with head 0's query, ever more strongly with the entry index
    # (and so with the tile), so the maximum keeps growing across tiles
    ramp = np.linspace(0.0, 14.0, N)[None, :, None]
    kv = kv + ramp * q[:, :1, 0, :] * np.sqrt(D)
    raw = rng.standard_normal((B, W + Q + 3, D))
    raw_pos0 = L - raw.shape[1]
    to_bf = lambda a: torch.from_numpy(O.round_to_bf16(a).astype(np.float32)).to(torch.bfloat16).to(cuda_device)
    tq, tkv, traw = to_bf(q), to_bf(kv), to_bf(raw)
    scale = 1.0 / np.sqrt(D)
    p = csa.params(B, m if not dense else 128, H, D, Dv, 1, 64, k, W, scale)
    out = torch.empty((B, Q, H, Dv), dtype=torch.bfloat16, device=cuda_device)
    if dense:
        n_ent = 300
        p = csa.params(B, 1, H, D, Dv, 1, 64, 0, W, scale)
        q_pos0 = n_ent - Q  # m = 1: query t sees entries 0..t
        raw = rng.standard_normal((B, W + Q + 3, D))
        raw_pos0 = q_pos0 + Q - raw.shape[1]
        traw = to_bf(raw)
        csa.hca(p, tq, csa.rows(tkv), csa.rows(traw), raw_pos0, q_pos0, N, out)
    else:
        idx = np.full((B, Q, k), -1, dtype=np.int32)
        for b in range(B):
            for i in range(Q):
                sel = np.sort(rng.choice(N, size=k - 40, replace=False))
                if i == 1:
                    sel = sel[::-1]
                row = np.concatenate([sel[:150], -np.ones(40, dtype=np.int64), sel[150:]])
                idx[b, i, :row.size] = row
        tidx = torch.from_numpy(idx).to(cuda_device)
        csa.attend(p, tq, csa.rows(tkv), csa.rows(traw), raw_pos0, tidx, q_pos0, N, out)
    torch.cuda.synchronize()
    csa.device_status()
    got = f64(out)
    for b in range(B):
        qv, kvv, rawv = f64(tq[b]), f64(tkv[b]), f64(traw[b])
        pos = q_pos0 + np.arange(Q)
        if dense:
            ref = O.hca_attend(qv, kvv, rawv, raw_pos0, pos, 1, W, Dv, scale)
        else:
            ref = O.csa_attend(qv, kvv, rawv, raw_pos0, idx[b], pos, W, Dv, scale)
        check_out(got[b], ref, False, unit_scale=False)  # keys grow to ~14x unit scale
