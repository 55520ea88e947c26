"""Pins of the CPU oracle against facts fixed outside the oracle itself:
closed forms, invariants of the method, special cases that reduce to a
library routine (torch scaled_dot_product_attention, numpy matmul / sort,
torch's float8 / bfloat16 casts) and brute force on tiny inputs.

Each test is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign or axis, an off-by-one in visibility or the window, a transposed
operand) makes it fail."""

import math

import numpy as np
import pytest
import torch

import oracle as O

rng = np.random.default_rng(1234)


# ----------------------------------------------------------------- formats
def test_bf16_decode_all_codes_match_torch():
    u = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = O.decode_bf16(u)
    assert np.all((np.isnan(ref) & np.isnan(got)) | (ref == got))


def test_bf16_round_matches_torch_on_fp32_values():
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-40, 40, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.encode_bf16(x.astype(np.float64)), ref)


def test_bf16_round_is_nearest_even_on_fp64_midpoints():
    # values just around bf16 midpoints, below fp32 resolution: the rounding
    # must be decided from the float64 value (no double rounding)
    base = O.decode_bf16(rng.integers(0x3000, 0x4f00, 5000).astype(np.uint16))
    ulp = np.ldexp(1.0, (np.floor(np.log2(base)) - 7).astype(int))
    for off, expect_up in ((0.5 + 2.0 ** -30, True), (0.5 - 2.0 ** -30, False)):
        r = O.round_to_bf16(base + off * ulp)
        assert np.array_equal(r, base + ulp if expect_up else base)
    # exact midpoints go to the even neighbour
    r = O.round_to_bf16(base + 0.5 * ulp)
    even = (O.encode_bf16(r) & 1) == 0
    assert even.all()


def test_e4m3_decode_all_codes_match_torch():
    u = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(u).view(torch.float8_e4m3fn).double().numpy()
    got = O.decode_e4m3(u)
    assert np.all((np.isnan(ref) & np.isnan(got)) | (ref == got))


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-14, 6, 200000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.encode_e4m3(x.astype(np.float64)), ref)
    big = np.array([449.0, 463.9, 464.0, 1e6, -500.0])
    assert np.array_equal(O.decode_e4m3(O.encode_e4m3(big)), [448, 448, 448, 448, -448])


def test_mixed_rows_roundtrip_error_bound():
    v = rng.standard_normal((64, 576))
    q = O.quantize_rows_e4m3(v, 512)
    back = O.dequantize_rows_e4m3(q["codes"], q["scale"], q["rope"])
    amax = np.abs(v[:, :512]).max(axis=1, keepdims=True)
    # e4m3 has 3 mantissa bits: relative half-spacing 2^-4 in the normal range,
    # absolute 2^-10 * scale in the subnormal range
    err = np.abs(back[:, :512] - v[:, :512])
    assert np.all(err <= np.maximum(np.abs(v[:, :512]) * 2.0 ** -4, amax / 448 * 2.0 ** -10) * 1.0001)
    assert np.array_equal(back[:, 512:], O.round_to_bf16(v[:, 512:]))
    # the largest element maps to the largest code 448 (or just below by scale rounding)
    assert np.all(np.abs(O.decode_e4m3(q["codes"])).max(axis=1) >= 416)


# ----------------------------------------------------------------- compress
def test_compress_weights_sum_to_one_and_positive():
    g = rng.standard_normal((64, 9))
    b = 0.1 * rng.standard_normal((4, 9))
    w = O.compress_weights(g, b, 4)
    assert w.shape == (16, 4, 9)
    assert np.all(w > 0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_compress_identical_tokens_give_that_token():
    tok = rng.standard_normal(7)
    x = np.tile(tok, (8, 1))
    e = O.compress(x, rng.standard_normal((8, 7)), rng.standard_normal((4, 7)), 4)
    np.testing.assert_allclose(e, np.tile(tok, (2, 1)), rtol=1e-15, atol=1e-15)


def test_compress_m1_is_identity():
    x = rng.standard_normal((5, 3))
    assert np.array_equal(O.compress(x, rng.standard_normal((5, 3)), rng.standard_normal((1, 3)), 1), x)


def test_compress_zero_gates_and_bias_is_block_mean():
    x = rng.standard_normal((12, 5))
    e = O.compress(x, np.zeros((12, 5)), np.zeros((4, 5)), 4)
    np.testing.assert_allclose(e, x.reshape(3, 4, 5).mean(axis=1), rtol=1e-14, atol=1e-15)


def test_compress_gate_shift_invariance():
    x = rng.standard_normal((8, 6))
    g = rng.standard_normal((8, 6))
    b = rng.standard_normal((4, 6))
    shift = np.repeat(rng.standard_normal((2, 6)) * 5, 4, axis=0)  # per (block, channel)
    np.testing.assert_allclose(O.compress(x, g + shift, b, 4), O.compress(x, g, b, 4), rtol=1e-12,
                               atol=1e-13)


def test_compress_bias_selects_position_per_channel():
    # a huge bias on position i of channel c makes the entry take token i there
    m, C = 4, 6
    x = rng.standard_normal((8, C))
    bias = np.zeros((m, C))
    pick = np.array([0, 3, 1, 2, 3, 0])
    bias[pick, np.arange(C)] = 1000.0
    e = O.compress(x, rng.standard_normal((8, C)), bias, m)
    want = np.stack([x[blk * m + pick, np.arange(C)] for blk in range(2)])
    np.testing.assert_allclose(e, want, rtol=0, atol=1e-300)


def test_compress_drops_partial_tail():
    assert O.compress(rng.standard_normal((11, 2)), rng.standard_normal((11, 2)), np.zeros((4, 2)), 4).shape == (2, 2)


# ----------------------------------------------------------------- indexer
def test_n_vis_matches_definition():
    for m in (1, 4, 128):
        for t in range(0, 600, 7):
            brute = sum(1 for s in range(1000) if (s + 1) * m - 1 <= t)
            assert O.n_vis(t, m) == brute


def test_index_single_head_nonnegative_is_matmul():
    q = np.abs(rng.standard_normal((6, 1, 16)))
    k = np.abs(rng.standard_normal((10, 16)))
    pos = np.arange(34, 40)  # m=4: n_vis = 8 .. 10
    got = O.index_scores(q, np.ones((6, 1)), k, pos, 4)
    ref = np.matmul(q[:, 0, :], k.T)
    vis = np.arange(10)[None] < ((pos + 1) // 4)[:, None]
    assert np.array_equal(np.isinf(got), ~vis)
    np.testing.assert_allclose(got[vis], ref[vis], rtol=1e-14)


def test_index_relu_clamps_negative_heads():
    k = rng.standard_normal((4, 8))
    q = np.stack([k[2], -k[2]])[None]  # head 0 aligned with key 2, head 1 opposite
    got = O.index_scores(q, np.array([[0.3, 0.7]]), k, np.array([100]), 4)
    assert got[0, 2] == pytest.approx(0.3 * float(k[2] @ k[2]), rel=1e-14)
    # every key: head 1 contributes only where its dot product is positive
    d0, d1 = q[0, 0] @ k.T, q[0, 1] @ k.T
    np.testing.assert_allclose(got[0], 0.3 * np.maximum(d0, 0) + 0.7 * np.maximum(d1, 0), rtol=1e-14)


def test_index_brute_force_tiny():
    Q, H_I, d, N, m = 3, 3, 5, 7, 2
    q = rng.standard_normal((Q, H_I, d))
    w = rng.uniform(0, 1, (Q, H_I))
    k = rng.standard_normal((N, d))
    pos = np.array([3, 8, 13])
    got = O.index_scores(q, w, k, pos, m)
    for i in range(Q):
        for s in range(N):
            if (s + 1) * m - 1 <= pos[i]:
                val = 0.0
                for j in range(H_I):
                    dot = sum(q[i, j, c] * k[s, c] for c in range(d))
                    val += w[i, j] * max(0.0, dot)
                assert got[i, s] == pytest.approx(val, rel=1e-13, abs=1e-14)
            else:
                assert got[i, s] == -math.inf


def test_index_linear_in_w():
    q = rng.standard_normal((4, 5, 8))
    k = rng.standard_normal((9, 8))
    w1, w2 = rng.uniform(0, 1, (4, 5)), rng.uniform(0, 1, (4, 5))
    pos = np.full(4, 100)
    np.testing.assert_allclose(O.index_scores(q, w1 + w2, k, pos, 4),
                               O.index_scores(q, w1, k, pos, 4) + O.index_scores(q, w2, k, pos, 4),
                               rtol=1e-13)


# ----------------------------------------------------------------- top-k
def test_topk_matches_stable_argsort():
    for _ in range(200):
        n = int(rng.integers(1, 300))
        k = int(rng.integers(1, 64))
        row = np.round(rng.standard_normal(n), int(rng.integers(0, 3)))  # plenty of ties
        got = O.topk_row(row, n, k)
        ref = np.sort(np.argsort(-row, kind="stable")[: min(k, n)])
        assert np.array_equal(got, ref)


def test_topk_brute_force_invariants_with_zero_ties():
    for _ in range(300):
        n = int(rng.integers(1, 12))
        k = int(rng.integers(1, 8))
        row = rng.choice([0.0, -0.0, 1.0, 2.0, -1.0], size=n)
        sel = O.topk_row(row, n, k)
        kk = min(k, n)
        assert sel.size == kk and len(set(sel.tolist())) == kk
        assert np.all(np.diff(sel) > 0) and np.all(sel < n)
        uns = np.setdiff1d(np.arange(n), sel)
        if uns.size and sel.size:
            assert row[sel].min() >= row[uns].max()
            tau = row[sel].min()
            # ties at tau resolved to lower indices (signed zeros are equal)
            tie_sel = sel[row[sel] == tau]
            tie_uns = uns[row[uns] == tau]
            if tie_uns.size:
                assert tie_sel.max() < tie_uns.min()


def test_topk_fewer_visible_than_k_pads():
    scores = rng.standard_normal((3, 20))
    pos = np.array([2, 9, 79])  # m=4: n_vis = 0, 2, 20
    out = O.topk(scores, pos, 4, 5)
    assert np.array_equal(out[0], [-1] * 5)
    assert np.array_equal(out[1], [0, 1, -1, -1, -1])
    assert np.array_equal(out[2], np.sort(np.argsort(-scores[2], kind="stable")[:5]))


# ----------------------------------------------------------------- attention
def _sdpa(q, k, v, scale, mask=None, causal=False):
    # q [Q, H, D] -> [H, Q, D]; MQA: one k/v for every head
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k)[None].expand(q.shape[1], -1, -1)
    vt = torch.from_numpy(v)[None].expand(q.shape[1], -1, -1)
    am = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am,
                                                         is_causal=causal, scale=scale)
    return o.permute(1, 0, 2).numpy()


def _dense_case(T=24, H=3, D=10, D_v=7):
    x = rng.standard_normal((T, D))
    q = rng.standard_normal((T, H, D))
    return x, q, D_v


def test_csa_m1_allk_nowindow_is_dense_causal_mqa():
    x, q, D_v = _dense_case()
    T, D = x.shape
    out, sel, _ = O.csa_pipeline(x=x, g=rng.standard_normal(x.shape), bias=np.zeros((1, D)),
                                 xi=rng.standard_normal((T, 4)), gi=rng.standard_normal((T, 4)),
                                 bias_i=np.zeros((1, 4)), q=q,
                                 q_idx=rng.standard_normal((T, 2, 4)), w=rng.uniform(0, 1, (T, 2)),
                                 m=1, k=T, W=0, D_v=D_v, scale=0.37, q_pos=np.arange(T),
                                 kv_dtype="f64", key_dtype="f64")
    ref = _sdpa(q, x, x[:, :D_v], 0.37, causal=True)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_hca_m1_nowindow_is_dense_causal_mqa():
    x, q, D_v = _dense_case()
    out = O.hca_attend(q, x, x, 0, np.arange(x.shape[0]), 1, 0, D_v, 0.21)
    np.testing.assert_allclose(out, _sdpa(q, x, x[:, :D_v], 0.21, causal=True), rtol=1e-12,
                               atol=1e-13)


def test_window_keys_duplicate_entries_as_log2_bias():
    # m = 1, all entries selected, window W: every window token is a key twice,
    # which equals one copy with +log 2 on its logit
    x, q, D_v = _dense_case(T=20)
    T = x.shape[0]
    W, scale = 5, 0.3
    sel = [np.arange(t + 1) for t in range(T)]
    out = O.csa_attend(q, x, x, 0, sel, np.arange(T), W, D_v, scale)
    mask = np.full((T, T), -np.inf)
    for t in range(T):
        mask[t, : t + 1] = 0.0
        mask[t, max(0, t - W + 1): t + 1] = math.log(2.0)
    np.testing.assert_allclose(out, _sdpa(q, x, x[:, :D_v], scale, mask=mask), rtol=1e-12,
                               atol=1e-13)


def test_hca_window_and_blocks_brute_force():
    # m = 4: query t sees entries s with 4s+3 <= t and raw tokens t-W+1..t
    T, m, W, D, H = 23, 4, 3, 6, 2
    e = rng.standard_normal((T // m, D))
    raw = rng.standard_normal((T, D))
    q = rng.standard_normal((T, H, D))
    out = O.hca_attend(q, e, raw, 0, np.arange(T), m, W, 4, 0.5)
    for t in (0, 2, 3, 7, 22):
        keys = [e[s] for s in range(T // m) if 4 * s + 3 <= t] + [raw[u] for u in range(max(0, t - W + 1), t + 1)]
        K = np.array(keys)
        for h in range(H):
            lg = np.array([0.5 * float(q[t, h] @ kk) for kk in K])
            p = np.exp(lg - lg.max())
            p /= p.sum()
            np.testing.assert_allclose(out[t, h], p @ K[:, :4], rtol=1e-12, atol=1e-14)


def test_attend_single_key_and_identical_keys_return_value():
    k = rng.standard_normal((1, 9))
    q = rng.standard_normal((4, 9))
    np.testing.assert_allclose(O.attend_keys(q, k, 6, 1.0), np.tile(k[0, :6], (4, 1)), rtol=1e-15)
    np.testing.assert_allclose(O.attend_keys(q, np.tile(k, (5, 1)), 6, 1.0), np.tile(k[0, :6], (4, 1)),
                               rtol=1e-14)
    assert np.array_equal(O.attend_keys(q, np.zeros((0, 9)), 6, 1.0), np.zeros((4, 6)))


def test_attend_invariant_to_selection_order():
    e = rng.standard_normal((30, 8))
    q = rng.standard_normal((1, 3, 8))
    sel = np.array([[3, 7, 11, 20, 29]])
    a = O.csa_attend(q, e, e, 0, sel, np.array([200]), 0, 8, 0.4)
    b = O.csa_attend(q, e, e, 0, sel[:, ::-1], np.array([200]), 0, 8, 0.4)
    np.testing.assert_allclose(a, b, rtol=1e-13)


def test_pipeline_selects_exactly_k_visible_entries():
    T, m, k = 64, 4, 5
    out, sel, scores = O.csa_pipeline(
        x=rng.standard_normal((T, 8)), g=rng.standard_normal((T, 8)), bias=rng.standard_normal((m, 8)),
        xi=rng.standard_normal((T, 4)), gi=rng.standard_normal((T, 4)), bias_i=rng.standard_normal((m, 4)),
        q=rng.standard_normal((T, 2, 8)), q_idx=rng.standard_normal((T, 3, 4)), w=rng.uniform(0, 1, (T, 3)),
        m=m, k=k, W=4, D_v=8, scale=0.3, q_pos=np.arange(T), kv_dtype="bf16", key_dtype="bf16")
    for t in range(T):
        nv = (t + 1) // m
        s = sel[t][sel[t] >= 0]
        assert s.size == min(k, nv)
        assert np.all(s < nv)


# ------------------------------------------- raw-row offset and the cache path
def test_window_rows_taken_by_absolute_position_when_raw_starts_late():
    """Raw rows that start at position raw_pos0 > 0: query t's window is the
    rows of absolute positions t-W+1 .. t.  The keys are assembled here by
    absolute position from the full token array and the result compared with
    torch's scaled_dot_product_attention; the oracle is given only the rows
    from raw_pos0 on."""
    T, W, D, D_v, H, scale = 40, 6, 10, 7, 3, 0.35
    x = rng.standard_normal((T, D))            # rows of absolute positions 0..T-1
    e = rng.standard_normal((9, D))            # cache entries
    pos = np.arange(30, T)
    q = rng.standard_normal((pos.size, H, D))
    sel = np.stack([np.sort(rng.choice(9, size=4, replace=False)) for _ in pos])
    r0 = 25                                    # first window row any query needs
    got = O.csa_attend(q, e, x[r0:], r0, sel, pos, W, D_v, scale)
    got_h = O.hca_attend(q, e, x[r0:], r0, pos, 4, W, D_v, scale)
    for i, t in enumerate(pos):
        win = x[t - W + 1: t + 1]
        keys = np.concatenate([e[sel[i]], win])
        ref = _sdpa(q[i:i + 1], keys, keys[:, :D_v], scale)
        np.testing.assert_allclose(got[i:i + 1], ref, rtol=1e-12, atol=1e-13)
        keys_h = np.concatenate([e[: (t + 1) // 4], win])  # entries ending at or before t
        ref_h = _sdpa(q[i:i + 1], keys_h, keys_h[:, :D_v], scale)
        np.testing.assert_allclose(got_h[i:i + 1], ref_h, rtol=1e-12, atol=1e-13)
    # the same rows through a view that starts at position 0 give bitwise the same result
    assert np.array_equal(got, O.csa_attend(q, e, x, 0, sel, pos, W, D_v, scale))
    assert np.array_equal(got_h, O.hca_attend(q, e, x, 0, pos, 4, W, D_v, scale))


def test_pipeline_reads_cached_entries_and_compresses_only_new_ones():
    """m = 1 (compression is the identity), W = 0, k >= entries: query t attends
    densely over entries 0..t.  Entries below n_cached must come from the
    caches (arbitrary rows here, unrelated to the raw rows) and the rest from
    the raw rows, which start at raw_pos0 > 0.  Checked against torch's
    scaled_dot_product_attention on keys assembled by hand."""
    T, D, D_v, H, dI, scale = 20, 8, 6, 2, 4, 0.4
    n_cached, r0 = 12, 12
    x_abs = rng.standard_normal((T, D))
    xi_abs = rng.standard_normal((T, dI))
    kv_cache = rng.standard_normal((T, D))
    key_cache = rng.standard_normal((T, dI))
    pos = np.arange(16, T)
    q = rng.standard_normal((pos.size, H, D))
    q_idx = rng.standard_normal((pos.size, 3, dI))
    w = rng.uniform(0, 1, (pos.size, 3))
    out, sel, scores = O.csa_pipeline(
        x=x_abs[r0:], g=rng.standard_normal((T - r0, D)), bias=np.zeros((1, D)),
        xi=xi_abs[r0:], gi=rng.standard_normal((T - r0, dI)), bias_i=np.zeros((1, dI)),
        q=q, q_idx=q_idx, w=w, m=1, k=T, W=0, D_v=D_v, scale=scale, q_pos=pos, raw_pos0=r0,
        kv_cache=kv_cache, key_cache=key_cache, n_cached=n_cached, kv_dtype="f64",
        key_dtype="f64")
    ents = np.concatenate([kv_cache[:n_cached], x_abs[n_cached:]])
    keys = np.concatenate([key_cache[:n_cached], xi_abs[n_cached:]])
    for i, t in enumerate(pos):
        assert np.array_equal(sel[i][sel[i] >= 0], np.arange(t + 1))
        ref = _sdpa(q[i:i + 1], ents[: t + 1], ents[: t + 1, :D_v], scale)
        np.testing.assert_allclose(out[i:i + 1], ref, rtol=1e-12, atol=1e-13)
        # indexer scores of the visible entries: keys from the cache, then the new rows
        dots = np.maximum(q_idx[i] @ keys[: t + 1].T, 0.0)
        np.testing.assert_allclose(scores[i, : t + 1], w[i] @ dots, rtol=1e-12, atol=1e-13)


def test_pipeline_with_a_filled_cache_equals_the_run_without_one():
    """m = 4, bf16 caches, window 5: running the pipeline on all raw rows from
    position 0 equals running it with the first n_cached entries already in
    the caches and only the raw rows from position n_cached*m on."""
    T, m, D, dI, H = 64, 4, 8, 4, 2
    x, g = rng.standard_normal((T, D)), rng.standard_normal((T, D))
    xi, gi = rng.standard_normal((T, dI)), rng.standard_normal((T, dI))
    bias, bias_i = 0.1 * rng.standard_normal((m, D)), 0.1 * rng.standard_normal((m, dI))
    pos = np.arange(50, T)
    q = rng.standard_normal((pos.size, H, D))
    q_idx, w = rng.standard_normal((pos.size, 3, dI)), rng.uniform(0, 1, (pos.size, 3))
    kw = dict(bias=bias, bias_i=bias_i, q=q, q_idx=q_idx, w=w, m=m, k=5, W=5, D_v=6, scale=0.3,
              q_pos=pos, kv_dtype="bf16", key_dtype="bf16")
    full = O.csa_pipeline(x=x, g=g, xi=xi, gi=gi, **kw)
    n_cached = 11  # entries 0..10 pool tokens 0..43
    r0 = n_cached * m
    kv_cache = np.zeros((T // m, D))
    key_cache = np.zeros((T // m, dI))
    kv_cache[:n_cached] = O.store_rows(O.compress(x[:r0], g[:r0], bias, m), "bf16")
    key_cache[:n_cached] = O.store_rows(O.compress(xi[:r0], gi[:r0], bias_i, m), "bf16")
    part = O.csa_pipeline(x=x[r0:], g=g[r0:], xi=xi[r0:], gi=gi[r0:], raw_pos0=r0,
                          kv_cache=kv_cache, key_cache=key_cache, n_cached=n_cached, **kw)
    for a, b in zip(full, part):
        assert np.array_equal(a, b)


# ------------------------------------------------ raw-token variant of the CSA attention
def test_raw_variant_with_m1_equals_the_entry_path():
    """m = 1: an entry is its one raw token (compression with m = 1 is the
    identity), so attending over the raw tokens of the selected blocks is
    attending over the selected entries."""
    x, q, D_v = _dense_case(T=30)
    T = x.shape[0]
    pos = np.arange(10, T)
    sel = np.stack([np.concatenate([np.sort(rng.choice(t + 1, size=6, replace=False)), [-1, -1]])
                    for t in pos])
    a = O.csa_attend_raw(q[10:], x, 0, sel, pos, 1, 4, D_v, 0.3)
    b = O.csa_attend(q[10:], x, x, 0, sel, pos, 4, D_v, 0.3)
    assert np.array_equal(a, b)


def test_raw_variant_all_blocks_no_window_is_block_causal_dense_attention():
    """m = 4, every visible block selected, W = 0: query t attends densely over
    the raw tokens 0 .. 4*n_vis(t)-1 (the tokens of its complete blocks);
    checked against torch's scaled_dot_product_attention with that mask."""
    T, m, H, D, D_v, scale = 26, 4, 3, 9, 5, 0.45
    x = rng.standard_normal((T, D))
    q = rng.standard_normal((T, H, D))
    pos = np.arange(T)
    nv = (pos + 1) // m
    sel = np.full((T, T // m), -1)
    for t in range(T):
        sel[t, : nv[t]] = rng.permutation(nv[t])  # any order: a set of keys
    got = O.csa_attend_raw(q, x, 0, sel, pos, m, 0, D_v, scale)
    mask = np.full((T, T), -np.inf)
    for t in range(T):
        mask[t, : nv[t] * m] = 0.0
    seen = nv > 0
    ref = _sdpa(q[seen], x, x[:, :D_v], scale, mask=mask[seen])
    np.testing.assert_allclose(got[seen], ref, rtol=1e-12, atol=1e-13)
    assert np.array_equal(got[~seen], np.zeros_like(got[~seen]))  # no key: zeros


def test_raw_variant_keys_by_absolute_position_with_window():
    """Raw rows that start at raw_pos0 > 0; the keys of each query are
    assembled here by absolute position (the 4 tokens of every selected block,
    then the window) and compared with torch's scaled_dot_product_attention."""
    T, m, W, H, D, D_v, scale = 64, 4, 5, 2, 8, 6, 0.3
    x = rng.standard_normal((T, D))
    pos = np.arange(56, T)
    q = rng.standard_normal((pos.size, H, D))
    sel = np.stack([np.sort(rng.choice((t + 1) // m, size=3, replace=False)) for t in pos])
    r0 = 16  # earliest selectable block below is 4 (tokens 16..19): make it so
    sel = np.maximum(sel, 4)
    sel = np.stack([np.unique(r)[:3] if np.unique(r).size >= 3 else np.array([4, 5, 6]) for r in sel])
    got = O.csa_attend_raw(q, x[r0:], r0, sel, pos, m, W, D_v, scale)
    for i, t in enumerate(pos):
        toks = [4 * s + j for s in sel[i] for j in range(4)] + list(range(t - W + 1, t + 1))
        keys = x[toks]
        ref = _sdpa(q[i:i + 1], keys, keys[:, :D_v], scale)
        np.testing.assert_allclose(got[i:i + 1], ref, rtol=1e-12, atol=1e-13)


# ------------------------------------------------- grouped output projection
def test_group_projection_brute_force_indices():
    """Every output element by an explicit sum over (head, dim) with the
    group's row index written out: pins the head-to-group assignment and the
    head-major concatenation inside a group."""
    T, H, D_v, G, d_g = 3, 6, 4, 3, 5
    o = rng.standard_normal((T, H, D_v))
    W = rng.standard_normal((G, (H // G) * D_v, d_g))
    y = O.group_output_projection(o, W)
    hg = H // G
    for t in range(T):
        for g in range(G):
            for n in range(d_g):
                acc = 0.0
                for h in range(g * hg, (g + 1) * hg):
                    for d in range(D_v):
                        acc += o[t, h, d] * W[g, (h - g * hg) * D_v + d, n]
                assert abs(y[t, g * d_g + n] - acc) <= 1e-12 * (1 + abs(acc))


def test_group_projection_is_the_block_diagonal_full_projection():
    """The grouped projection equals one projection of the flattened output
    [T, H*D_v] by the block-diagonal matrix of the group matrices (a matrix
    built with scipy, multiplied with numpy)."""
    from scipy.linalg import block_diag
    T, H, D_v, G, d_g = 7, 8, 16, 4, 12
    o = rng.standard_normal((T, H, D_v))
    W = rng.standard_normal((G, (H // G) * D_v, d_g))
    full = o.reshape(T, H * D_v) @ block_diag(*W)
    np.testing.assert_allclose(O.group_output_projection(o, W), full, rtol=1e-12, atol=1e-12)


def test_group_projection_one_group_is_a_plain_matmul_and_groups_are_local():
    T, H, D_v, d_g = 5, 4, 8, 6
    o = rng.standard_normal((T, H, D_v))
    W1 = rng.standard_normal((1, H * D_v, d_g))
    np.testing.assert_allclose(O.group_output_projection(o, W1),
                               np.matmul(o.reshape(T, -1), W1[0]), rtol=1e-12, atol=1e-12)
    # changing the heads of group 1 changes only group 1's columns
    G = 2
    W = rng.standard_normal((G, (H // G) * D_v, d_g))
    y0 = O.group_output_projection(o, W)
    o2 = o.copy()
    o2[:, 2:4, :] += 1.0
    y1 = O.group_output_projection(o2, W)
    assert np.array_equal(y0[:, :d_g], y1[:, :d_g])
    assert not np.allclose(y0[:, d_g:], y1[:, d_g:])


# ------------------------------------------------------- bf16 index scores
def test_bf16_index_scores_are_torch_rounded_scores_and_ties_go_low():
    """The bf16 scores equal torch's bf16 cast of the scores (through float32;
    the few scores whose float64 value lies within 2^-12 of a bf16 ulp from a
    rounding midpoint are left out, where float32 could round across it), -inf
    stays -inf, and the top-k over them breaks the many bf16 ties by the
    lower index."""
    g = np.random.default_rng(77)
    Q, H_I, d_I, N, m, k = 3, 4, 8, 600, 4, 37
    q = g.standard_normal((Q, H_I, d_I))
    keys = g.standard_normal((N, d_I))
    w = g.uniform(0, 1, (Q, H_I))
    pos = np.array([m * N - 1, 1000, 3])
    s64 = O.index_scores(q, w, keys, pos, m)
    s16 = O.index_scores_bf16(q, w, keys, pos, m)
    ref = torch.from_numpy(s64).float().to(torch.bfloat16).double().numpy()
    fin = np.isfinite(s64) & (s64 != 0)
    ulp = np.zeros_like(s64)
    ulp[fin] = 2.0 ** (np.floor(np.log2(np.abs(s64[fin]))) - 7)
    frac = np.zeros_like(s64)
    frac[fin] = np.abs(s64[fin]) / ulp[fin] % 1.0
    clear = ~fin | (np.abs(frac - 0.5) > 2.0 ** -12)
    assert clear.mean() > 0.99
    assert np.array_equal(s16[clear], ref[clear])
    assert np.array_equal(np.isneginf(s16), np.isneginf(s64))
    sel = O.topk(s16, pos, m, k)
    for i in range(Q):
        nv = int(min(O.n_vis(pos[i], m), N))
        kk = min(k, nv)
        order = np.lexsort((np.arange(nv), -s16[i, :nv]))  # score desc, then index asc
        assert np.array_equal(sel[i, :kk], np.sort(order[:kk]))
    # a tie group straddling the k-th place keeps only its lowest index
    vals, counts = np.unique(s16[0, :N], return_counts=True)
    tie = vals[counts > 1][-1]
    k2 = int(np.count_nonzero(s16[0, :N] > tie)) + 1
    sel2 = O.topk(s16[:1], pos[:1], m, k2)[0]
    group = np.flatnonzero(s16[0, :N] == tie)
    assert group[0] in sel2 and not np.isin(group[1:], sel2).any()


# ------------------------------------------------------------------ FP4 keys
def test_e2m1_values_are_e4m3_values_and_the_format_extremes():
    """Every E2M1 value converts to E4M3 without loss (the FP4 -> FP8 step of
    the indexer keys; the E4M3 codec is pinned against torch above), the codes
    0..7 increase from 0 through the smallest nonzero magnitude 0.5 to the
    largest 6, and codes 8..15 are their negatives."""
    c = np.arange(16, dtype=np.uint8)
    v = O.decode_e2m1(c)
    assert np.array_equal(O.decode_e4m3(O.encode_e4m3(v)), v)
    assert np.all(np.diff(v[:8]) > 0) and v[0] == 0 and v[1] == 0.5 and v[7] == 6.0
    assert np.array_equal(v[8:], -v[:8]) and np.signbit(v[8])


def test_e2m1_encode_is_nearest_with_ties_to_even_by_brute_force():
    g = np.random.default_rng(31)
    x = np.concatenate([g.uniform(-7, 7, 20000), np.arange(-6.5, 6.75, 0.25)])
    vals = O.decode_e2m1(np.arange(8, dtype=np.uint8))
    code = O.encode_e2m1(x)
    for xi, ci in zip(x, code):
        ax = min(abs(xi), 6.0)
        d = np.abs(vals - ax)
        best = np.flatnonzero(d == d.min())
        want = best[0] if best.size == 1 else [b for b in best if b % 2 == 0][0]
        assert (ci & 7) == want, (xi, ci)
        assert (ci >> 3) == (1 if np.signbit(xi) else 0)


def test_e2m1_rows_round_trip_within_half_a_spacing_and_keep_the_row_max():
    g = np.random.default_rng(32)
    v = g.standard_normal((50, 128))
    q = O.quantize_rows_e2m1(v)
    back = O.dequantize_rows_e2m1(q["codes"], q["scale"])
    s = q["scale"].astype(np.float64)[:, None]
    spacing = np.where(np.abs(v) / s < 2, 0.5, np.where(np.abs(v) / s < 4, 1.0, 2.0)) * s
    assert np.all(np.abs(back - v) <= spacing / 2 * (1 + 1e-6))
    i = np.argmax(np.abs(v), axis=1)
    r = np.arange(50)
    np.testing.assert_allclose(np.abs(back[r, i]), np.abs(v[r, i]), rtol=1e-6)
    # the row maximum takes the largest code magnitude (the scale is amax / 6)
    assert np.all((q["codes"][r, i] & 7) == 7)
