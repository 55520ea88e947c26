"""float64 CPU oracle of the CSA / HCA forward pass (test infrastructure only).

Plain numpy, one step per function, in the order the pages give the method:

  1. compress   -- m adjacent tokens pooled into one entry by per-channel
                   softmax weights with a learned position bias;
  2. index      -- the lightning indexer scores every visible entry;
  3. top-k      -- each query keeps its k best entries;
  4. attend     -- shared-KV (MQA) attention over the kept entries plus a
                   sliding window of recent raw tokens;
  HCA           -- compress with m' = 128 and attend densely (no top-k).

Sources ("page title", section):
  [csdn]   "一文搞懂 DeepSeek：从 V3 的 KV 压缩与 MoE，到 V4 的百万 token 上下文",
           section "V4 改进一：CSA 与 HCA"; MLA layout in "V3 看家本领一：MLA".
  [yudong] "DeepSeek-V4 详解", section 2.2 Steps 1-4 (CSA), section 2.3
           Steps 1-2 (HCA).
  [jaylab] "DeepSeek-V4 — 百万 Token 上下文的高效 MoE 模型", section
           "3. Muon 优化器" (the bullet on RMSNorm of the attention queries and
           KV entries) and section "其他技术细节" (the bullet on the mixed
           BF16 / FP8 KV cache).

Readings where the pages are silent:
  * compression is a per-channel softmax over the m positions of
    (gate logit + bias[i]); the projections that produce X and the gates are
    upstream inputs;
  * indexer score = sum_j w[t,j] * ReLU(q_I[t,j] . K_I[s]) with one key per
    entry shared by all indexer heads;
  * entry s is visible to the query at position t iff (s+1)*m - 1 <= t;
  * the window holds tokens max(0, t-W+1) .. t, t included, and is not
    de-duplicated against the entries that cover the same tokens;
  * fewer than k visible entries -> all of them are kept; ties go to the lower
    entry index; -0.0 == +0.0;
  * scores use all D_qk = 576 dims; the value is the first D_v = 512 dims (the
    latent), as in MLA where the decoupled RoPE key only enters the score;
  * compressed entries are stored in the cache dtype (fp32 / bf16, or the
    mixed e4m3 + bf16 layout) before anything reads them.

  * the grouped output projection splits the H heads into G consecutive
    groups of H/G heads; group g's head outputs, concatenated head by head,
    are projected by its own matrix to d_g features, and the G results are
    concatenated in group order.

Nothing here is blocked, fused or reordered beyond what the steps state.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "decode_bf16", "encode_bf16", "round_to_bf16", "decode_e4m3", "encode_e4m3",
    "decode_e2m1", "encode_e2m1", "quantize_rows_e2m1", "dequantize_rows_e2m1",
    "round_to_f32", "quantize_rows_e4m3", "dequantize_rows_e4m3", "store_rows",
    "compress_weights", "compress", "n_vis", "index_scores", "index_scores_bf16", "topk_row",
    "topk",
    "window_range", "attend_keys", "csa_attend", "raw_block_tokens", "csa_attend_raw",
    "hca_attend", "csa_pipeline", "group_output_projection",
]

E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# Number formats (exact, written from the format definitions)
# ---------------------------------------------------------------------------

def decode_bf16(u16: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> exact float64 values.

    bfloat16 is the upper half of an IEEE binary32 word, so widening the bit
    pattern by 16 zero bits gives the binary32 value exactly.
    """
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significand bits (7 stored), exponent range as binary32.
    For |x| in [2^e, 2^(e+1)) the spacing is 2^(e-7); below the smallest
    normal 2^-126 the spacing is fixed at 2^-133.  numpy's ``round`` is
    round-half-to-even, applied to x / spacing which is exact (power of two).
    Values at or beyond the midpoint above the largest finite bfloat16
    (2 - 2^-8) * 2^127 round to infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    fin = np.isfinite(x) & (x != 0)
    ax = np.abs(x[fin])
    e = np.floor(np.log2(ax))
    # log2 may be off by one next to a power of two: fix it exactly.
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, -126.0)
    q = np.ldexp(1.0, (e - 7).astype(np.int64))
    r = np.round(ax / q) * q
    big = r > (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(big, np.inf, r)
    out[fin] = np.sign(x[fin]) * r
    nonfin = ~np.isfinite(x)
    out[nonfin] = x[nonfin]
    out[x == 0] = x[x == 0]
    return out


def encode_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bit patterns (round to nearest even)."""
    r = round_to_bf16(x).astype(np.float32)  # exact: a bf16 value is a binary32 value
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def decode_e4m3(u8: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 (the 'fn' variant) bit patterns -> float64.

    Layout s eeee mmm, exponent bias 7.  e == 0: subnormal (m/8) * 2^-6.
    e == 15 and m == 7: NaN (no infinities).  Otherwise (1 + m/8) * 2^(e-7).
    """
    b = np.asarray(u8, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6,
                   (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7)))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """float64 -> E4M3 bit patterns, round to nearest even, saturating.

    Magnitudes that round above the largest finite value 448 become 448 (the
    'satfinite' convention).  Spacing is 2^(e-3) for |x| in [2^e, 2^(e+1)),
    e >= -6, and 2^-9 in the subnormal range.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, -6.0)
    q = np.ldexp(1.0, (e - 3).astype(np.int64))
    r = np.round(ax / q) * q
    r = np.minimum(r, E4M3_MAX)
    # encode the (now representable) magnitude
    code = np.zeros(x.shape, dtype=np.int64)
    sub = r < 2.0 ** -6
    code = np.where(sub, np.round(r / 2.0 ** -9).astype(np.int64), code)
    rn = np.where(sub, 1.0, r)
    en = np.floor(np.log2(rn))
    en = np.where(np.ldexp(1.0, en.astype(np.int64)) > rn, en - 1, en)
    mn = np.round((rn / np.ldexp(1.0, en.astype(np.int64)) - 1.0) * 8).astype(np.int64)
    code = np.where(sub, code, ((en.astype(np.int64) + 7) << 3) | mn)
    sign = np.where(np.signbit(x), 0x80, 0)  # the sign survives rounding to zero
    return (code | sign).astype(np.uint8)


def decode_e2m1(u4: np.ndarray) -> np.ndarray:
    """FP4 E2M1 codes (one per uint8, values 0..15) -> float64.

    Layout s ee m, exponent bias 1, no infinities or NaN.  e == 0: subnormal
    m * 0.5; otherwise (1 + m/2) * 2^(e-1): the magnitudes 0, 0.5, 1, 1.5, 2,
    3, 4, 6.
    """
    b = np.asarray(u4, dtype=np.uint8).astype(np.int64) & 0xF
    s = np.where(b & 0x8, -1.0, 1.0)
    e = (b >> 1) & 0x3
    m = b & 0x1
    val = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.ldexp(1.0, e - 1))
    return s * val


def encode_e2m1(x: np.ndarray) -> np.ndarray:
    """float64 -> E2M1 codes (one per uint8), round to nearest even, saturating
    at +-6.  Spacing 0.5 below 2, 1 in [2, 4), 2 in [4, 6]; a tie goes to the
    code with an even mantissa bit."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.minimum(np.abs(x), 6.0)
    q = np.where(ax < 2.0, 0.5, np.where(ax < 4.0, 1.0, 2.0))
    r = np.round(ax / q) * q  # round half to even on the grid: even multiples win
    r = np.minimum(r, 6.0)
    # magnitude -> code: 0, .5, 1, 1.5, 2, 3, 4, 6 -> 0..7
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    code = np.searchsorted(mags, r)
    sign = np.where(np.signbit(x), 0x8, 0)
    return (code | sign).astype(np.uint8)


def quantize_rows_e2m1(v: np.ndarray) -> dict:
    """FP4 storage of indexer-key rows ([csdn] section "V4 的其他升级": the
    indexer's QK path is quantised to FP4 and dequantised to FP8 without
    loss): one float32 scale per row, amax / 6 (1.0 for an all-zero row), and
    each code the E2M1 rounding, taken directly from float64, of value /
    scale.  Codes are returned one per uint8 (the cache packs two per byte)."""
    v = np.asarray(v, dtype=np.float64)
    amax = np.max(np.abs(v), axis=-1)
    scale = np.where(amax > 0, amax / 6.0, 1.0).astype(np.float32)
    codes = encode_e2m1(v / scale.astype(np.float64)[..., None])
    return {"codes": codes, "scale": scale}


def dequantize_rows_e2m1(codes, scale) -> np.ndarray:
    """Exact float64 value of FP4 rows: code * scale."""
    return decode_e2m1(codes) * np.asarray(scale, dtype=np.float64)[..., None]


def round_to_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def quantize_rows_e4m3(v: np.ndarray, nope: int) -> dict:
    """Mixed-precision row storage: the first ``nope`` channels in E4M3 with one
    float32 scale per row, the remaining (RoPE) channels in bfloat16.

    [jaylab] section "其他技术细节", the KV-cache bullet: RoPE dims stay in
    BF16, the other dims are stored in FP8.  Reading: the scale
    is amax / 448 over the nope channels, rounded to float32 (1.0 for an
    all-zero row); each code is the E4M3 rounding, taken directly from float64,
    of value / scale.
    """
    v = np.asarray(v, dtype=np.float64)
    amax = np.max(np.abs(v[..., :nope]), axis=-1)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)
    codes = encode_e4m3(v[..., :nope] / scale.astype(np.float64)[..., None])
    rope = encode_bf16(v[..., nope:]) if v.shape[-1] > nope else None
    return {"codes": codes, "scale": scale, "rope": rope}


def dequantize_rows_e4m3(codes, scale, rope=None) -> np.ndarray:
    """Exact float64 value of mixed-precision rows: code * scale ++ bf16 rope."""
    nope = decode_e4m3(codes) * np.asarray(scale, dtype=np.float64)[..., None]
    if rope is None:
        return nope
    return np.concatenate([nope, decode_bf16(rope)], axis=-1)


def store_rows(v: np.ndarray, dtype: str, nope: int | None = None) -> np.ndarray:
    """Value the cache holds after storing float64 rows ``v`` in ``dtype``.

    'f32' and 'bf16' round each element to nearest even; 'e4m3' is the mixed
    layout of ``quantize_rows_e4m3`` (``nope`` leading channels quantised);
    'e2m1' the FP4 rows of ``quantize_rows_e2m1``.
    """
    if dtype == "f64":
        return np.asarray(v, dtype=np.float64)
    if dtype == "f32":
        return round_to_f32(v)
    if dtype == "bf16":
        return round_to_bf16(v)
    if dtype == "e4m3":
        q = quantize_rows_e4m3(v, v.shape[-1] if nope is None else nope)
        return dequantize_rows_e4m3(q["codes"], q["scale"], q["rope"])
    if dtype == "e2m1":
        q = quantize_rows_e2m1(v)
        return dequantize_rows_e2m1(q["codes"], q["scale"])
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# Step 1: compression ([csdn] section "V4 改进一：CSA 与 HCA", the first CSA
# step: m adjacent tokens pooled into one entry by softmax weights that carry
# a position bias; [yudong] 2.2 Step 1, and 2.3 Step 1 for m' = 128)
# ---------------------------------------------------------------------------

def compress_weights(g: np.ndarray, bias: np.ndarray, m: int) -> np.ndarray:
    """Pooling weights [T//m, m, C]: for each block and channel, the softmax over
    the block's m positions of (gate logit + position bias).  A trailing partial
    block (T % m tokens) is not compressed."""
    g = np.asarray(g, dtype=np.float64)
    n = g.shape[0] // m
    z = g[: n * m].reshape(n, m, -1) + np.asarray(bias, dtype=np.float64)[None]
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=1, keepdims=True)


def compress(x: np.ndarray, g: np.ndarray, bias: np.ndarray, m: int) -> np.ndarray:
    """Compressed entries [T//m, C]: E[s,c] = sum_i w[s,i,c] * x[s*m+i, c]."""
    x = np.asarray(x, dtype=np.float64)
    w = compress_weights(g, bias, m)
    n = w.shape[0]
    return (w * x[: n * m].reshape(n, m, -1)).sum(axis=1)


# ---------------------------------------------------------------------------
# Step 2: lightning indexer ([csdn] section "V4 改进一：CSA 与 HCA", the second
# CSA step: a light indexer scores each compressed entry against the query;
# [yudong] 2.2 Step 2)
# ---------------------------------------------------------------------------

def n_vis(t, m: int):
    """Number of entries a query at absolute position t may see: the blocks that
    end at or before t, i.e. entry s is visible iff (s+1)*m - 1 <= t."""
    return (np.asarray(t, dtype=np.int64) + 1) // m


def index_scores(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray,
                 q_pos: np.ndarray, m: int) -> np.ndarray:
    """Indexer scores [Q, N] for one sequence.

    q_idx [Q, H_I, d_I], w [Q, H_I], keys [N, d_I] (all float64 values, already
    dequantised).  I[t, s] = sum_j w[t,j] * max(0, q_idx[t,j] . keys[s]) for
    visible s; -inf where s is not yet visible to t.
    """
    q_idx = np.asarray(q_idx, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    Q, H_I, d_I = q_idx.shape
    N = keys.shape[0]
    dots = (q_idx.reshape(Q * H_I, d_I) @ keys.T).reshape(Q, H_I, N)
    scores = np.einsum("qj,qjn->qn", w, np.maximum(dots, 0.0))
    vis = np.arange(N)[None, :] < n_vis(np.asarray(q_pos), m)[:, None]
    return np.where(vis, scores, -np.inf)


def index_scores_bf16(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray,
                      q_pos: np.ndarray, m: int) -> np.ndarray:
    """The indexer scores stored in bf16 ([csdn] section "V4 的其他升级": the
    index scores drop to BF16, which doubles the speed of the top-k
    selection): each score of index_scores rounded to the nearest bf16 value
    (ties to even); invisible entries stay -inf.  The top-k then runs on these
    values, ties (now frequent) going to the lower index as before."""
    return round_to_bf16(index_scores(q_idx, w, keys, q_pos, m))


# ---------------------------------------------------------------------------
# Step 3: top-k ([csdn] section "V4 改进一：CSA 与 HCA": only the k best-scoring
# entries go on to attention; [yudong] 2.2 Step 3)
# ---------------------------------------------------------------------------

def topk_row(scores: np.ndarray, nv: int, k: int) -> np.ndarray:
    """Indices of the min(k, nv) best of scores[:nv], ascending.

    The kk-th largest value tau is found by partition; every score above tau
    is kept, then the lowest-index scores equal to tau fill the rest.
    (-0.0 == +0.0 under IEEE comparison, so signed zeros tie.)
    """
    cand = np.asarray(scores[:nv], dtype=np.float64)
    kk = min(k, nv)
    if kk <= 0:
        return np.zeros(0, dtype=np.int64)
    tau = np.partition(cand, nv - kk)[nv - kk]
    above = np.flatnonzero(cand > tau)
    ties = np.flatnonzero(cand == tau)
    sel = np.concatenate([above, ties[: kk - above.size]])
    return np.sort(sel)


def topk(scores: np.ndarray, q_pos: np.ndarray, m: int, k: int) -> np.ndarray:
    """[Q, k] int64 index lists, ascending, padded with -1."""
    Q = scores.shape[0]
    out = np.full((Q, k), -1, dtype=np.int64)
    nvs = n_vis(np.asarray(q_pos), m)
    for i in range(Q):
        nv = int(min(nvs[i], scores.shape[1]))
        sel = topk_row(scores[i], nv, k)
        out[i, : sel.size] = sel
    return out


# ---------------------------------------------------------------------------
# Step 4: shared-KV MQA over the kept entries plus the raw window
# ([csdn] section "V4 改进一：CSA 与 HCA": a short sliding window of recent raw
# KV is kept uncompressed, and attention is MQA over one shared KV; [yudong]
# 2.2 Step 4, 2.3 Step 2; value = latent part, as in [csdn] MLA)
# ---------------------------------------------------------------------------

def window_range(t: int, W: int) -> tuple[int, int]:
    """Raw tokens attended directly by a query at position t: [max(0,t-W+1), t]."""
    return max(0, t - W + 1), t + 1


def attend_keys(q_t: np.ndarray, keys: np.ndarray, D_v: int, scale: float) -> np.ndarray:
    """One query: q_t [H, D_qk], keys [n, D_qk] shared by all heads.
    o[h] = sum_j softmax_j(scale * q_t[h] . keys[j]) * keys[j, :D_v].
    An empty key set gives zeros."""
    H = q_t.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((H, D_v))
    logits = scale * (q_t @ keys.T)
    logits = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ keys[:, :D_v]


def csa_attend(q, entries, raw, raw_pos0: int, sel, q_pos, W: int, D_v: int,
               scale: float) -> np.ndarray:
    """CSA attention for one sequence.

    q [Q, H, D_qk]; entries [N, D_qk] (cache values); raw [R, D_qk] holding
    positions raw_pos0 .. raw_pos0+R-1; sel [Q, k] entry indices (-1 = none).
    Keys of query i: entries[sel[i]] followed by raw tokens of its window.
    """
    q = np.asarray(q, dtype=np.float64)
    Q, H, _ = q.shape
    out = np.zeros((Q, H, D_v))
    for i in range(Q):
        t = int(q_pos[i])
        s = np.asarray(sel[i])
        s = s[s >= 0]
        lo, hi = window_range(t, W)
        keys = np.concatenate([entries[s], raw[lo - raw_pos0: hi - raw_pos0]], axis=0)
        out[i] = attend_keys(q[i], keys, D_v, scale)
    return out


def raw_block_tokens(sel_row, m: int) -> np.ndarray:
    """Positions of the raw tokens inside the selected blocks, block by block in
    list order: entry s covers tokens s*m .. s*m+m-1 (-1 slots skipped)."""
    s = np.asarray(sel_row, dtype=np.int64)
    s = s[s >= 0]
    return (s[:, None] * m + np.arange(m, dtype=np.int64)[None, :]).ravel()


def csa_attend_raw(q, raw, raw_pos0: int, sel, q_pos, m: int, W: int, D_v: int,
                   scale: float) -> np.ndarray:
    """Raw-token variant of the CSA attention for one sequence ([yudong] 2.2
    Steps 3-4: the top blocks stand for the 4 original tokens each, and the
    attention runs over those original tokens; [hongke] 2.2, item 3: standard
    attention over the raw tokens inside the retrieved blocks).

    Keys of query i: the raw rows of the m tokens of every selected block, in
    list order, followed by the raw window of query i (kept, as in the entry
    path, without de-duplication).  The value is a key row's first D_v dims.
    raw [R, D_qk] holds positions raw_pos0 .. raw_pos0+R-1."""
    q = np.asarray(q, dtype=np.float64)
    Q, H, _ = q.shape
    out = np.zeros((Q, H, D_v))
    for i in range(Q):
        t = int(q_pos[i])
        toks = raw_block_tokens(sel[i], m)
        lo, hi = window_range(t, W)
        keys = np.concatenate([raw[toks - raw_pos0], raw[lo - raw_pos0: hi - raw_pos0]], axis=0)
        out[i] = attend_keys(q[i], keys, D_v, scale)
    return out


def hca_attend(q, entries, raw, raw_pos0: int, q_pos, m: int, W: int, D_v: int,
               scale: float) -> np.ndarray:
    """HCA attention for one sequence: every visible entry (no selection) plus
    the raw window ([csdn] section "V4 改进一：CSA 与 HCA": HCA entries are few
    enough to attend to all of them; [yudong] 2.3 Step 2)."""
    q = np.asarray(q, dtype=np.float64)
    Q, H, _ = q.shape
    out = np.zeros((Q, H, D_v))
    for i in range(Q):
        t = int(q_pos[i])
        nv = int(min(n_vis(t, m), entries.shape[0]))
        lo, hi = window_range(t, W)
        keys = np.concatenate([entries[:nv], raw[lo - raw_pos0: hi - raw_pos0]], axis=0)
        out[i] = attend_keys(q[i], keys, D_v, scale)
    return out


# ---------------------------------------------------------------------------
# The whole CSA forward for one sequence
# ---------------------------------------------------------------------------

def csa_pipeline(*, x, g, bias, xi, gi, bias_i, q, q_idx, w, m, k, W, D_v, scale,
                 q_pos, raw_pos0=0, kv_cache=None, key_cache=None, n_cached=0,
                 kv_dtype="f32", key_dtype="f32", kv_nope=None):
    """Steps 1-4 for one sequence; returns (out [Q,H,D_v], sel [Q,k], scores).

    x, g [R, D_qk] / xi, gi [R, d_I] are the raw rows for positions
    raw_pos0 .. raw_pos0+R-1 (KV and indexer-key inputs with their gate
    logits).  kv_cache / key_cache (float64 cache values, [N, .]) hold entries
    0 .. n_cached-1 when given; entries n_cached .. n_vis(last query)-1 are
    compressed from the raw rows and stored in the cache dtype.
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    n_end = int(n_vis(int(q_pos.max()), m))
    new = range(n_cached, n_end)
    d_qk = x.shape[1]
    entries = np.zeros((n_end, d_qk)) if kv_cache is None else np.array(kv_cache[:n_end], dtype=np.float64)
    keys = np.zeros((n_end, xi.shape[1])) if key_cache is None else np.array(key_cache[:n_end], dtype=np.float64)
    if len(new):
        a, b = new.start * m - raw_pos0, new.stop * m - raw_pos0
        entries[new.start:new.stop] = store_rows(compress(x[a:b], g[a:b], bias, m), kv_dtype, kv_nope)
        keys[new.start:new.stop] = store_rows(compress(xi[a:b], gi[a:b], bias_i, m), key_dtype)
    scores = index_scores(q_idx, w, keys, q_pos, m)
    sel = topk(scores, q_pos, m, k)
    out = csa_attend(q, entries, x, raw_pos0, sel, q_pos, W, D_v, scale)
    return out, sel, scores


# ---------------------------------------------------------------------------
# Grouped output projection after the shared-KV MQA
# ---------------------------------------------------------------------------

def group_output_projection(o: np.ndarray, W: np.ndarray) -> np.ndarray:
    """[csdn] section "V4 改进一：CSA 与 HCA", the CSA paragraph's last
    sentence: the attention output is projected in groups to save compute.

    o [T, H, D_v] attention outputs; W [G, (H/G)*D_v, d_g], one matrix per
    group.  Group g holds heads g*H/G .. (g+1)*H/G - 1; its input row is those
    heads' outputs concatenated head by head, and its d_g outputs fill columns
    g*d_g .. (g+1)*d_g - 1 of the result [T, G*d_g]."""
    o = np.asarray(o, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    T, H, D_v = o.shape
    G, K, d_g = W.shape
    assert H % G == 0 and K == (H // G) * D_v, (o.shape, W.shape)
    hg = H // G
    y = np.zeros((T, G * d_g))
    for g in range(G):
        x_g = o[:, g * hg:(g + 1) * hg, :].reshape(T, K)
        y[:, g * d_g:(g + 1) * d_g] = x_g @ W[g]
    return y
