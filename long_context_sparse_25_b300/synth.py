"""Seeded synthetic inputs for the CSA / HCA forward pass.

This module only draws inputs: normal / uniform random numbers from a seeded
torch generator (one generator per tensor, keyed on (seed, tensor id), so a
tensor never depends on the size of another), the RMSNorm that the input
recipe applies to query and KV rows, and the storage formats (bf16, or the
mixed e4m3 + bf16 cache layout built with torch's own float8 cast).  It holds
none of the method's arithmetic: no compression, scoring, selection or
attention.  The same bytes feed the CUDA library and the CPU oracle.

Workloads (sizes from the pages' configurations):

* ``csa_tiny_f32``   -- CSA prefill, fp32, L=4096, m=4, indexer 4x64, k=64,
  window 64, 16 heads x 128, K = V = entry.
* ``csa_prefill_64k``-- CSA prefill, bf16, L=65536, indexer 64x128, k=1024,
  128 heads, KV 512 + 64 rope dims, window 128.
* ``csa_decode_1m``  -- CSA decode, bf16, B=32, context 1,048,576
  (262,144 entries), k=1024, window 128.
* ``hca_prefill_1m`` / ``hca_decode_1m`` -- HCA, m'=128 -> 8192 entries, an
  8192-query tail chunk, and decode at B=32.
* ``csa_decode_fp8_512k`` -- mixed-precision CSA decode, B=64, context
  524,288: nope dims e4m3 + per-entry fp32 scale, rope dims bf16; indexer keys
  and queries e4m3 with per-row scales; 1% of values x20.
* ``csa_decode_raw_1m`` -- the CSA decode step of ``csa_decode_1m`` with the
  raw-token attention: the raw KV rows of all 2^20 positions are resident
  (``x_all``), and each query attends over the 4 raw tokens of each of its
  1024 selected blocks plus the window.
* ``csa_decode_fp4_512k`` -- ``csa_decode_fp8_512k``'s shapes and seed with
  the indexer keys stored in FP4 (E2M1 codes, two per byte, one fp32 scale
  per row: amax / 6), and without the x20 outliers (a per-row FP4 scale would
  flush the rest of such a row to zero; trained FP4 keys have none).
* ``csa_decode_1m_bf16s`` -- ``csa_decode_1m`` (same inputs) with the indexer
  scores stored in bf16 and the top-k over those.
* ``gproj_prefill_64k`` / ``gproj_decode_b32`` (``GPROJ``) -- the grouped
  output projection of the attention output of a 65,536-token prefill and of
  a 32-sequence decode step: 128 heads x 512 in 8 groups of 16 heads, each
  group projected to 1,024 features; o ~ N(0, 1), weights ~ N(0, 1/K).
* ``hybrid_decode_1m`` (``HYBRID``) -- a CSA layer and an HCA layer decoding
  128 consecutive tokens of B=32 sequences at the end of a 2^20 context (the
  last token completes a 128-token block), caches drawn like the decode
  workloads' and raw rows drawn for the positions the sliding buffers hold.
"""

from __future__ import annotations

import dataclasses
import math
import types
from dataclasses import dataclass

import torch

RMS_EPS = 1e-6
E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str          # "csa_prefill" | "csa_decode" | "hca_prefill" | "hca_decode"
    B: int             # sequences
    L: int             # tokens per sequence (the last query sits at L-1)
    m: int             # block size (4 for CSA, 128 for HCA)
    H: int
    D_qk: int
    D_v: int
    H_I: int
    d_I: int
    k: int
    W: int             # raw window
    Q: int             # queries per sequence (tail chunk ending at L-1)
    dtype: str         # "f32" | "bf16" | "mixed"
    seed: int
    rmsnorm: bool = True
    outliers: float = 0.0   # probability that an element is multiplied by 20
    q_std: float = 1.0      # extra factor on Q (the tiny case folds 1/sqrt(128))
    softmax_scale: float | None = None
    attend: str = "entries"  # "entries" | "raw": the raw tokens of the selected blocks
    scores: str = "f32"      # dtype of the indexer scores: "f32" | "bf16"
    keys: str = "auto"       # indexer-key cache: "auto" (as dtype) | "e2m1" (FP4, mixed only)

    @property
    def N(self) -> int:
        """Entries per sequence."""
        return self.L // self.m

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.D_qk)

    @property
    def q_pos0(self) -> int:
        return self.L - self.Q

    @property
    def raw_rows(self) -> int:
        """Raw rows held in memory: all L for prefill; for decode the windows of
        the step's Q queries (W + Q - 1 rows), which also cover the block the
        last token completes."""
        return self.L if self.mode.endswith("prefill") else max(self.W + self.Q - 1, self.m)

    @property
    def raw_pos0(self) -> int:
        return self.L - self.raw_rows

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "csa_tiny_f32": Workload("csa_tiny_f32", "csa_prefill", B=1, L=4096, m=4, H=16, D_qk=128,
                             D_v=128, H_I=4, d_I=64, k=64, W=64, Q=4096, dtype="f32", seed=0,
                             rmsnorm=False, q_std=1.0 / math.sqrt(128), softmax_scale=1.0),
    "csa_prefill_64k": Workload("csa_prefill_64k", "csa_prefill", B=1, L=65536, m=4, H=128,
                                D_qk=576, D_v=512, H_I=64, d_I=128, k=1024, W=128, Q=65536,
                                dtype="bf16", seed=1),
    "csa_decode_1m": Workload("csa_decode_1m", "csa_decode", B=32, L=1 << 20, m=4, H=128,
                              D_qk=576, D_v=512, H_I=64, d_I=128, k=1024, W=128, Q=1,
                              dtype="bf16", seed=2),
    "hca_prefill_1m": Workload("hca_prefill_1m", "hca_prefill", B=1, L=1 << 20, m=128, H=128,
                               D_qk=576, D_v=512, H_I=0, d_I=0, k=0, W=128, Q=8192,
                               dtype="bf16", seed=3),
    "hca_decode_1m": Workload("hca_decode_1m", "hca_decode", B=32, L=1 << 20, m=128, H=128,
                              D_qk=576, D_v=512, H_I=0, d_I=0, k=0, W=128, Q=1,
                              dtype="bf16", seed=3),
    "csa_decode_fp8_512k": Workload("csa_decode_fp8_512k", "csa_decode", B=64, L=1 << 19, m=4,
                                    H=128, D_qk=576, D_v=512, H_I=64, d_I=128, k=1024, W=128,
                                    Q=1, dtype="mixed", seed=4, outliers=0.01),
    "csa_decode_raw_1m": Workload("csa_decode_raw_1m", "csa_decode", B=32, L=1 << 20, m=4, H=128,
                                  D_qk=576, D_v=512, H_I=64, d_I=128, k=1024, W=128, Q=1,
                                  dtype="bf16", seed=2, attend="raw"),
    "csa_decode_fp4_512k": Workload("csa_decode_fp4_512k", "csa_decode", B=64, L=1 << 19, m=4,
                                    H=128, D_qk=576, D_v=512, H_I=64, d_I=128, k=1024, W=128,
                                    Q=1, dtype="mixed", seed=4, outliers=0.0, keys="e2m1"),
    "csa_decode_1m_bf16s": Workload("csa_decode_1m_bf16s", "csa_decode", B=32, L=1 << 20, m=4,
                                    H=128, D_qk=576, D_v=512, H_I=64, d_I=128, k=1024, W=128, Q=1,
                                    dtype="bf16", seed=2, scores="bf16"),
}

# tensor ids (the generator of tensor `name` is seeded with seed * 1000 + id)
_IDS = {"x": 1, "g": 2, "bias": 3, "xi": 4, "gi": 5, "bias_i": 6, "q": 7, "q_idx": 8,
        "w": 9, "kv": 10, "keys": 11, "outl_kv": 12, "outl_keys": 13, "outl_q_idx": 14,
        "outl_x": 15, "outl_q": 16, "x1": 17, "g1": 18, "bias1": 19, "q1": 20, "ent": 21,
        "o": 22, "wproj": 23}


def _gen(wl: Workload, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed * 1000 + _IDS[name])
    return g


def _normal(wl, name, shape, device, std=1.0, rms=False, outl=None, chunk_rows=1 << 16,
            out_dtype=torch.float32):
    """N(0, std^2) tensor, optionally RMSNorm'd per last-dim row and with
    outliers, drawn in float32 in row chunks of a fixed size (so that memory
    stays bounded) and stored in out_dtype (round to nearest even)."""
    gen = _gen(wl, name, device)
    gen_o = _gen(wl, outl, device) if (outl is not None and wl.outliers > 0) else None
    out = torch.empty(shape, dtype=out_dtype, device=device)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        v = torch.randn((r1 - r0, shape[-1]), generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        if rms:
            v.mul_(torch.rsqrt(v.pow(2).mean(dim=-1, keepdim=True) + RMS_EPS))
        if gen_o is not None:
            u = torch.rand((r1 - r0, shape[-1]), generator=gen_o, device=device)
            v = torch.where(u < wl.outliers, v * 20.0, v)
        flat[r0:r1] = v
    return out


def _uniform(wl, name, shape, device):
    return torch.rand(shape, generator=_gen(wl, name, device), device=device, dtype=torch.float32)


def _store(v: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return v
    return v.to(torch.bfloat16)


def quantize_e4m3_rows(v: torch.Tensor, nope: int):
    """(codes e4m3 [.., nope], scale f32 [..], rope bf16 [.., rest] or None):
    per-row scale amax/448 over the nope channels (1 for an all-zero row)."""
    amax = v[..., :nope].abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).float()
    codes = (v[..., :nope] / scale.unsqueeze(-1)).to(torch.float8_e4m3fn)
    rope = v[..., nope:].to(torch.bfloat16).contiguous() if v.shape[-1] > nope else None
    return codes.contiguous(), scale.contiguous(), rope


_E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_e2m1_rows(v: torch.Tensor):
    """(codes [.., d/2] as torch.float4_e2m1fn_x2 -- channel 2i in the low, 2i+1
    in the high four bits of byte i --, scale f32 [..]): per-row scale
    amax / 6 (1 for an all-zero row), codes the nearest E2M1 value of
    value / scale (ties to the even code), saturating at 6."""
    amax = v.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / 6.0, torch.ones_like(amax)).float()
    x = v / scale.unsqueeze(-1)
    ax = x.abs().clamp(max=6.0)
    q = torch.where(ax < 2.0, 0.5, torch.where(ax < 4.0, 1.0, 2.0))
    r = torch.minimum(torch.round(ax / q) * q, torch.tensor(6.0, device=v.device))
    mags = torch.tensor(_E2M1_MAGS, device=v.device)
    code = torch.searchsorted(mags, r.contiguous()).to(torch.uint8)
    code = code | (torch.signbit(x).to(torch.uint8) << 3)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).contiguous()
    return packed.view(torch.float4_e2m1fn_x2), scale.contiguous()


def make_inputs(wl: Workload, device="cpu") -> dict:
    """All inputs of one workload as torch tensors on ``device``.

    Keys: x, g (raw KV rows and gate logits, [B, raw_rows, D_qk]); bias [m, D_qk];
    xi, gi, bias_i (indexer-key rows, gates, bias); q [B, Q, H, D_qk];
    q_idx [B, Q, H_I, d_I] (+ q_idx_scale [B, Q, H_I] for mixed); w [B, Q, H_I];
    for decode also the caches kv [B, N, D_qk] (or kv_nope / kv_rope / kv_scale)
    and keys [B, N, d_I] (or keys + keys_scale), holding entries 0 .. N-2; the
    decode step compresses entry N-1 from the raw rows.
    """
    B, R = wl.B, wl.raw_rows
    rows_dtype = "f32" if wl.dtype == "f32" else "bf16"
    tdt = torch.float32 if rows_dtype == "f32" else torch.bfloat16
    inp = {}
    if wl.attend == "raw" and R < wl.L:
        # the raw-token attention reads raw rows of every position: all L rows
        # are drawn, and the step's own rows are their last R
        inp["x_all"] = _normal(wl, "x", (B, wl.L, wl.D_qk), device, rms=wl.rmsnorm, out_dtype=tdt)
        inp["x"] = inp["x_all"][:, wl.L - R:].contiguous()
    else:
        inp["x"] = _store(_normal(wl, "x", (B, R, wl.D_qk), device, rms=wl.rmsnorm), rows_dtype)
        if wl.attend == "raw":
            inp["x_all"] = inp["x"]
    inp["g"] = _store(_normal(wl, "g", (B, R, wl.D_qk), device), rows_dtype)
    inp["bias"] = _normal(wl, "bias", (wl.m, wl.D_qk), device, std=0.1)
    inp["q"] = _store(_normal(wl, "q", (B, wl.Q, wl.H, wl.D_qk), device, std=wl.q_std,
                              rms=wl.rmsnorm, outl="outl_q"), rows_dtype)
    if wl.mode.startswith("csa"):
        inp["xi"] = _store(_normal(wl, "xi", (B, R, wl.d_I), device, rms=wl.rmsnorm), rows_dtype)
        inp["gi"] = _store(_normal(wl, "gi", (B, R, wl.d_I), device), rows_dtype)
        inp["bias_i"] = _normal(wl, "bias_i", (wl.m, wl.d_I), device, std=0.1)
        qi = _normal(wl, "q_idx", (B, wl.Q, wl.H_I, wl.d_I), device, rms=wl.rmsnorm,
                     outl="outl_q_idx")
        if wl.dtype == "mixed":
            codes, scale, _ = quantize_e4m3_rows(qi, wl.d_I)
            inp["q_idx"], inp["q_idx_scale"] = codes, scale
        else:
            inp["q_idx"] = _store(qi, rows_dtype)
        inp["w"] = _uniform(wl, "w", (B, wl.Q, wl.H_I), device)
    if wl.mode.endswith("decode"):
        N = wl.N
        kv = _normal(wl, "kv", (B, N, wl.D_qk), device, rms=wl.rmsnorm, outl="outl_kv")
        kv[:, N - 1].zero_()  # computed by the decode step
        if wl.dtype == "mixed":
            codes, scale, rope = quantize_e4m3_rows(kv, wl.D_v)
            inp["kv_nope"], inp["kv_scale"], inp["kv_rope"] = codes, scale, rope
        else:
            inp["kv"] = _store(kv, rows_dtype)
        del kv
        if wl.mode.startswith("csa"):
            keys = _normal(wl, "keys", (B, N, wl.d_I), device, rms=wl.rmsnorm, outl="outl_keys")
            keys[:, N - 1].zero_()
            if wl.keys == "e2m1":
                inp["keys"], inp["keys_scale"] = quantize_e2m1_rows(keys)
            elif wl.dtype == "mixed":
                codes, scale, _ = quantize_e4m3_rows(keys, wl.d_I)
                inp["keys"], inp["keys_scale"] = codes, scale
            else:
                inp["keys"] = _store(keys, rows_dtype)
    return inp


def small(wl: Workload, **kw) -> Workload:
    """A reduced copy of a workload (same recipe and dtypes, smaller sizes)."""
    return wl.replace(**kw)


# ---------------------------------------------------------------------------
# Hybrid decoding: a CSA layer and an HCA layer, token by token
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class HybridWorkload:
    name: str
    B: int
    t0: int          # position of the first decoded token
    steps: int       # tokens decoded
    H: int
    D_qk: int
    D_v: int
    H_I: int
    d_I: int
    k: int
    W: int
    seed: int
    m: int = 4       # CSA block
    m1: int = 128    # HCA block
    raw_rows: int = 512
    held: int | None = None  # raw rows before t0 in the buffers (None: what the first step needs)
    history: bool = False    # draw the raw rows of every position; the caches are then
                             # compressed from them (else drawn like the decode workloads')

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D_qk)

    @property
    def need(self) -> int:
        return self.W + self.m1

    @property
    def p0(self) -> int:
        """First position whose raw rows are drawn."""
        if self.history:
            return 0
        return max(0, self.t0 - (self.held or self.need))

    def layer(self, which: str) -> Workload:
        """The single-layer workload whose recipe (and seed) the layer's
        tensors follow."""
        if which == "csa":
            return Workload(self.name + ":csa", "csa_decode", self.B, self.t0 + self.steps, self.m,
                            self.H, self.D_qk, self.D_v, self.H_I, self.d_I, self.k, self.W, 1,
                            "bf16", self.seed)
        return Workload(self.name + ":hca", "hca_decode", self.B, self.t0 + self.steps, self.m1,
                        self.H, self.D_qk, self.D_v, 0, 0, 0, self.W, 1, "bf16", self.seed)

    def replace(self, **kw) -> "HybridWorkload":
        return dataclasses.replace(self, **kw)


HYBRID = {
    "hybrid_decode_1m": HybridWorkload("hybrid_decode_1m", B=32, t0=(1 << 20) - 128, steps=128,
                                       H=128, D_qk=576, D_v=512, H_I=64, d_I=128, k=1024, W=128,
                                       seed=5),
}


def make_hybrid_inputs(hw: HybridWorkload, device="cpu") -> dict:
    """Inputs of a hybrid decode run as torch tensors on ``device`` (bf16 rows,
    fp32 biases and weights).

    Raw rows of positions p0 .. t0+steps-1 ([B, rows, width]): x0, g0, xi0,
    gi0 (CSA layer: KV rows, gates, indexer-key rows, gates) and x1, g1 (HCA
    layer).  Biases bias0 [m, D_qk], bias_i0 [m, d_I], bias1 [m', D_qk].  Per
    decoded token s: q0[s] [B, 1, H, D_qk], q_idx0[s] [B, 1, H_I, d_I],
    w0[s] [B, 1, H_I], q1[s] [B, 1, H, D_qk] (stacked on a leading steps
    axis).  Without ``history``, also the caches before t0: kv [B, t0//m,
    D_qk], keys [B, t0//m, d_I], ent [B, t0//m', D_qk]."""
    lc, lh = hw.layer("csa"), hw.layer("hca")
    B, S = hw.B, hw.steps
    rows = hw.t0 + S - hw.p0
    bf = torch.bfloat16
    inp = {
        "x0": _normal(lc, "x", (B, rows, hw.D_qk), device, rms=True, out_dtype=bf),
        "g0": _normal(lc, "g", (B, rows, hw.D_qk), device, out_dtype=bf),
        "xi0": _normal(lc, "xi", (B, rows, hw.d_I), device, rms=True, out_dtype=bf),
        "gi0": _normal(lc, "gi", (B, rows, hw.d_I), device, out_dtype=bf),
        "x1": _normal(lh, "x1", (B, rows, hw.D_qk), device, rms=True, out_dtype=bf),
        "g1": _normal(lh, "g1", (B, rows, hw.D_qk), device, out_dtype=bf),
        "bias0": _normal(lc, "bias", (hw.m, hw.D_qk), device, std=0.1),
        "bias_i0": _normal(lc, "bias_i", (hw.m, hw.d_I), device, std=0.1),
        "bias1": _normal(lh, "bias1", (hw.m1, hw.D_qk), device, std=0.1),
        "q0": _normal(lc, "q", (S, B, 1, hw.H, hw.D_qk), device, rms=True, out_dtype=bf),
        "q_idx0": _normal(lc, "q_idx", (S, B, 1, hw.H_I, hw.d_I), device, rms=True,
                          out_dtype=bf),
        "w0": _uniform(lc, "w", (S, B, 1, hw.H_I), device),
        "q1": _normal(lh, "q1", (S, B, 1, hw.H, hw.D_qk), device, rms=True, out_dtype=bf),
    }
    if not hw.history:
        n, n1 = hw.t0 // hw.m, hw.t0 // hw.m1
        inp["kv"] = _normal(lc, "kv", (B, n, hw.D_qk), device, rms=True, out_dtype=bf)
        inp["keys"] = _normal(lc, "keys", (B, n, hw.d_I), device, rms=True, out_dtype=bf)
        inp["ent"] = _normal(lh, "ent", (B, n1, hw.D_qk), device, rms=True, out_dtype=bf)
    return inp


# ---------------------------------------------------------------------------
# Grouped output projection
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class GprojWorkload:
    name: str
    T: int      # rows of the attention output (tokens)
    H: int
    D_v: int
    G: int      # groups of H/G heads
    d_g: int    # features per group
    seed: int

    @property
    def K(self) -> int:
        return self.H // self.G * self.D_v

    def replace(self, **kw) -> "GprojWorkload":
        return dataclasses.replace(self, **kw)


GPROJ = {
    "gproj_prefill_64k": GprojWorkload("gproj_prefill_64k", T=65536, H=128, D_v=512, G=8,
                                       d_g=1024, seed=6),
    "gproj_decode_b32": GprojWorkload("gproj_decode_b32", T=32, H=128, D_v=512, G=8, d_g=1024,
                                      seed=6),
}


def make_gproj_inputs(gw: GprojWorkload, device="cpu") -> dict:
    """o [T, H, D_v] bf16 ~ N(0, 1); w [G, d_g, K] bf16 ~ N(0, 1/K) (row n of
    group g = column n of that group's projection matrix)."""
    seed = types.SimpleNamespace(seed=gw.seed, outliers=0.0)
    o = _normal(seed, "o", (gw.T, gw.H, gw.D_v), device, out_dtype=torch.bfloat16)
    w = _normal(seed, "wproj", (gw.G, gw.d_g, gw.K), device, std=1.0 / math.sqrt(gw.K),
                out_dtype=torch.bfloat16)
    return {"o": o, "w": w}
