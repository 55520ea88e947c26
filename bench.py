#!/usr/bin/env python
"""CSA on one B300: decode tokens/s at 1M-token context (the headline value)
and prefill query-tokens/s at 64K tokens, each with the roofline fraction of
its dominant kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload (``csa_decode_1m``): 32 sequences, one new token each at
position 2^20 - 1, 262,144 compressed entries per sequence (576-wide bf16 KV
entries, 128-wide bf16 indexer keys), 64 indexer heads, top-1024, 128 query
heads sharing the KV, raw window 128.  A step is the whole CSA path for that
token: compress the block the token completes (KV entry and indexer key),
score all entries, keep the top 1024, attend over them plus the window.  The
caches (12 GB) are resident; each step streams 2.2 GB, far more than the
126 MB L2, so no L2 flush is needed between steps.

Second line of the same JSON object (``prefill``): ``csa_prefill_64k``, one
65,536-token sequence, every query causal: compress 16,384 entries and keys,
score the 5.4e8 visible (query, entry) pairs, keep the top 1024 per query,
attend over them plus 128 window tokens.  Its 9.7 GB query tensor and 4.3 GB
score matrix are far larger than L2.

The line's ``roofline`` describes the part of the step that takes the longest
(each part timed alone), lists every part's fraction, and gives the step's own
fraction (all algorithmic bytes or flops of a step over its time).  ``e2e``
runs the same step with its new inputs copied from pinned host memory every
step (decode: the new token's query rows and its raw rows; the earlier raw
rows of the window arrived with earlier steps and stay resident) and the
output read back, the copies overlapped with the neighbouring steps.  Every
line carries ``cpu_baseline``: the oracle timed on a bounded sample of the
same workload on the host cores.

``others`` holds the other rows of the path, each with its own roofline,
e2e and CPU baseline: HCA prefill and decode, the mixed-precision decode,
the raw-token decode, and ``hybrid_decode_1m``: a CSA layer and an HCA layer
decoding 128 consecutive tokens of 32 sequences at the end of a 2^20
context, block compression included at the tokens that complete a block.

With --gpus N > 1 (torchrun, one process per GPU) every rank runs its own
batch (replicas, weak scaling; no collective on the data path) and the time
is the max over ranks.

--impl reference times the CPU oracle (float64 numpy) on the host cores over
a bounded sample of the same workload: each step is the complete decode step
of one sequence.
"""

from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
METRIC = "CSA decode tok/s & prefill query-tok/s at 1M ctx; % of HBM/tensor roofline"
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
NOMINAL_BF16_TFLOPS = 2250.0  # datasheet dense bf16 of one B300 (context for the fractions)


def _peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {k: d.get(k, v) for k, v in FALLBACK.items()}, "measured"
    return dict(FALLBACK), "fallback"


def max_over_ranks(x: float, dist, dev) -> float:
    """The largest x of any rank: a job's time is its slowest rank's."""
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_units(wl, world: int) -> int:
    """Units (tokens) the whole job processes per step: each rank runs its own
    batch of the workload (replicas, no exchange on the data path)."""
    return wl.B * wl.Q * world


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------- CPU oracle
# The timed CPU baseline: the float64 oracle as it stands, on the host cores,
# over a bounded sample of each workload (test infrastructure; this leg and
# --impl reference are the only places bench.py runs it).

def _f64(t):
    """Exact float64 values of a tensor's elements (fp32 / bf16 / e4m3)."""
    import numpy as np
    import oracle as O
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.double().numpy()
    if t.dtype == torch.bfloat16:
        return O.decode_bf16(t.view(torch.int16).numpy().view(np.uint16))
    return O.decode_e4m3(t.view(torch.uint8).numpy())


def _seq_inputs(wl, inp, b):
    """One sequence's inputs of a decode step as float64 arrays (caches
    dequantised exactly)."""
    d = {k: _f64(inp[k][b]) for k in ("x", "g", "q") if k in inp}
    d["bias"] = _f64(inp["bias"])
    if wl.dtype == "mixed":
        import oracle as O
        import numpy as np
        d["kv"] = O.dequantize_rows_e4m3(inp["kv_nope"][b].cpu().view(torch.uint8).numpy(),
                                         inp["kv_scale"][b].cpu().numpy(),
                                         inp["kv_rope"][b].cpu().view(torch.int16).numpy().view(np.uint16))
    else:
        d["kv"] = _f64(inp["kv"][b])
    if wl.mode.startswith("csa"):
        for k in ("xi", "gi", "w"):
            d[k] = _f64(inp[k][b])
        d["bias_i"] = _f64(inp["bias_i"])
        if wl.keys == "e2m1":  # FP4 codes, two per byte
            import numpy as np
            import oracle as O
            u = inp["keys"][b].cpu().view(torch.uint8).numpy()
            codes = np.stack([u & 15, u >> 4], axis=-1).reshape(u.shape[0], -1)
            d["keys"] = O.dequantize_rows_e2m1(codes, inp["keys_scale"][b].cpu().numpy())
            d["q_idx"] = _f64(inp["q_idx"][b]) * inp["q_idx_scale"][b].cpu().double().numpy()[..., None]
        elif wl.dtype == "mixed":
            d["keys"] = _f64(inp["keys"][b]) * inp["keys_scale"][b].cpu().double().numpy()[:, None]
            d["q_idx"] = _f64(inp["q_idx"][b]) * inp["q_idx_scale"][b].cpu().double().numpy()[..., None]
        else:
            d["keys"] = _f64(inp["keys"][b])
            d["q_idx"] = _f64(inp["q_idx"][b])
    return d


def _oracle_decode_step(wl, d):
    """The oracle's complete decode step of one sequence: compress the block
    the token completes into both caches, score every entry, keep the top-k,
    attend (CSA); compress and attend densely (HCA)."""
    import numpy as np
    import oracle as O
    N, m = wl.N, wl.m
    store = "e4m3" if wl.dtype == "mixed" else "bf16"
    kv = np.array(d["kv"])
    a = (N - 1) * m - wl.raw_pos0
    kv[N - 1] = O.store_rows(O.compress(d["x"][a:a + m], d["g"][a:a + m], d["bias"], m), store,
                             wl.D_v)[0]
    pos = np.array([wl.q_pos0])
    if wl.mode.startswith("hca"):
        return O.hca_attend(d["q"], kv, d["x"], wl.raw_pos0, pos, m, wl.W, wl.D_v, wl.scale)
    keys = np.array(d["keys"])
    keys[N - 1] = O.store_rows(O.compress(d["xi"][a:a + m], d["gi"][a:a + m], d["bias_i"], m),
                               "e2m1" if wl.keys == "e2m1" else store)[0]
    scores = O.index_scores(d["q_idx"], d["w"], keys, pos, m)
    sel = O.topk(scores, pos, m, wl.k)
    return O.csa_attend(d["q"], kv, d["x"], wl.raw_pos0, sel, pos, wl.W, wl.D_v, wl.scale)


def cpu_baseline(wl, inp, budget_s=12.0):
    """Time the oracle on a bounded sample of the workload (inputs are the
    same seeded tensors the GPU ran on).  Decode: complete steps of whole
    sequences until the budget is spent.  Prefill: the compression of the
    sequence (HCA: of a sample of blocks, scaled by the block count) plus
    index / top-k / attention of sampled queries, extrapolated to every query
    by the exact per-query work (flops of the index and attention steps)."""
    import numpy as np
    import oracle as O
    cores = _blas_threads()
    unit = "tok/s" if wl.mode.endswith("decode") else "query-tok/s"
    if wl.mode.endswith("decode"):
        sec, nseq = 0.0, 0
        while nseq < wl.B and (nseq == 0 or sec < budget_s):
            d = _seq_inputs(wl, inp, nseq)
            t0 = time.perf_counter()
            _oracle_decode_step(wl, d)
            sec += time.perf_counter() - t0
            nseq += 1
        return {"value": nseq / sec, "unit": unit, "cores": cores, "kind": "oracle",
                "sample": f"{nseq} of {wl.B} sequences, complete decode step each"}
    m, N, Q = wl.m, wl.N, wl.Q
    pos_all = wl.q_pos0 + np.arange(Q)
    nv_all = np.minimum((pos_all + 1) // m, N)
    win_all = np.minimum(wl.W, pos_all + 1)
    csa_ = wl.mode.startswith("csa")
    if csa_:
        work_all = (nv_all * wl.H_I * wl.d_I * 2
                    + (np.minimum(wl.k, nv_all) + win_all) * wl.H * (wl.D_qk + wl.D_v) * 2)
    else:
        work_all = (nv_all + win_all) * wl.H * (wl.D_qk + wl.D_v) * 2
    bias = _f64(inp["bias"])
    if csa_:
        x, g = _f64(inp["x"][0]), _f64(inp["g"][0])
        xi, gi = _f64(inp["xi"][0]), _f64(inp["gi"][0])
        bias_i = _f64(inp["bias_i"])
        t0 = time.perf_counter()
        kv = O.store_rows(O.compress(x, g, bias, m), "bf16")
        keys = O.store_rows(O.compress(xi, gi, bias_i, m), "bf16")
        t_comp = time.perf_counter() - t0
        comp_note = "compression of all entries timed whole"
    else:
        nb = min(64, N)
        blocks = np.linspace(0, N - 1, nb).astype(np.int64)
        rows = torch.from_numpy((blocks[:, None] * m + np.arange(m)[None]).ravel() - wl.raw_pos0)
        xs = _f64(inp["x"][0][rows.to(inp["x"].device)])
        gs = _f64(inp["g"][0][rows.to(inp["g"].device)])
        t0 = time.perf_counter()
        ents = O.store_rows(O.compress(xs, gs, bias, m), "bf16")
        t_comp = (time.perf_counter() - t0) * N / nb
        kv = np.tile(ents, (N // nb + 1, 1))[:N]  # timing only: the sampled blocks' entries, tiled
        comp_note = f"compression of {nb} of {N} blocks, scaled by the block count"
    nq = 6
    qs = np.unique(np.linspace(0, Q - 1, nq).astype(np.int64))
    sec, work = 0.0, 0.0
    for i in qs:
        t = int(pos_all[i])
        qd = _f64(inp["q"][0][int(i):int(i) + 1])
        lo = max(0, t - wl.W + 1) - wl.raw_pos0
        raw = _f64(inp["x"][0][lo:t + 1 - wl.raw_pos0])
        p = np.array([t])
        if csa_:
            qi = _f64(inp["q_idx"][0][int(i):int(i) + 1])
            wv = _f64(inp["w"][0][int(i):int(i) + 1])
            t0 = time.perf_counter()
            sc = O.index_scores(qi, wv, keys, p, m)
            sel = O.topk(sc, p, m, wl.k)
            O.csa_attend(qd, kv, raw, lo + wl.raw_pos0, sel, p, wl.W, wl.D_v, wl.scale)
        else:
            t0 = time.perf_counter()
            O.hca_attend(qd, kv, raw, lo + wl.raw_pos0, p, m, wl.W, wl.D_v, wl.scale)
        sec += time.perf_counter() - t0
        work += float(work_all[i])
    est = t_comp + sec / work * float(work_all.sum())
    return {"value": Q / est, "unit": unit, "cores": cores, "kind": "oracle",
            "sample": f"extrapolated: {comp_note}; index/top-k/attention of {qs.size} of {Q} "
                      f"queries, scaled by the exact per-query flop counts",
            "seconds_timed": t_comp + sec}


def _cpu_inputs(wl, nseq):
    from long_context_sparse_25_b300 import synth
    return synth.make_inputs(wl.replace(B=nseq), "cpu")


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    d = _seq_inputs(wl, _cpu_inputs(wl, 1), 0)
    for _ in range(args.warmup):
        _oracle_decode_step(wl, d)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_decode_step(wl, d)
        times.append(time.perf_counter() - t0)
    sec = sum(times) / len(times)
    value = 1.0 / sec
    cores = _blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": "one sequence's complete decode step per timed step "
                                   "(compress tail, index 262144 entries, top-1024, attend)"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def _config(wl):
    kind = "CSA decode" if wl.mode == "csa_decode" else wl.mode.replace("_", " ")
    cfg = {"workload": f"{wl.name}: {kind}, B={wl.B}, context {wl.L} tokens ({wl.N} entries), "
                       f"Q={wl.Q} per sequence, k={wl.k}, H={wl.H}, D={wl.D_v}+{wl.D_qk - wl.D_v}, "
                       f"indexer {wl.H_I}x{wl.d_I}, window {wl.W}, {wl.dtype}",
           "B": wl.B, "context": wl.L, "entries": wl.N, "queries_per_seq": wl.Q, "k": wl.k}
    w = algorithmic_work(wl)
    streamed = sum(v for k, v in w.items() if k.endswith("_bytes"))
    if wl.mode == "csa_prefill":
        streamed += wl.B * wl.Q * wl.N * 4  # the score matrix, written and read back
    cfg["l2"] = (f"inputs larger than L2 ({streamed / 1e9:.2f} GB streamed per step > 126 MB), "
                 "no flush")
    return cfg


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons (read only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        fd, name = tempfile.mkstemp(prefix="csa_clocks_", suffix=".csv")
        os.close(fd)
        self.path = Path(name)

    def start(self):
        try:
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            except Exception:
                pass
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if uuid:
                cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        text = self.path.read_text()
        self.path.unlink(missing_ok=True)
        rows = [r.split(",") for r in text.strip().splitlines() if r.strip()]
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def _traffic(name: str):
    """DRAM bytes per launch of kernel `name` from the committed ncu summary
    (profiles/traffic.json), or None when the kernel's source changed since
    those counters were taken."""
    import hashlib
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text()).get(name)
    if not d:
        return None
    src = ROOT / d["source"]
    if not src.exists() or hashlib.sha256(src.read_bytes()).hexdigest()[:16] != d["sha"]:
        return None
    return d["bytes_per_launch"]


def algorithmic_work(wl):
    """Algorithmic bytes (HBM-bound parts) and flops (tensor parts) of one step,
    per part, from the method's definition (not from what a kernel does)."""
    import numpy as np
    B, N, m = wl.B, wl.N, wl.m
    t = wl.q_pos0 + np.arange(wl.Q, dtype=np.int64)
    nv = np.minimum((t + 1) // m, N)
    win = np.minimum(wl.W, t + 1)
    esz = 2
    mixed = wl.dtype == "mixed"
    # bytes of one stored entry / indexer key (mixed: e4m3 codes + fp32 scale, bf16 RoPE dims)
    entry_b = (wl.D_v + 4 + (wl.D_qk - wl.D_v) * 2) if mixed else wl.D_qk * esz
    key_b = (wl.d_I + 4) if mixed else wl.d_I * esz
    if wl.keys == "e2m1":  # FP4 codes, two per byte, + fp32 scale
        key_b = wl.d_I // 2 + 4
    qi_b = (wl.H_I * (wl.d_I + 4)) if mixed else wl.H_I * wl.d_I * esz
    decode = wl.mode.endswith("decode")
    new = N - (N - 1 if decode else 0)
    w = {}
    if wl.mode.startswith("csa"):
        # raw rows + gates in, entries out, for the KV and the indexer keys
        w["compress_bytes"] = B * new * (m * 2 * (wl.D_qk + wl.d_I) * esz + entry_b + key_b)
        w["index_bytes"] = B * (N * key_b + wl.Q * (qi_b + wl.H_I * 4))
        w["index_flops"] = float(B * nv.sum() * wl.H_I * wl.d_I * 2)
        # the visible scores read once (fp32 or bf16), the index lists written
        sb = 2 if wl.scores == "bf16" else 4
        w["topk_bytes"] = B * (nv.sum() * sb + wl.Q * wl.k * 4)
        sel = np.minimum(wl.k, nv)
        if wl.attend == "raw":  # the m raw tokens of every selected block
            keys = sel * m + win
            gathered = sel.sum() * m * wl.D_qk * esz
        else:
            keys = sel + win
            gathered = sel.sum() * entry_b
        w["attend_flops"] = float(B * keys.sum() * wl.H * (wl.D_qk + wl.D_v) * 2)
        w["attend_bytes"] = B * (gathered + win.sum() * wl.D_qk * esz
                                 + wl.Q * wl.H * (wl.D_qk + wl.D_v) * esz)
    else:  # HCA: every visible entry plus the window
        w["compress_bytes"] = B * new * (m * 2 * wl.D_qk * esz + entry_b)
        keys = nv + win
        w["hca_flops"] = float(B * keys.sum() * wl.H * (wl.D_qk + wl.D_v) * 2)
        w["hca_bytes"] = B * (N * entry_b + win.max() * wl.D_qk * esz
                              + wl.Q * wl.H * (wl.D_qk + wl.D_v) * esz)
    return {k: float(v) for k, v in w.items()}


def part_bounds(wl):
    """The roofline of each timed part of a step: (bound, algorithmic work),
    bytes for the HBM streams, flops for the tensor-core contractions."""
    w = algorithmic_work(wl)
    decode = wl.mode.endswith("decode")
    b = {"compress": ("hbm", w["compress_bytes"])}
    if wl.mode.startswith("csa"):
        b["index"] = ("hbm", w["index_bytes"]) if decode else ("tensor", w["index_flops"])
        b["topk"] = ("hbm", w["topk_bytes"])
        b["attend"] = ("hbm", w["attend_bytes"]) if decode else ("tensor", w["attend_flops"])
    else:
        b["hca"] = ("hbm", w["hca_bytes"]) if decode else ("tensor", w["hca_flops"])
    return b


def measure(args, wl, dev, dist, world, rank, parts_wanted=True, e2e_steps=None,
            with_clocks=True, want_cpu=False):
    """Time one workload: the whole step as a CUDA graph, each part in a graph
    of its own, and the end-to-end path with host copies."""
    import numpy as np
    from long_context_sparse_25_b300 import csa, synth
    from long_context_sparse_25_b300.pipeline import Step

    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
    # the inputs were drawn on the default stream; the step runs on its own
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    p = step.p
    N = wl.N
    decode = wl.mode.endswith("decode")
    n0 = N - 1 if decode else 0
    if wl.mode.startswith("csa"):
        scores, sel = step.scores(), step.selected()
        off = sel.data_ptr() - step.ws.data_ptr() + sel.numel() * 4
        off = (off + 255) // 256 * 256
        rest = step.ws[off:]

    # the step's C-ABI calls one by one (the kernels csa_forward launches),
    # each timed in a graph of its own
    hca_parts = {
        "compress": lambda: csa.compress(inp["x"], inp["g"], inp["bias"], wl.m, n0, N, step.kv,
                                         x_pos0=wl.raw_pos0, stream=stream),
        "hca": lambda: csa.hca(p, inp["q"], step.kv, step.raw, wl.raw_pos0, wl.q_pos0, N, step.out,
                               ws=step.ws, stream=stream),
    }
    parts = hca_parts if wl.mode.startswith("hca") else {
        "compress": lambda: (csa.compress(inp["x"], inp["g"], inp["bias"], wl.m, n0, N, step.kv,
                                          x_pos0=wl.raw_pos0, stream=stream),
                             csa.compress(inp["xi"], inp["gi"], inp["bias_i"], wl.m, n0, N,
                                          step.keys, x_pos0=wl.raw_pos0, stream=stream)),
        "index": lambda: csa.index(p, inp["q_idx"], inp["w"], step.keys, wl.q_pos0, N, scores,
                                   q_scale=inp.get("q_idx_scale"), stream=stream),
        "topk": lambda: csa.topk(p, scores, wl.q_pos0, sel, ws=rest, stream=stream),
        "attend": (lambda: csa.attend_raw(p, inp["q"], csa.rows(inp["x_all"]), 0, sel, wl.q_pos0,
                                          N, step.out, ws=rest, stream=stream))
        if wl.attend == "raw" else
        (lambda: csa.attend(p, inp["q"], step.kv, step.raw, wl.raw_pos0, sel, wl.q_pos0, N,
                            step.out, ws=rest, stream=stream)),
    }
    if not parts_wanted:
        parts = {}
    with torch.cuda.stream(stream):
        for _ in range(2):
            step.run(stream=stream)
            for f in parts.values():
                f()
    torch.cuda.synchronize()
    csa.device_status(stream)
    g_full = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full, stream=stream):
        step.run(stream=stream)
    g_part = {}
    for name, f in parts.items():
        g_part[name] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_part[name], stream=stream):
            f()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_full.replay()
    torch.cuda.synchronize()

    def timed(graph, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        with torch.cuda.stream(stream):
            for a_, b_ in evs:
                a_.record(stream)
                graph.replay()
                b_.record(stream)
        torch.cuda.synchronize()
        return sum(a_.elapsed_time(b_) for a_, b_ in evs)

    clocks = Clocks() if (rank == 0 and with_clocks) else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    total_ms = timed(g_full, args.steps)
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(total_ms, dist, dev) / args.steps
    csa.device_status(stream)

    per_part = {name: timed(g_, args.steps) / args.steps for name, g_ in g_part.items()}

    # end to end: every step copies its new inputs from pinned host memory and
    # its output back.  Two sets of per-step buffers (the caches are shared)
    # with a graph each let step i+1's input copies and step i-1's output copy
    # run while step i computes: host->device on one stream, device->host on
    # another, the step on the compute stream, ordered by events.
    keys_in = [k for k in ("q", "q_idx", "w", "x", "g", "xi", "gi", "q_idx_scale") if k in inp]
    inp2 = dict(inp)
    for k in keys_in:
        inp2[k] = inp[k].clone()
    step2 = Step(wl, inp2)
    g_full2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_full2, stream=stream):
        step2.run(stream=stream)

    def new_inputs(d):
        # What a step brings in: a decode step's new token (its query rows and
        # its raw KV / indexer-key rows with their gates; the earlier raw rows
        # of the window arrived with earlier steps and stay resident, as do the
        # raw rows of every position that the raw-token attention reads); every
        # input of a prefill step.
        out = []
        for k in keys_in:
            t = d[k]
            if decode and k in ("x", "g", "xi", "gi"):
                t = t[:, -1:]
            out.append(t)
        return out

    sets = [(step, g_full, new_inputs(inp)), (step2, g_full2, new_inputs(inp2))]
    host_in = [t.cpu().pin_memory() for t in new_inputs(inp)]
    host_out = [torch.empty(st_.out.shape, dtype=st_.out.dtype, pin_memory=True) for st_, _, _ in sets]
    bi = sum(t_.numel() * t_.element_size() for t_ in host_in)
    bo = host_out[0].numel() * host_out[0].element_size()
    ne = e2e_steps or args.steps
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    in_done, step_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_steps_run(n, first):
        for it in range(n):
            k = it % 2
            st_, g_, dev_in = sets[k]
            if it >= 2 or not first:
                h2d_s.wait_event(step_done[k])  # the step that last read set k is done
            with torch.cuda.stream(h2d_s):
                for d_, h_ in zip(dev_in, host_in):
                    d_.copy_(h_, non_blocking=True)
                in_done[k].record(h2d_s)
            stream.wait_event(in_done[k])
            if it >= 2 or not first:
                stream.wait_event(out_done[k])  # set k's output has been read back
            with torch.cuda.stream(stream):
                g_.replay()
                step_done[k].record(stream)
            d2h_s.wait_event(step_done[k])
            with torch.cuda.stream(d2h_s):
                host_out[k].copy_(st_.out, non_blocking=True)
                out_done[k].record(d2h_s)

    e2e_steps_run(2, True)  # warm-up
    torch.cuda.synchronize()
    e0.record(h2d_s)
    e2e_steps_run(ne, False)
    stream.wait_stream(d2h_s)
    stream.wait_stream(h2d_s)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / ne, dist, dev)
    units = job_units(wl, world)
    recall = None
    if wl.keys == "e2m1":
        # how much of the selection with the same keys in e4m3 the FP4 keys keep
        # (the same draws; the keys quantised to e4m3 instead of FP4)
        wl8 = wl.replace(keys="auto")
        inp8 = synth.make_inputs(wl8, dev)
        ref_step = Step(wl8, inp8)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            step.run(stream=stream)
            ref_step.run(stream=stream)
        torch.cuda.synchronize()
        csa.device_status(stream)
        a4, a8 = step.selected().cpu().numpy(), ref_step.selected().cpu().numpy()
        hits = sum(np.intersect1d(a4[b, i], a8[b, i][a8[b, i] >= 0]).size
                   for b in range(wl.B) for i in range(wl.Q))
        recall = {"value": hits / int((a8 >= 0).sum()),
                  "of": "the top-k sets with the same keys stored in e4m3", "sets": wl.B * wl.Q}
        del ref_step, inp8
    if wl.scores == "bf16":
        # how much of the fp32-score selection the bf16-score selection keeps
        # (the same inputs, the step run once with each score dtype)
        ref_step = Step(wl.replace(scores="f32"), inp)
        with torch.cuda.stream(stream):
            step.run(stream=stream)
            ref_step.run(stream=stream)
        torch.cuda.synchronize()
        csa.device_status(stream)
        a16, a32 = step.selected().cpu().numpy(), ref_step.selected().cpu().numpy()
        hits = sum(np.intersect1d(a16[b, i], a32[b, i][a32[b, i] >= 0]).size
                   for b in range(wl.B) for i in range(wl.Q))
        total = int((a32 >= 0).sum())
        recall = {"value": hits / total, "of": "the fp32-score top-k sets, same inputs",
                  "sets": wl.B * wl.Q}
        del ref_step
    cpu = None
    if want_cpu:
        torch.cuda.synchronize()
        cpu = cpu_baseline(wl, inp)
    res = {"ms": ms, "value": units / (ms / 1e3), "per_part_ms": per_part, "clocks": clk,
           "cpu_baseline": cpu,
           "e2e": {"value": units / (e2e_ms / 1e3), "unit": "tok/s" if decode else "query-tok/s",
                   "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
           "launches_per_step": step.launches_per_step(), "recall": recall}
    del step, step2, inp, inp2, g_full, g_full2, g_part, host_in, host_out
    gc.collect()
    torch.cuda.empty_cache()
    return res


def roofline(wl, per_part, ms_step, peaks, peak_kind):
    """Roofline of the part that takes the longest (each part timed alone in a
    graph of its own, so the burst peaks apply), every part's fraction, and
    the step's: all algorithmic bytes (decode) or flops (prefill) of the step
    over the time of the whole step."""
    bounds = part_bounds(wl)

    def frac_of(bound, amount, ms):
        if bound == "hbm":
            ach = amount / (ms / 1e3) / 1e9
            return ach, peaks["hbm_gbs"], "GB/s"
        ach = amount / (ms / 1e3) / 1e12
        return ach, peaks["bf16_tflops"], "TFLOP/s"

    name = max(per_part, key=lambda k: per_part[k])
    bound, amount = bounds[name]
    ach, peak, unit = frac_of(bound, amount, per_part[name])
    r = {"bound": bound, "kernel": name, "achieved": ach, "peak": peak, "unit": unit,
         "frac": ach / peak, "traffic": _traffic(f"{name}:{wl.name}"),
         "peak_kind": f"{peak_kind} " + ("HBM copy" if bound == "hbm" else "bf16 burst"),
         ("algorithmic_bytes_per_launch" if bound == "hbm" else "algorithmic_flops_per_launch"): amount}
    if bound == "tensor":
        r["frac_sustained"] = ach / peaks["bf16_tflops_sustained"]
        r["frac_nominal"] = ach / NOMINAL_BF16_TFLOPS
    r["parts"] = {}
    for k, t in per_part.items():
        b_, a_ = bounds[k]
        x, p_, u_ = frac_of(b_, a_, t)
        r["parts"][k] = {"bound": b_, "ms": t, "achieved": x, "unit": u_, "frac": x / p_}
    if wl.mode.endswith("decode"):
        tot_b = sum(a_ for b_, a_ in bounds.values())
        ach = tot_b / (ms_step / 1e3) / 1e9
        r["step"] = {"bound": "hbm", "algorithmic_bytes": tot_b, "achieved": ach, "unit": "GB/s",
                     "peak": peaks["hbm_gbs"], "frac": ach / peaks["hbm_gbs"]}
    else:
        tot_f = sum(a_ for b_, a_ in bounds.values() if b_ == "tensor")
        ach = tot_f / (ms_step / 1e3) / 1e12
        r["step"] = {"bound": "tensor", "algorithmic_flops": tot_f, "achieved": ach,
                     "unit": "TFLOP/s", "peak": peaks["bf16_tflops"],
                     "frac": ach / peaks["bf16_tflops"],
                     "frac_sustained": ach / peaks["bf16_tflops_sustained"]}
    return r


def _hybrid_token(hw, t):
    """The single-layer workloads of one hybrid token at position t: the CSA
    layer's decode step and the HCA layer's, each over the entries visible
    at t (the compress part counts only when t completes a block)."""
    lc = hw.layer("csa").replace(L=t + 1)
    lh = hw.layer("hca").replace(L=t + 1)
    return lc, lh


def hybrid_work(hw):
    """Algorithmic bytes and launches of the hybrid run's hw.steps tokens, from
    the single-layer definitions: per token, the CSA layer's index, top-k and
    attention and the HCA layer's attention; the compression of a block only
    at the token that completes it."""
    tot, launches = 0.0, 0
    for t in range(hw.t0, hw.t0 + hw.steps):
        lc, lh = _hybrid_token(hw, t)
        wc, wh = algorithmic_work(lc), algorithmic_work(lh)
        tot += wc["index_bytes"] + wc["topk_bytes"] + wc["attend_bytes"] + wh["hca_bytes"]
        n_keys = (hw.k + 3) // 4 * 4 + hw.W
        # launch plan (as in the single-layer steps): indexer; top-k (three
        # kernels for few long rows); tensor-core attention plus a combine
        # when a decode query's keys exceed 5 tiles of 128
        launches += 1 + (3 if (lc.N > 16384 and hw.k <= 4096 and hw.B < 256) else 1)
        launches += 1 + (1 if -(-n_keys // 128) > 5 else 0)
        nh = lh.N + hw.W
        launches += 1 + (1 if -(-nh // 128) > 5 else 0)
        if (t + 1) % hw.m == 0:
            tot += wc["compress_bytes"]
            launches += 1  # both caches in one launch
        if (t + 1) % hw.m1 == 0:
            tot += wh["compress_bytes"]
            launches += 1
    return tot, launches


def measure_hybrid(args, hw, dev, peaks, peak_kind, reps):
    """Hybrid decoding: a CSA layer and an HCA layer decode hw.steps
    consecutive tokens of B sequences.  The run of hw.steps tokens is one CUDA
    graph, replayed `reps` times (the decoder rewinds to t0 between replays;
    every replay recomputes the same cache entries from the same rows); e2e
    runs the decoder's own per-token calls eagerly with each token's rows and
    queries copied from pinned host memory and both outputs read back."""
    from long_context_sparse_25_b300 import csa, hybrid, synth

    inp = synth.make_hybrid_inputs(hw, dev)
    pc = csa.params(hw.B, hw.m, hw.H, hw.D_qk, hw.D_v, hw.H_I, hw.d_I, hw.k, hw.W, hw.scale)
    ph = csa.params(hw.B, hw.m1, hw.H, hw.D_qk, hw.D_v, 0, 0, 0, hw.W, hw.scale)
    t0, S = hw.t0, hw.steps
    dec = hybrid.HybridDecoder(pc, ph, t0=t0, max_len=t0 + S, device=dev, bias0=inp["bias0"],
                               bias_i0=inp["bias_i0"], bias1=inp["bias1"],
                               raw_rows=hw.raw_rows, held=hw.held)
    n, n1 = t0 // hw.m, t0 // hw.m1
    dec.kv[:, :n].copy_(inp.pop("kv"))
    dec.keys[:, :n].copy_(inp.pop("keys"))
    dec.ent[:, :n1].copy_(inp.pop("ent"))
    held = t0 - dec.p0
    assert dec.p0 == hw.p0 and held + S <= hw.raw_rows, "the run must fit the raw buffers"
    for name in hybrid.RAW_NAMES:
        # the rows already held, and every decoded token's rows written ahead
        dec.raw[name][:, :held + S].copy_(inp[name])
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)

    def run_all():
        dec.rewind(t0)
        for s in range(S):
            dec.step(inp["q0"][s], inp["q_idx0"][s], inp["w0"][s], inp["q1"][s], stream=stream)

    with torch.cuda.stream(stream):
        run_all()
    torch.cuda.synchronize()
    csa.device_status(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run_all()
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // 2)):
            g.replay()
    torch.cuda.synchronize()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a_.record(stream)
        for _ in range(reps):
            g.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    csa.device_status(stream)
    ms_tok = a_.elapsed_time(b_) / (reps * S)
    tot_bytes, launches = hybrid_work(hw)
    ach = tot_bytes / S / (ms_tok / 1e3) / 1e9

    # end to end through the decoder's calls: per token, its six raw rows and
    # four query tensors from pinned host memory, both outputs back
    names_q = ("q0", "q_idx0", "w0", "q1")
    host_rows = {k: inp[k][:, held:held + S].transpose(0, 1).unsqueeze(2).cpu().contiguous()
                 .pin_memory() for k in hybrid.RAW_NAMES}  # [S, B, 1, w]
    host_q = {k: inp[k].cpu().pin_memory() for k in names_q}
    dq = {k: torch.empty_like(inp[k][0]) for k in names_q}
    out_h = [torch.empty(dec.out0.shape, dtype=dec.out0.dtype, pin_memory=True),
             torch.empty(dec.out1.shape, dtype=dec.out1.dtype, pin_memory=True)]
    bi = sum(v[0].numel() * v.element_size() for v in host_rows.values()) + \
        sum(v[0].numel() * v.element_size() for v in host_q.values())
    bo = sum(o.numel() * o.element_size() for o in out_h)

    def e2e_run():
        dec.rewind(t0)
        for s in range(S):
            with torch.cuda.stream(stream):
                for k in hybrid.RAW_NAMES:
                    dec.slot(k).copy_(host_rows[k][s], non_blocking=True)
                for k in names_q:
                    dq[k].copy_(host_q[k][s], non_blocking=True)
                o0, o1 = dec.step(dq["q0"], dq["q_idx0"], dq["w0"], dq["q1"], stream=stream)
                out_h[0].copy_(o0, non_blocking=True)
                out_h[1].copy_(o1, non_blocking=True)

    e2e_run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run()
    e1.record(stream)
    torch.cuda.synchronize()
    csa.device_status(stream)
    e2e_ms = e0.elapsed_time(e1) / S
    # leave the decoder's state as the graph left it (the raw rows of the
    # decoded tokens were rewritten with the same values)
    row = {
        "workload": (f"{hw.name}: a CSA layer (k={hw.k}, indexer {hw.H_I}x{hw.d_I}) and an HCA "
                     f"layer (m'={hw.m1}), H={hw.H}, D={hw.D_v}+{hw.D_qk - hw.D_v}, window "
                     f"{hw.W}, B={hw.B}, {S} consecutive tokens at positions {t0}..{t0 + S - 1} "
                     f"(context 2^20, one 128-token block completed), bf16"),
        "value": hw.B / (ms_tok / 1e3), "unit": "tok/s", "ms_per_token": ms_tok,
        "steps": reps * S,
        "timing": f"one CUDA graph of the {S} tokens, replayed {reps} times; CUDA events",
        "roofline": {"bound": "hbm", "algorithmic_bytes_per_token": tot_bytes / S,
                     "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "peak_kind": f"{peak_kind} HBM copy"},
        "e2e": {"value": hw.B / (e2e_ms / 1e3), "unit": "tok/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo,
                "note": "eager per-token calls (host launch cost included), copies on the "
                        "compute stream"},
        "gpu_launches": launches * reps,
    }
    del dec, inp, g, host_rows, host_q
    gc.collect()
    torch.cuda.empty_cache()
    return row


def measure_gproj(args, gw, dev, peaks, peak_kind, steps):
    """The grouped output projection (csa_group_proj) of one attention output:
    a CUDA graph of one call, CUDA events; e2e copies o from pinned host
    memory and reads y back every step."""
    from long_context_sparse_25_b300 import csa, synth

    inp = synth.make_gproj_inputs(gw, dev)
    y = torch.empty((gw.T, gw.G * gw.d_g), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    f = lambda: csa.group_proj(inp["o"], inp["w"], y, stream=stream)
    with torch.cuda.stream(stream):
        f()
    torch.cuda.synchronize()
    csa.device_status(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        f()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a_.record(stream)
        for _ in range(steps):
            g.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    csa.device_status(stream)
    ms = a_.elapsed_time(b_) / steps
    flops = 2.0 * gw.T * gw.G * gw.K * gw.d_g
    nbytes = (gw.T * gw.H * gw.D_v + gw.G * gw.d_g * gw.K + gw.T * gw.G * gw.d_g) * 2.0
    decode = gw.T < 1024
    if decode:  # the weights stream from HBM
        ach = nbytes / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": nbytes,
                "peak_kind": f"{peak_kind} HBM copy"}
    else:
        ach = flops / (ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                "frac_sustained": ach / peaks["bf16_tflops_sustained"],
                "frac_nominal": ach / NOMINAL_BF16_TFLOPS, "algorithmic_flops_per_launch": flops,
                "peak_kind": f"{peak_kind} bf16 burst"}
    # end to end: o in from pinned host memory, y back
    host_o = inp["o"].cpu().pin_memory()
    host_y = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    ne = 2 if not decode else steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(ne):
            inp["o"].copy_(host_o, non_blocking=True)
            g.replay()
            host_y.copy_(y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / ne
    unit = "tok/s" if decode else "query-tok/s"
    row = {"workload": (f"{gw.name}: grouped output projection of a [{gw.T}, {gw.H}, {gw.D_v}] "
                        f"attention output, {gw.G} groups of {gw.H // gw.G} heads -> {gw.d_g} "
                        f"features each (K = {gw.K}), bf16"),
           "value": gw.T / (ms / 1e3), "unit": unit, "ms_per_step": ms, "steps": steps,
           "roofline": roof,
           "e2e": {"value": gw.T / (e2e_ms / 1e3), "unit": unit,
                   "h2d_bytes_per_step": host_o.numel() * 2, "d2h_bytes_per_step": host_y.numel() * 2},
           "gpu_launches": steps}
    del inp, y, g, host_o, host_y
    gc.collect()
    torch.cuda.empty_cache()
    return row


def run_ours(args, wl):
    from long_context_sparse_25_b300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_kind = _peaks()

    # the oracle's timed baseline: rank 0 of a one-GPU run only
    want_cpu = world == 1 and rank == 0 and not args.no_cpu_baseline
    head = measure(args, wl, dev, dist, world, rank, want_cpu=want_cpu)

    def secondary(name, steps):
        sw = synth.WORKLOADS[name]
        sargs = argparse.Namespace(**vars(args))
        sargs.steps = steps
        r = measure(sargs, sw, dev, dist, world, rank, e2e_steps=min(steps, 5), with_clocks=False,
                    want_cpu=want_cpu)
        dec = sw.mode.endswith("decode")
        return {"workload": _config(sw)["workload"], "value": r["value"],
                "unit": "tok/s" if dec else "query-tok/s", "ms_per_step": r["ms"],
                "steps": steps, "per_part_ms": r["per_part_ms"],
                "roofline": roofline(sw, r["per_part_ms"], r["ms"], peaks, peak_kind),
                "e2e": r["e2e"], "gpu_launches": r["launches_per_step"] * steps,
                "cpu_baseline": r["cpu_baseline"],
                **({"recall": r["recall"]} if r.get("recall") else {})}

    prefill = None
    others = {}
    if not args.no_prefill and wl.mode == "csa_decode":
        prefill = secondary("csa_prefill_64k", args.steps)
        if not args.no_others:
            # the other rows of the path: HCA prefill and decode, mixed-precision decode
            for name in ("hca_prefill_1m", "hca_decode_1m", "csa_decode_fp8_512k",
                         "csa_decode_raw_1m", "csa_decode_1m_bf16s", "csa_decode_fp4_512k"):
                others[name] = secondary(name, min(args.steps, 10))
            # a CSA layer and an HCA layer decoding token by token
            others["hybrid_decode_1m"] = measure_hybrid(args, synth.HYBRID["hybrid_decode_1m"],
                                                        dev, peaks, peak_kind, reps=3)
            # the grouped output projection after the attention
            for name in ("gproj_prefill_64k", "gproj_decode_b32"):
                others[name] = measure_gproj(args, synth.GPROJ[name], dev, peaks, peak_kind,
                                             steps=min(args.steps, 10))

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    cpu = head["cpu_baseline"]
    decode = wl.mode.endswith("decode")
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tok/s" if decode else "query-tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": _config(wl),
        "roofline": roofline(wl, head["per_part_ms"], head["ms"], peaks, peak_kind),
        "per_part_ms": head["per_part_ms"],
        "timing": "CUDA graph of the whole step replayed per timed step; CUDA events on the "
                  "launching stream; each part timed alone in a graph of its own for the roofline",
        "e2e": head["e2e"],
        "gpu_launches": head["launches_per_step"] * args.steps,
        "clocks": head["clocks"],
        "cpu_baseline": cpu,
        "prefill": prefill,
        "others": others or None,
    }
    if head.get("recall"):
        line["recall"] = head["recall"]
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="csa_decode_1m")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the secondary measurements (64K prefill and the others)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the HCA and mixed-precision measurements")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller cases for profiler captures)")
    ap.add_argument("--context", type=int, default=None,
                    help="override the workload's context length (a prefill keeps every query)")
    args = ap.parse_args()
    from long_context_sparse_25_b300 import synth
    if args.workload in synth.GPROJ and args.impl == "ours":
        torch.cuda.set_device(0)
        peaks, peak_kind = _peaks()
        gw = synth.GPROJ[args.workload]
        if args.context:
            gw = gw.replace(T=args.context)
        row = measure_gproj(args, gw, torch.device("cuda", 0), peaks, peak_kind, steps=args.steps)
        print(json.dumps(row), flush=True)
        return
    if args.workload in synth.HYBRID and args.impl == "ours":
        # the hybrid decode row alone
        torch.cuda.set_device(0)
        peaks, peak_kind = _peaks()
        row = measure_hybrid(args, synth.HYBRID[args.workload], torch.device("cuda", 0), peaks,
                             peak_kind, reps=max(1, args.steps // 5))
        print(json.dumps(row), flush=True)
        return
    wl = synth.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.replace(B=args.batch)
    if args.context:
        wl = wl.replace(L=args.context, Q=args.context if wl.mode == "csa_prefill" else wl.Q)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
