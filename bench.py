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
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
METRIC = "CSA decode tok/s & prefill query-tok/s at 1M ctx; % of HBM/tensor roofline"
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


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
def _oracle_decode_step(wl, inp, b):
    """The oracle's complete decode step for sequence b (test infrastructure:
    used here only for the timed CPU baseline)."""
    import numpy as np
    import oracle as O

    def f64(t):
        t = t.contiguous()
        if t.dtype == torch.float32:
            return t.double().numpy()
        return O.decode_bf16(t.view(torch.int16).numpy().view(np.uint16))

    N, m = wl.N, wl.m
    x, g = f64(inp["x"][b]), f64(inp["g"][b])
    xi, gi = f64(inp["xi"][b]), f64(inp["gi"][b])
    kv = np.array(f64(inp["kv"][b]))
    keys = np.array(f64(inp["keys"][b]))
    a = (N - 1) * m - wl.raw_pos0
    kv[N - 1] = O.store_rows(O.compress(x[a:a + m], g[a:a + m], f64(inp["bias"]), m), "bf16")
    keys[N - 1] = O.store_rows(O.compress(xi[a:a + m], gi[a:a + m], f64(inp["bias_i"]), m), "bf16")
    pos = np.array([wl.q_pos0])
    scores = O.index_scores(f64(inp["q_idx"][b]), f64(inp["w"][b]), keys, pos, m)
    sel = O.topk(scores, pos, m, wl.k)
    return O.csa_attend(f64(inp["q"][b]), kv, x, wl.raw_pos0, sel, pos, wl.W, wl.D_v, wl.scale)


def _cpu_inputs(wl, nseq):
    from long_context_sparse_25_b300 import synth
    return synth.make_inputs(wl.replace(B=nseq), "cpu")


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = _cpu_inputs(wl, 1)
    for _ in range(args.warmup):
        _oracle_decode_step(wl, inp, 0)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_decode_step(wl, inp, 0)
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
        self.path = ROOT / "gpurun_out" / f"clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.path.parent.mkdir(exist_ok=True)
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
        rows = [r.split(",") for r in self.path.read_text().strip().splitlines() if r.strip()]
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
    qi_b = (wl.H_I * (wl.d_I + 4)) if mixed else wl.H_I * wl.d_I * esz
    decode = wl.mode.endswith("decode")
    new = N - (N - 1 if decode else 0)
    w = {}
    if wl.mode.startswith("csa"):
        # raw rows + gates in, entries out, for the KV and the indexer keys
        w["compress_bytes"] = B * new * (m * 2 * (wl.D_qk + wl.d_I) * esz + entry_b + key_b)
        w["index_bytes"] = B * (N * key_b + wl.Q * (qi_b + wl.H_I * 4))
        w["index_flops"] = float(B * nv.sum() * wl.H_I * wl.d_I * 2)
        keys = np.minimum(wl.k, nv) + win
        w["attend_flops"] = float(B * keys.sum() * wl.H * (wl.D_qk + wl.D_v) * 2)
        w["attend_bytes"] = B * (np.minimum(wl.k, nv).sum() * entry_b + win.sum() * wl.D_qk * esz
                                 + wl.Q * wl.H * (wl.D_qk + wl.D_v) * esz)
    else:  # HCA: every visible entry plus the window
        w["compress_bytes"] = B * new * (m * 2 * wl.D_qk * esz + entry_b)
        keys = nv + win
        w["hca_flops"] = float(B * keys.sum() * wl.H * (wl.D_qk + wl.D_v) * 2)
        w["hca_bytes"] = B * (N * entry_b + win.max() * wl.D_qk * esz
                              + wl.Q * wl.H * (wl.D_qk + wl.D_v) * esz)
    return {k: float(v) for k, v in w.items()}


def measure(args, wl, dev, dist, world, rank, parts_wanted=True, e2e_steps=None,
            with_clocks=True):
    """Time one workload: the whole step as a CUDA graph, each part in a graph
    of its own, and the end-to-end path with host copies."""
    from long_context_sparse_25_b300 import csa, synth
    from long_context_sparse_25_b300.pipeline import Step

    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
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
        "attend": lambda: csa.attend(p, inp["q"], step.kv, step.raw, wl.raw_pos0, sel, wl.q_pos0,
                                     N, step.out, ws=rest, stream=stream),
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
    sets = [(step, g_full, [inp[k] for k in keys_in]), (step2, g_full2, [inp2[k] for k in keys_in])]
    host_in = [inp[k].cpu().pin_memory() for k in keys_in]
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
    res = {"ms": ms, "value": units / (ms / 1e3), "per_part_ms": per_part, "clocks": clk,
           "e2e": {"value": units / (e2e_ms / 1e3), "unit": "tok/s" if decode else "query-tok/s",
                   "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
           "launches_per_step": step.launches_per_step()}
    del step, step2, inp, inp2, g_full, g_full2, g_part, host_in, host_out
    gc.collect()
    torch.cuda.empty_cache()
    return res


def roofline(wl, per_part, peaks, peak_kind):
    """Roofline of the dominant part: HBM for the decode streams (the CSA
    indexer over the key cache, the HCA attention over the entry cache), the
    bf16 tensor peak for the prefill contractions (parts timed alone, so the
    burst peak applies)."""
    w = algorithmic_work(wl)
    if wl.mode == "hca_decode":
        name = "hca"
        achieved = w["hca_bytes"] / (per_part[name] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peak,
                "peak_kind": f"{peak_kind} HBM copy", "unit": "GB/s", "frac": achieved / peak,
                "traffic": _traffic(f"{name}:{wl.name}"), "algorithmic_bytes_per_launch": w["hca_bytes"],
                "tensor_frac": w["hca_flops"] / (per_part[name] / 1e3) / 1e12 / peaks["bf16_tflops"]}
    if wl.mode == "hca_prefill":
        name = "hca"
        achieved = w["hca_flops"] / (per_part[name] / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        return {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak,
                "peak_kind": f"{peak_kind} bf16 burst", "unit": "TFLOP/s", "frac": achieved / peak,
                "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
                "traffic": _traffic(f"{name}:{wl.name}"), "algorithmic_flops_per_launch": w["hca_flops"]}
    if wl.mode == "csa_decode":
        name = "index"
        achieved = w["index_bytes"] / (per_part[name] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peak,
                "peak_kind": f"{peak_kind} HBM copy", "unit": "GB/s", "frac": achieved / peak,
                "traffic": _traffic(f"index_tc_kernel:{wl.name}"),
                "algorithmic_bytes_per_launch": w["index_bytes"]}
    name = max(("index", "attend"), key=lambda k: per_part[k])
    achieved = w[f"{name}_flops"] / (per_part[name] / 1e3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak,
            "peak_kind": f"{peak_kind} bf16 burst", "unit": "TFLOP/s", "frac": achieved / peak,
            "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
            "traffic": _traffic(f"{name}:{wl.name}"),
            "algorithmic_flops_per_launch": w[f"{name}_flops"],
            "other_part": {k: (w[f"{k}_flops"] / (per_part[k] / 1e3) / 1e12) / peak
                           for k in ("index", "attend") if k != name}}


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

    head = measure(args, wl, dev, dist, world, rank)

    def secondary(name, steps):
        sw = synth.WORKLOADS[name]
        sargs = argparse.Namespace(**vars(args))
        sargs.steps = steps
        r = measure(sargs, sw, dev, dist, world, rank, e2e_steps=min(steps, 5), with_clocks=False)
        dec = sw.mode.endswith("decode")
        return {"workload": _config(sw)["workload"], "value": r["value"],
                "unit": "tok/s" if dec else "query-tok/s", "ms_per_step": r["ms"],
                "steps": steps, "per_part_ms": r["per_part_ms"],
                "roofline": roofline(sw, r["per_part_ms"], peaks, peak_kind),
                "e2e": r["e2e"], "gpu_launches": r["launches_per_step"] * steps}

    prefill = None
    others = {}
    if not args.no_prefill and wl.mode == "csa_decode":
        prefill = secondary("csa_prefill_64k", args.steps)
        if not args.no_others:
            # the other rows of the path: HCA prefill and decode, mixed-precision decode
            for name in ("hca_prefill_1m", "hca_decode_1m", "csa_decode_fp8_512k"):
                others[name] = secondary(name, min(args.steps, 10))

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline and wl.mode == "csa_decode":
        nseq = 2
        cinp = _cpu_inputs(wl, nseq)
        t0 = time.perf_counter()
        for b in range(nseq):
            _oracle_decode_step(wl, cinp, b)
        sec = time.perf_counter() - t0
        cpu = {"value": nseq / sec, "unit": "tok/s", "cores": _blas_threads(), "kind": "oracle",
               "sample": f"{nseq} of {wl.B} sequences, complete decode step each "
                         f"(compress tail, index {wl.N} entries, top-{wl.k}, attend)"}
    decode = wl.mode.endswith("decode")
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tok/s" if decode else "query-tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": _config(wl),
        "roofline": roofline(wl, head["per_part_ms"], peaks, peak_kind),
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
