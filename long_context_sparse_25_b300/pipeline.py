"""One forward step of CSA / HCA for a synthetic workload, through the C ABI.

``Step(wl, inputs)`` owns the output, cache and workspace buffers of one
workload and runs the whole path with ``run()``:

* CSA prefill / decode: one ``csa_forward`` call (compress the new entries,
  index, top-k, attend over the selected entries or, for the raw-token
  workloads, over the raw tokens of the selected blocks);
* HCA prefill / decode: ``csa_compress`` of the new entries (m' = 128) then
  ``hca_attend``.

Buffers are allocated once in the constructor; ``run()`` only launches.
"""

from __future__ import annotations

import torch

from . import csa
from .synth import Workload


class Step:
    def __init__(self, wl: Workload, inp: dict, out_dtype=None):
        self.wl = wl
        self.inp = inp
        dev = inp["x"].device
        self.device = dev
        B, N = wl.B, wl.N
        f32 = wl.dtype == "f32"
        self.out_dtype = out_dtype or (torch.float32 if f32 else torch.bfloat16)
        self.out = torch.empty((B, wl.Q, wl.H, wl.D_v), dtype=self.out_dtype, device=dev)
        self.p = csa.params(B, wl.m, wl.H, wl.D_qk, wl.D_v, wl.H_I, wl.d_I, wl.k, wl.W, wl.scale)
        decode = wl.mode.endswith("decode")
        self.n_cached = N - 1 if decode else 0
        # entry cache (and indexer-key cache for CSA)
        if decode:
            if wl.dtype == "mixed":
                self.kv = csa.rows(inp["kv_nope"], inp["kv_rope"], inp["kv_scale"])
            else:
                self.kv = csa.rows(inp["kv"])
        else:
            dt = torch.float32 if f32 else torch.bfloat16
            self.kv_buf = torch.empty((B, N, wl.D_qk), dtype=dt, device=dev)
            self.kv = csa.rows(self.kv_buf)
        self.raw = csa.rows(inp["x"])
        if wl.mode.startswith("csa"):
            if decode:
                if wl.dtype == "mixed":
                    self.keys = csa.rows(inp["keys"], None, inp["keys_scale"])
                else:
                    self.keys = csa.rows(inp["keys"])
            else:
                self.keys_buf = torch.empty((B, N, wl.d_I), dtype=self.kv_buf.dtype, device=dev)
                self.keys = csa.rows(self.keys_buf)
            self.args = csa.forward_args(
                x=inp["x"], gate=inp["g"], bias=inp["bias"], xi=inp["xi"], gate_i=inp["gi"],
                bias_i=inp["bias_i"], raw_pos0=wl.raw_pos0, q=inp["q"], q_idx=inp["q_idx"],
                w=inp["w"], q_pos0=wl.q_pos0, kv=self.kv, keys=self.keys,
                n_cached=self.n_cached, out=self.out, q_idx_scale=inp.get("q_idx_scale"),
                raw_all=inp.get("x_all") if wl.attend == "raw" else None,
                score_dtype=csa.BF16 if wl.scores == "bf16" else csa.F32)
            nbytes = csa.workspace_size(self.p, csa.WS_FORWARD, wl.Q, N)
        else:
            nbytes = csa.workspace_size(self.p, csa.WS_HCA, wl.Q, N)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)

    # views into the forward workspace (CSA only)
    def scores(self) -> torch.Tensor:
        """The indexer scores in the forward workspace (fp32, or bf16 for a
        bf16-score workload; the region is sized for fp32 either way)."""
        wl = self.wl
        n = wl.B * wl.Q * wl.N
        if wl.scores == "bf16":
            return self.ws[: n * 2].view(torch.bfloat16).view(wl.B, wl.Q, wl.N)
        return self.ws[: n * 4].view(torch.float32).view(wl.B, wl.Q, wl.N)

    def selected(self) -> torch.Tensor:
        wl = self.wl
        off = (wl.B * wl.Q * wl.N * 4 + 255) // 256 * 256
        n = wl.B * wl.Q * wl.k
        return self.ws[off: off + n * 4].view(torch.int32).view(wl.B, wl.Q, wl.k)

    def launches_per_step(self) -> int:
        """Kernels one run() launches, following the library's launch plan:
        compress (both caches in one launch unless one is e4m3), the indexer, top-k (three kernels for a few
        long rows, one otherwise), attention (the tensor-core kernel for bf16 /
        mixed caches with 128 heads, plus a combine kernel when a decode query
        is split; the CUDA-core kernel plus a combine when its rows are split)."""
        wl = self.wl
        rows = wl.B * wl.Q
        tc = wl.dtype != "f32" and wl.H == 128
        if wl.mode.startswith("hca"):
            kd = min((wl.q_pos0 + wl.Q) // wl.m, wl.N)
        elif wl.attend == "raw":
            kd = wl.k * wl.m
        else:
            kd = wl.k
        n_keys = ((kd + 3) // 4) * 4 + wl.W
        if tc:  # decode splits a list of more than 5 tiles of 128 keys (mixed caches: 12)
            run = 12 if wl.dtype == "mixed" else 5
            attend = 1 + (1 if (wl.Q == 1 and -(-n_keys // 128) > run) else 0)
        else:
            attend = 1 + (1 if (rows < 1024 and kd + wl.W > 128) else 0)
        if wl.mode.startswith("hca"):
            return 1 + attend
        topk = 3 if (wl.N > 16384 and wl.k <= 4096 and rows < 256) else 1
        return self._compress_launches() + 1 + topk + attend

    def _compress_launches(self) -> int:
        """csa_forward pools the new blocks into both caches with one launch when
        neither cache is e4m3 and both take the same channels-per-thread width
        (16-byte loads, or one channel per thread for a step of few blocks)."""
        wl = self.wl
        n_s = wl.N - self.n_cached
        if n_s <= 0:
            return 0
        if wl.dtype == "mixed":
            return 2
        few = wl.B * n_s * wl.m < 4096
        per = 4 if wl.dtype == "f32" else 8
        vec = [1 if (few or c % per) else per for c in (wl.D_qk, wl.d_I)]
        return 1 if vec[0] == vec[1] else 2

    def run(self, stream=None):
        wl = self.wl
        if wl.mode.startswith("csa"):
            csa.forward(self.p, self.args, self.ws, stream=stream)
        else:
            inp = self.inp
            csa.compress(inp["x"], inp["g"], inp["bias"], wl.m, self.n_cached, wl.N, self.kv,
                         x_pos0=wl.raw_pos0, stream=stream)
            csa.hca(self.p, inp["q"], self.kv, self.raw, wl.raw_pos0, wl.q_pos0, wl.N, self.out,
                    ws=self.ws, stream=stream)
        return self.out
