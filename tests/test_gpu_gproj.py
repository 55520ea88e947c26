"""Grouped output projection on the GPU (csa_group_proj through the C ABI)
against the oracle's float64 projection.

Tolerance from the arithmetic: the kernel multiplies bf16 values exactly and
accumulates K products in fp32; with rounding errors of random sign that
error is about sqrt(K) * 2^-24 * sum_j |o_j w_j| (K = 8192: ~2^-17 of that
sum), and the test allows 2^-12 of it, far above a correct accumulation and
far below a wrong term; the bf16 output adds half an ulp, 2^-9 |y| (2^-8
allowed).  A dropped K block, a wrong group or a transposed weight moves the
result by O(|y|)."""

import numpy as np
import pytest
import torch

import oracle as O
from harness import f64
from long_context_sparse_25_b300 import csa, synth

pytestmark = pytest.mark.gpu

BASE = synth.GPROJ["gproj_prefill_64k"]


def _check(y_gpu, o, w, rows, f32):
    """Rows `rows` of the GPU output against the oracle on the same rows."""
    o64 = f64(o[rows])
    w64 = f64(w)                              # [G, d_g, K]
    ref = O.group_output_projection(o64, np.transpose(w64, (0, 2, 1)))
    mag = O.group_output_projection(np.abs(o64), np.abs(np.transpose(w64, (0, 2, 1))))
    got = f64(y_gpu[rows])
    bound = 2.0 ** -12 * mag + (0.0 if f32 else 2.0 ** -8 * np.abs(ref))
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{int(bad.sum())} elements off; worst "
                           f"{float(np.max(np.abs(got - ref) - bound)):.3e} above the bound")


@pytest.mark.parametrize("T,G,d_g,f32", [
    (300, 8, 256, False),    # 3 token blocks, the last one partial; 8 groups of 16 heads
    (129, 4, 512, True),     # 4 groups of 32 heads (K = 16384), fp32 output
    (32, 8, 1024, False),    # a decode step of 32 sequences
    (1, 128, 256, False),    # one head per group (K = 512)
])
def test_group_proj_matches_oracle(cuda_device, T, G, d_g, f32):
    gw = BASE.replace(T=T, G=G, d_g=d_g)
    inp = synth.make_gproj_inputs(gw, cuda_device)
    y = torch.full((T, G * d_g), float("nan"), device=cuda_device,
                   dtype=torch.float32 if f32 else torch.bfloat16)
    csa.group_proj(inp["o"], inp["w"], y)
    csa.device_status()
    assert torch.isfinite(y.float()).all(), "an output element was not written"
    _check(y, inp["o"], inp["w"], np.arange(T), f32)


def test_group_proj_full_size_sampled_rows(cuda_device):
    """The bench's prefill size (65,536 tokens, 8 groups x 1,024 features):
    every element written, sampled rows (first, last, and spread over the
    token blocks) against the oracle, and the same bits on a second call."""
    gw = BASE
    inp = synth.make_gproj_inputs(gw, cuda_device)
    y = torch.full((gw.T, gw.G * gw.d_g), float("nan"), device=cuda_device, dtype=torch.bfloat16)
    csa.group_proj(inp["o"], inp["w"], y)
    csa.device_status()
    assert torch.isfinite(y.float()).all()
    rows = np.unique(np.concatenate([np.arange(0, 3), np.arange(gw.T - 3, gw.T),
                                     np.arange(127, gw.T, 4099)]))
    _check(y, inp["o"], inp["w"], rows, False)
    y2 = torch.empty_like(y)
    csa.group_proj(inp["o"], inp["w"], y2)
    csa.device_status()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
