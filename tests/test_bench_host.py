"""Host logic of bench.py (no GPU): the algorithmic work every roofline
fraction divides by, checked against closed forms of the workloads' sizes,
and the kernels a step launches."""

import numpy as np

import bench
from long_context_sparse_25_b300 import csa, synth


def test_decode_index_bytes_are_the_key_cache_and_query_blocks():
    wl = synth.WORKLOADS["csa_decode_1m"]
    w = bench.algorithmic_work(wl)
    # every sequence's 262,144 bf16 keys of 128 dims, its 64 x 128 bf16 query
    # block and its 64 fp32 head weights
    assert w["index_bytes"] == 32 * (262144 * 128 * 2 + 64 * 128 * 2 + 64 * 4)
    # the attention's gathers: 1,024 selected entries + 128 window rows of 576
    # bf16 values, q in and o out (128 heads x (576 + 512) bf16)
    assert w["attend_bytes"] == 32 * ((1024 + 128) * 576 * 2 + 128 * (576 + 512) * 2)
    # the top-k reads the 262,144 fp32 scores and writes 1,024 indices
    assert w["topk_bytes"] == 32 * (262144 * 4 + 1024 * 4)


def test_prefill_flops_follow_the_causal_counts():
    wl = synth.WORKLOADS["csa_prefill_64k"]
    w = bench.algorithmic_work(wl)
    t = np.arange(wl.Q, dtype=np.int64) + wl.q_pos0
    nv = np.minimum((t + 1) // 4, wl.N)
    # Σ_u floor(u / 4) for u = 1..65536, in closed form: 4 Σ_{q<16384} q + 16384
    assert int(nv.sum()) == 4 * (16383 * 16384 // 2) + 16384
    assert abs(w["index_flops"] - 8.796e12) / 8.796e12 < 1e-3
    keys = np.minimum(wl.k, nv) + np.minimum(wl.W, t + 1)
    assert w["attend_flops"] == float(keys.sum() * 128 * (576 + 512) * 2)
    assert abs(w["attend_flops"] - 20.44e12) / 20.44e12 < 1e-3


def test_hca_prefill_flops():
    w = bench.algorithmic_work(synth.WORKLOADS["hca_prefill_1m"])
    assert abs(w["hca_flops"] - 18.91e12) / 18.91e12 < 1e-3


def test_step_launch_count_matches_the_library_plan():
    wl = synth.WORKLOADS["csa_decode_1m"]
    p = csa.params(wl.B, wl.m, wl.H, wl.D_qk, wl.D_v, wl.H_I, wl.d_I, wl.k, wl.W, wl.scale)
    # compress (both caches in one launch), indexer, three top-k kernels for a
    # few long rows, attention and its split combine
    assert csa.topk_launches(p, wl.Q, wl.N) == 3
    assert csa.topk_launches(csa.params(wl.B, wl.m, k=wl.k), wl.Q, 16384) == 1
