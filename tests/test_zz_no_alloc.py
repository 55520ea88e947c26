"""csa_topk_noalloc: top-k for callers that cannot allocate device memory at
the point of the call (code inside a host framework that owns every device
allocation, or a path that must not call cudaMalloc because it can
synchronise the device).  Its scratch is a static device array inside the
library.  Through the C ABI, its index lists must equal those of csa_topk
given a caller workspace and the oracle's top-k on the same scores, bit for
bit, on two calls in a row (the second call must not see anything the first
left in the shared array).  Sizes
beyond the array are rejected with CSA_ERR_WORKSPACE.

This file is collected last on purpose, and it passes both alone in a fresh
process and after the other tests."""

import numpy as np
import pytest
import torch

import oracle as O
from long_context_sparse_25_b300 import csa

pytestmark = pytest.mark.gpu


def _scores(rng, B, Q, N, ties):
    s = rng.standard_normal((B, Q, N)).astype(np.float32)
    if ties:
        s = np.where(rng.uniform(size=s.shape) < 0.4, np.round(s, 1), s).astype(np.float32)
        s[..., ::7] = 0.0
    return s


def test_noalloc_topk_equals_workspace_topk_twice(cuda_device):
    rng = np.random.default_rng(2024)
    B, Q, N, k, m = 3, 1, 150001, 1024, 4
    q_pos0 = m * N - 1  # every entry visible
    p = csa.params(B, m, k=k)
    need = csa.workspace_size(p, csa.WS_TOPK, Q, N)
    assert 0 < need <= csa.TOPK_NOALLOC_MAX_BYTES  # this case uses the scratch
    for call, ties in enumerate((False, True)):
        s = torch.from_numpy(_scores(rng, B, Q, N, ties)).to(cuda_device)
        ref = torch.full((B, Q, k), -7, dtype=torch.int32, device=cuda_device)
        got = torch.full((B, Q, k), -7, dtype=torch.int32, device=cuda_device)
        csa.topk(p, s, q_pos0, ref)  # existing entry point, caller workspace
        csa.topk_noalloc(p, s, q_pos0, got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}: index lists differ"
        # and both are the oracle's selection on the same fp32 scores: the k
        # largest, ties to the lower index, ascending
        g = got.cpu().numpy()
        s64 = s.cpu().double().numpy()
        for b in range(B):
            want = O.topk(s64[b], np.array([q_pos0]), m, k)
            assert np.array_equal(g[b], want), f"call {call}, sequence {b}: not the oracle's top-k"


def test_noalloc_topk_rejects_sizes_beyond_the_static_buffer(cuda_device):
    B, Q, N, k, m = 8, 1, 500000, 1024, 4
    p = csa.params(B, m, k=k)
    assert csa.workspace_size(p, csa.WS_TOPK, Q, N) > csa.TOPK_NOALLOC_MAX_BYTES
    s = torch.zeros((B, Q, N), dtype=torch.float32, device=cuda_device)
    idx = torch.empty((B, Q, k), dtype=torch.int32, device=cuda_device)
    with pytest.raises(csa.CsaError) as e:
        csa.topk_noalloc(p, s, m * N - 1, idx)
    assert e.value.code == -4 and "static buffer" in str(e.value)
