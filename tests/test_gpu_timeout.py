"""The failure path of the bounded device-side waits, without a GPU fault.

csa_debug_stall_next arms a one-shot test aid: the next launch of the named
tensor-core kernel makes its first CTA's MMA issuer wait, while that CTA's
first loads are in flight, on a device flag that nothing sets.  That wait
gives up after 0.1 s like any wait that runs out: it records its site, the
launch's other waits give up, every CTA lets its own copies and MMAs in flight
land, and the kernel exits.  The test checks that csa_device_status reports
CSA_ERR_TIMEOUT with the site, and that the next call on the same context
runs normally and gives the same result as before the stall."""

import numpy as np
import pytest
import torch

from long_context_sparse_25_b300 import csa, synth
from long_context_sparse_25_b300.pipeline import Step

pytestmark = pytest.mark.gpu


def _index_case(dev):
    wl = synth.WORKLOADS["csa_decode_1m"].replace(B=2, L=80000)
    inp = synth.make_inputs(wl, dev)
    step = Step(wl, inp)
    step.run()  # fills the tail entry and key of both caches
    torch.cuda.synchronize()
    csa.device_status()
    return wl, inp, step


def _index(wl, inp, step, scores):
    csa.index(step.p, inp["q_idx"], inp["w"], step.keys, wl.q_pos0, wl.N, scores)


def test_indexer_wait_that_runs_out_is_reported_and_the_context_recovers(cuda_device):
    wl, inp, step = _index_case(cuda_device)
    want = torch.empty((wl.B, wl.Q, wl.N), device=cuda_device)
    _index(wl, inp, step, want)
    torch.cuda.synchronize()
    csa.device_status()

    csa.debug_stall_next(csa.STALL_INDEX)
    got = torch.full_like(want, 3.0)
    _index(wl, inp, step, got)  # the launch itself succeeds
    with pytest.raises(csa.CsaError) as e:
        csa.device_status()
    assert e.value.code == -6, str(e.value)  # CSA_ERR_TIMEOUT
    assert "site 7" in str(e.value), str(e.value)

    # the status was read and cleared: the same call now runs normally
    _index(wl, inp, step, got)
    torch.cuda.synchronize()
    csa.device_status()
    assert torch.equal(got, want)
    # and so does the whole step
    first = step.out.clone()
    step.run()
    torch.cuda.synchronize()
    csa.device_status()
    assert torch.equal(step.out, first)


def test_disarmed_aid_changes_nothing(cuda_device):
    wl, inp, step = _index_case(cuda_device)
    csa.debug_stall_next(csa.STALL_INDEX)
    csa.debug_stall_next(0)  # disarm
    out = step.out.clone()
    step.run()
    torch.cuda.synchronize()
    csa.device_status()
    assert torch.equal(step.out, out)


def test_attention_wait_that_runs_out_is_reported_and_the_context_recovers(cuda_device):
    """The same for the tensor-core attention: the stalled launch's first CTA
    has its first gathers in flight; the report names the attention's site."""
    wl = synth.WORKLOADS["csa_decode_1m"].replace(B=2, L=20000)
    inp = synth.make_inputs(wl, cuda_device)
    step = Step(wl, inp)
    step.run()
    torch.cuda.synchronize()
    csa.device_status()
    want = step.out.clone()
    sel = step.selected()
    csa.debug_stall_next(csa.STALL_ATTEND)
    csa.attend(step.p, inp["q"], step.kv, step.raw, wl.raw_pos0, sel, wl.q_pos0, wl.N, step.out)
    with pytest.raises(csa.CsaError) as e:
        csa.device_status()
    assert e.value.code == -6 and "site 28" in str(e.value), str(e.value)
    csa.attend(step.p, inp["q"], step.kv, step.raw, wl.raw_pos0, sel, wl.q_pos0, wl.N, step.out)
    torch.cuda.synchronize()
    csa.device_status()
    assert torch.equal(step.out, want)
