"""Failure detection on the GPU without a fault: every wait inside the
kernels is bounded, and a wait that runs out records a code in a device word
that the host reads (sa_device_error).  The self-test entry point makes one
warp wait, through the kernels' own wait routine and a short cycle limit, on
a barrier phase that nothing completes; the context must stay usable."""

import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

WAIT_TIMED_OUT = 1


def test_bounded_wait_times_out_and_reports():
    assert binding.sa_selftest_wait_timeout(2_000_000) == WAIT_TIMED_OUT   # ~1 ms at 2 GHz
    assert binding.sa_device_error(True) == 0                              # the self-test left the word clear


def test_context_stays_usable_after_a_timeout():
    assert binding.sa_selftest_wait_timeout(100_000) == WAIT_TIMED_OUT
    inp = workloads.tiny()
    d = inp.to("cuda")
    o = binding.sparse_attn(d.q, d.kv, d.attn_sink, d.topk_idxs, d.softmax_scale)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    ref = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    assert (abs(o.float().cpu().double().numpy() - ref) <= 1e-2 + 1e-2 * abs(ref)).all()


def test_selftest_rejects_bad_limits():
    assert binding.sa_selftest_wait_timeout(0) == -1
    assert binding.sa_selftest_wait_timeout(1 << 29) == -1


def test_one_timeout_drains_every_waiting_cta_quickly():
    # CTA 0 gives up after ~1 ms; 511 other CTAs wait with the kernels' full
    # limit (~0.1 s each) and must return as soon as CTA 0 has recorded its
    # timeout, because every bounded wait also watches the error word
    code, ms = binding.sa_selftest_wait_drain(512, 2_000_000)
    assert code == WAIT_TIMED_OUT
    assert ms < 40.0, f"drain took {ms:.1f} ms"
    assert binding.sa_device_error(True) == 0
    # and the context is still usable
    test_context_stays_usable_after_a_timeout()
