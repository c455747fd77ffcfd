"""The allocation-free entry point, sa_sparse_attn_fwd_static_ws.

It serves callers that cannot hand the library device memory (a C host
program without a device allocator, or a serving loop that forbids cudaMalloc
on its hot path): the split-KV workspace is an array inside the library.  It
must give what the regular entry point gives with a caller-supplied
workspace, on consecutive calls that reuse the same array, and match the
oracle to the attention parity bar.  This file is
collected last so that a run stopping at the first failure has already run
every other test."""

import numpy as np
import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


def _regular(d, ns):
    B, S, H, D = d.q.shape
    K = d.topk_idxs.shape[-1]
    out = torch.empty_like(d.q)
    ws = binding.workspace_for(B, S, H, D, K, ns)
    assert ws is not None, "the case must take the split-KV path"
    binding.sparse_attn(d.q, d.kv, d.attn_sink, d.topk_idxs, d.softmax_scale, out=out, workspace=ws, num_splits=ns)
    return out


def _static(d, ns):
    B, S, H, D = d.q.shape
    T, K = d.kv.shape[1], d.topk_idxs.shape[-1]
    out = torch.full_like(d.q, float("nan"))
    rc = binding.sa_sparse_attn_fwd_static_ws(d.q.data_ptr(), d.kv.data_ptr(), d.attn_sink.data_ptr(),
                                              d.topk_idxs.data_ptr(), d.softmax_scale, out.data_ptr(), B, S, H, D,
                                              T, K, ns, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.sa_status_string(rc)
    return out


def _close(a, b):
    a64, b64 = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert np.all(np.abs(a64 - b64) <= ATOL + RTOL * np.abs(b64))


def test_static_workspace_matches_regular_entry_on_consecutive_calls():
    first = workloads.v4_ratio4_decode(B=8).to("cuda")          # 8 tokens: the planner splits
    second = workloads.random_attn(3, 2, 128, 512, 3000, 1152, p_invalid=0.2, seed=77).to("cuda")
    for d, ns in ((first, 0), (second, 5)):
        ref = _regular(d, ns)
        got = _static(d, ns)
        torch.cuda.synchronize()
        assert binding.sa_device_error(True) == 0
        _close(got, ref)
    # the array now holds the second call's partials; the first case again
    ref = _regular(first, 0)
    got = _static(first, 0)
    torch.cuda.synchronize()
    _close(got, ref)


@pytest.mark.parametrize("ns", [0, 5])
def test_static_workspace_matches_the_oracle(ns):
    # the same bar as every attention parity test, straight against the
    # oracle: splits combined in the cluster (planner's choice) and by the
    # separate combine kernel (5 splits)
    c = workloads.random_attn(3, 2, 128, 512, 3000, 1152, p_invalid=0.2, seed=78 + ns)
    got = _static(c.to("cuda"), ns)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    want = oracle.sparse_attn(c.q, c.kv, c.attn_sink, c.topk_idxs, c.softmax_scale)
    g = got.double().cpu().numpy()
    assert np.all(np.abs(g - want) <= ATOL + RTOL * np.abs(want))


def test_static_workspace_rejects_plans_larger_than_the_array():
    d = workloads.random_attn(16, 8, 128, 512, 4096, 4096, p_invalid=0.0, seed=3).to("cuda")
    B, S, H, D = d.q.shape
    need = binding.sa_sparse_attn_workspace_size(B, S, H, D, 4096, 64)
    assert need > (32 << 20)
    rc = binding.sa_sparse_attn_fwd_static_ws(d.q.data_ptr(), d.kv.data_ptr(), d.attn_sink.data_ptr(),
                                              d.topk_idxs.data_ptr(), d.softmax_scale, d.q.data_ptr(), B, S, H, D,
                                              4096, 4096, 64, torch.cuda.current_stream().cuda_stream)
    assert binding.sa_status_string(rc) == "SA_ERR_WORKSPACE"


def test_static_workspace_reports_invalid_arguments_before_the_size_check():
    # num_splits above 64 is an invalid argument, also when the plan it asks
    # for would not fit the array
    d = workloads.random_attn(16, 8, 128, 512, 4096, 4096, p_invalid=0.0, seed=3).to("cuda")
    B, S, H, D = d.q.shape
    stream = torch.cuda.current_stream().cuda_stream
    for ns in (65, 1000):
        rc = binding.sa_sparse_attn_fwd_static_ws(d.q.data_ptr(), d.kv.data_ptr(), d.attn_sink.data_ptr(),
                                                  d.topk_idxs.data_ptr(), d.softmax_scale, d.q.data_ptr(), B, S,
                                                  H, D, 4096, 4096, ns, stream)
        assert binding.sa_status_string(rc) == "SA_ERR_INVALID_ARG"
    rc = binding.sa_sparse_attn_fwd_static_ws(d.q.data_ptr(), d.kv.data_ptr(), d.attn_sink.data_ptr(),
                                              d.topk_idxs.data_ptr(), float("nan"), d.q.data_ptr(), B, S, H, D,
                                              4096, 4096, 64, stream)
    assert binding.sa_status_string(rc) == "SA_ERR_INVALID_ARG"


def test_static_workspace_with_more_than_2048_slots():
    # K > 2048 forces ceil(K / 2048) splits whatever the batch: 64 tokens x 2
    # splits x 128 x 512 x 4 bytes exceed the array, 16 tokens fit and match
    # the regular entry point
    stream = torch.cuda.current_stream().cuda_stream
    big = workloads.random_attn(64, 1, 128, 512, 3000, 2560, p_invalid=0.1, seed=11).to("cuda")
    B, S, H, D = big.q.shape
    assert binding.sa_sparse_attn_workspace_size(B, S, H, D, 2560, 0) > (32 << 20)
    out = torch.full_like(big.q, float("nan"))
    rc = binding.sa_sparse_attn_fwd_static_ws(big.q.data_ptr(), big.kv.data_ptr(), big.attn_sink.data_ptr(),
                                              big.topk_idxs.data_ptr(), big.softmax_scale, out.data_ptr(), B, S, H,
                                              D, 3000, 2560, 0, stream)
    assert binding.sa_status_string(rc) == "SA_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all(), "a rejected call writes no output"
    small = workloads.random_attn(16, 1, 128, 512, 3000, 2560, p_invalid=0.1, seed=12).to("cuda")
    assert binding.sa_sparse_attn_workspace_size(16, 1, 128, 512, 2560, 0) <= (32 << 20)
    ref = _regular(small, 0)
    got = _static(small, 0)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    _close(got, ref)
