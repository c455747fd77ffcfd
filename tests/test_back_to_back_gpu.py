"""Calls issued back to back on one stream, sharing one workspace, with no
synchronisation between them: every kernel of the library launches with a
programmatic dependency on the stream's previous kernel (its launch overlaps
the previous kernel's run) and waits for that kernel before its first global
memory access.  Each output must equal, bit for bit, the output of the same
call made alone, and the first one must match the oracle."""

import numpy as np
import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,S,H,D,T,K,splits", [
    (2, 1, 128, 512, 2048, 1152, 0),    # splits combined inside the cluster
    (1, 2, 128, 512, 4096, 1152, 6),    # more splits than a cluster holds: a separate combine kernel
    (4, 2, 64, 128, 700, 300, 0),       # one CTA per unit
])
def test_back_to_back_calls_equal_isolated_calls(B, S, H, D, T, K, splits):
    dev = torch.device("cuda")
    sets = [workloads.random_attn(B, S, H, D, T, K, p_invalid=0.1, seed=40 + i).to(dev) for i in range(6)]
    ws = binding.workspace_for(B, S, H, D, K, splits, device=dev)
    outs = [torch.empty_like(s.q) for s in sets]
    alone = []
    for s in sets:
        o = binding.sparse_attn(s.q, s.kv, s.attn_sink, s.topk_idxs, s.softmax_scale, workspace=ws, num_splits=splits)
        torch.cuda.synchronize()
        alone.append(o.clone())
    for _ in range(3):                                  # three rounds over the six sets, no sync in between
        for s, o in zip(sets, outs):
            binding.sparse_attn(s.q, s.kv, s.attn_sink, s.topk_idxs, s.softmax_scale, out=o, workspace=ws,
                                num_splits=splits)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    for i, (o, a) in enumerate(zip(outs, alone)):
        assert torch.equal(o, a), f"set {i}: a back-to-back call differs from the same call made alone"
    c = workloads.random_attn(B, S, H, D, T, K, p_invalid=0.1, seed=40)
    want = oracle.sparse_attn(c.q, c.kv, c.attn_sink, c.topk_idxs, c.softmax_scale)
    g = outs[0].float().cpu().numpy().astype(np.float64)
    assert (np.abs(g - want) <= 1e-2 + 1e-2 * np.abs(want)).all()


def test_mask_build_and_consumer_back_to_back():
    # build, consume, build again into the same mask buffer, consume again:
    # the second build must not overwrite the mask while the first consumer
    # still reads it, and each consumer sees its own mask
    dev = torch.device("cuda")
    a = workloads.topk_mask(seed=51, B=2, Q=64, max_key_len=700, K=100, key_starts=None)
    b = workloads.topk_mask(seed=52, B=2, Q=64, max_key_len=700, K=100, key_starts=None)
    g = torch.Generator().manual_seed(53)
    H, D = 8, 64
    q = torch.randn(2, 64, H, D, generator=g).to(torch.bfloat16).to(dev)
    kv = torch.randn(2, 700, D, generator=g).to(torch.bfloat16).to(dev)
    sink = torch.randn(H, generator=g).to(dev)
    shape = binding.topk_mask_shape(2, 64, 700, False)
    mask = torch.zeros(shape, dtype=torch.int32, device=dev)
    ws_n = binding.sa_masked_dense_attn_workspace_size(2, 64, H, D, 700)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=dev)
    outs = []
    for m in (a, b):
        md = m.to(dev)
        binding.build_topk_mask(md.topk, md.cu_q_lens, md.max_q_len, md.max_key_len, None, out=mask)
        outs.append(binding.masked_dense_attn(q, kv, sink, mask, D ** -0.5, workspace=ws))
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    for m, o in zip((a, b), outs):
        mk = oracle.build_topk_mask(m.topk, m.cu_q_lens, m.batch, m.max_q_len, m.max_key_len, None)
        want = oracle.masked_dense_attn(q.cpu(), kv.cpu(), sink.cpu(), mk, D ** -0.5)
        got = o.float().cpu().numpy().astype(np.float64)
        assert (np.abs(got - want) <= 1e-2 + 1e-2 * np.abs(want)).all()
