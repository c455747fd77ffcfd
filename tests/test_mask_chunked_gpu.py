"""GPU parity of the chunked mask path: mask windows of query rows with
per-request live key ends (bit-exact against the oracle's window builder),
the consumer over a window with live ends, and the windowed build + consume
driver against the oracle's whole-mask consumer.

Bars: bit-exact for the mask; |gpu - oracle| <= 1e-2 + 1e-2 |oracle| for the
attention, on the live query rows (rows past a request's query count are
unspecified)."""

import numpy as np
import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

SENT = np.uint32(workloads.SENTINEL_U32)
ATOL = RTOL = 1e-2


def assert_close(gpu, ref, what=""):
    g = gpu.float().cpu().numpy().astype(np.float64) if isinstance(gpu, torch.Tensor) else gpu
    bad = np.abs(g - ref) > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first at {tuple(i)}: "
                             f"gpu={g[tuple(i)]} oracle={ref[tuple(i)]}")


def _case(seed, B, max_q, keys, K):
    rng = np.random.default_rng(seed)
    q_lens = [int(rng.integers(1, max_q + 1)) for _ in range(B)]
    q_lens[0] = max_q
    topk = rng.integers(-2, keys + 2, size=(sum(q_lens), K)).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return rng, q_lens, topk, cu


@pytest.mark.parametrize("q0,rows,ends,ks", [
    (0, 300, None, None),
    (128, 128, [0, 333, 5000], None),
    (256, 100, [64, 700, 31], [5, 0, 7]),
    (0, 77, [1, 640, 700], [1, 2, 3]),
])
def test_mask_window_bit_exact(q0, rows, ends, ks):
    _, q_lens, topk, cu = _case(71, 3, 300, 700, 48)
    shape = binding.topk_mask_shape(3, rows, 700, ks is not None)
    out = torch.from_numpy(np.full(shape, SENT, dtype=np.uint32).view(np.int32)).cuda()
    t = lambda x: None if x is None else torch.tensor(x, dtype=torch.int32).cuda()
    binding.build_topk_mask_window(torch.from_numpy(topk).cuda(), torch.from_numpy(cu).cuda(), q0, rows, 700,
                                   key_starts=t(ks), key_ends=t(ends), out=out)
    torch.cuda.synchronize()
    want = oracle.build_topk_mask_window(topk, cu, 3, q0, rows, 700,
                                         key_starts=None if ks is None else np.array(ks, np.int32),
                                         key_ends=None if ends is None else np.array(ends, np.int32),
                                         out=np.full(shape, SENT, dtype=np.uint32))
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want)


def test_wide_rows_window_with_live_ends():
    # rows wider than the warp path (CTA-per-row builder)
    _, q_lens, topk, cu = _case(72, 2, 40, 100000, 300)
    ends = [70000, 99999]
    shape = binding.topk_mask_shape(2, 20, 100000)
    out = torch.from_numpy(np.full(shape, SENT, dtype=np.uint32).view(np.int32)).cuda()
    binding.build_topk_mask_window(torch.from_numpy(topk).cuda(), torch.from_numpy(cu).cuda(), 10, 20, 100000,
                                   key_ends=torch.tensor(ends, dtype=torch.int32).cuda(), out=out)
    torch.cuda.synchronize()
    want = oracle.build_topk_mask_window(topk, cu, 2, 10, 20, 100000, key_ends=np.array(ends, np.int32),
                                         out=np.full(shape, SENT, dtype=np.uint32))
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want)


def _attn_inputs(B, Q, H, D, T, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, Q, H, D, generator=g).to(torch.bfloat16),
            torch.randn(B, T, D, generator=g).to(torch.bfloat16),
            torch.randn(H, generator=g))


@pytest.mark.parametrize("H,D", [(8, 64), (16, 128), (32, 256)])
@pytest.mark.parametrize("with_ks", [False, True])
@pytest.mark.parametrize("cap", [0, 60000, 30000])
def test_windowed_build_and_consume_matches_the_whole_mask_oracle(cap, with_ks, H, D):
    # max_q 300 queries, 700 key positions; cap 60000 B -> windows of 256
    # rows, 30000 B -> windows of 128 rows, 0 -> the whole mask at once; the
    # packed consumer with one (D = 64) or two (D = 128, 256) S / P buffers
    B, Q, keys, K = 2, 300, 700, 50
    _, q_lens, topk, cu = _case(73 + cap, B, Q, keys, K)
    ks = np.array([0, 0], np.int32) if not with_ks else np.array([100, 37], np.int32)
    T = keys - int(ks.max())                  # kv[b] holds mask positions ks_b .. ks_b + T - 1
    ends = np.array([640, 700], np.int32)
    q, kv, sink = _attn_inputs(B, Q, H, D, T, seed=74)
    o = binding.topk_masked_attn(q.cuda(), kv.cuda(), sink.cuda(), torch.from_numpy(topk).cuda(),
                                 torch.from_numpy(cu).cuda(), D ** -0.5, keys,
                                 key_starts=torch.from_numpy(ks).cuda() if with_ks else None,
                                 key_ends=torch.from_numpy(ends).cuda(), cap_bytes=cap)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    full = oracle.build_topk_mask_window(topk, cu, B, 0, Q, keys, key_starts=ks if with_ks else None, key_ends=ends)
    want = oracle.masked_dense_attn(q, kv, sink, full, D ** -0.5,
                                    key_offset=ks.astype(np.int64) if with_ks else None, key_ends=ends)
    for b in range(B):
        assert_close(o[b, :q_lens[b]], want[b, :q_lens[b]], f"cap={cap} ks={with_ks} request {b}")
