"""GPU parity of the bit-packed top-k mask builder against the CPU oracle.

The bar is bit-exactness over the WHOLE buffer: every buffer starts filled
with a sentinel, so padding words, rows past a request's query count and
padded query rows must come back holding the sentinel (the pages' "padding is
preserved" contract), and live words must equal the oracle's bit by bit."""

import numpy as np
import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

SENT = np.uint32(workloads.SENTINEL_U32)


def _gpu_build(mi: workloads.MaskInputs, fill=SENT):
    shape = binding.topk_mask_shape(mi.batch, mi.max_q_len, mi.max_key_len, mi.key_starts is not None)
    out = torch.from_numpy(np.full(shape, fill, dtype=np.uint32).view(np.int32)).cuda()
    d = mi.to("cuda")
    binding.build_topk_mask(d.topk, d.cu_q_lens, mi.max_q_len, mi.max_key_len, d.key_starts, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


def _oracle_build(mi: workloads.MaskInputs, fill=SENT):
    shape = oracle.topk_mask_shape(mi.batch, mi.max_q_len, mi.max_key_len, mi.key_starts is not None)
    out = np.full(shape, fill, dtype=np.uint32)
    return oracle.build_topk_mask(mi.topk.numpy(), mi.cu_q_lens.numpy(), mi.batch, mi.max_q_len, mi.max_key_len,
                                  None if mi.key_starts is None else mi.key_starts.numpy(), out=out)


def test_worked_example_from_the_page():
    # one request, one query, 129 keys, top-k [0, 128] -> row [1,0,0,0,1,0,0,0]
    shape = binding.topk_mask_shape(1, 1, 129)
    out = torch.zeros(shape, dtype=torch.int32, device="cuda")
    topk = torch.tensor([[0, 128]], dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    mask = binding.build_topk_mask(topk, cu, 1, 129, out=out)
    assert mask[:1, :1].shape == (1, 1, 8)
    assert mask[0, 0].tolist() == [1, 0, 0, 0, 1, 0, 0, 0]
    assert int(mask[0, 1:].abs().sum()) == 0


@pytest.mark.parametrize("seed", range(8))
def test_random_cases_bit_exact(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 5))
    q_lens = [int(rng.integers(0, 40)) for _ in range(B)]
    max_q = max(q_lens + [1]) + int(rng.integers(0, 3))
    keys = int(rng.integers(1, 3000))
    K = int(rng.integers(1, 300))
    rows = sum(q_lens)
    topk = torch.from_numpy(rng.integers(-5, keys + 5, size=(rows, K)).astype(np.int32))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    ks = torch.from_numpy(rng.integers(-2**31, 2**31 - 1, size=B).astype(np.int32)) if seed % 2 else None
    mi = workloads.MaskInputs(topk, cu, B, max_q, keys, ks)
    np.testing.assert_array_equal(_gpu_build(mi), _oracle_build(mi))


def test_full_workload_bit_exact():
    mi = workloads.topk_mask()  # B=4, Q=2048, 8193 keys, K=2048, key_starts reserved
    got = _gpu_build(mi)
    assert got.shape == (4, 2048, 260)
    np.testing.assert_array_equal(got, _oracle_build(mi))
    assert (got[:, :, 257:259] == SENT).all()        # padding words untouched
    assert [int(got[b, 0, 259]) for b in range(4)] == [0, 1, 31, 8192]


def test_ragged_requests_leave_rows_past_q_len_untouched():
    mi = workloads.topk_mask(seed=7, B=3, Q=300, max_key_len=700, K=96, key_starts=(5, 6, 7), q_lens=[300, 1, 0])
    got = _gpu_build(mi)
    np.testing.assert_array_equal(got, _oracle_build(mi))
    assert (got[1, 1:] == SENT).all() and (got[2, 1:] == SENT).all()
    assert (got[2, 0, :-1] == SENT).all() and got[2, 0, -1] == 7


def test_single_request_equals_same_rows_of_a_batch():
    mi = workloads.topk_mask(seed=9, B=3, Q=200, max_key_len=1000, K=128, key_starts=None)
    full = _gpu_build(mi)
    one = workloads.MaskInputs(mi.topk[200:400], torch.tensor([0, 200], dtype=torch.int32), 1, 200, 1000, None)
    np.testing.assert_array_equal(_gpu_build(one)[0], full[1])


def test_wide_rows_use_global_path_bit_exact():
    # 300000 keys -> 9375 words per row: wider than the shared-memory row image
    rng = np.random.default_rng(5)
    topk = torch.from_numpy(rng.integers(-1, 300000, size=(6, 700)).astype(np.int32))
    mi = workloads.MaskInputs(topk, torch.tensor([0, 4, 6], dtype=torch.int32), 2, 4, 300000,
                              torch.tensor([3, 4], dtype=torch.int32))
    np.testing.assert_array_equal(_gpu_build(mi), _oracle_build(mi))


def test_mid_width_rows_use_cta_path_bit_exact():
    # 100000 keys -> 3125 words per row: too wide for a warp's image, one CTA per row
    rng = np.random.default_rng(8)
    topk = torch.from_numpy(rng.integers(-3, 100003, size=(7, 1000)).astype(np.int32))
    mi = workloads.MaskInputs(topk, torch.tensor([0, 3, 7], dtype=torch.int32), 2, 5, 100000,
                              torch.tensor([-1, 12], dtype=torch.int32))
    np.testing.assert_array_equal(_gpu_build(mi), _oracle_build(mi))


def test_unaligned_topk_rows_scalar_path():
    rng = np.random.default_rng(6)
    topk = torch.from_numpy(rng.integers(0, 500, size=(9, 37)).astype(np.int32))  # K % 4 != 0
    mi = workloads.MaskInputs(topk, torch.tensor([0, 5, 9], dtype=torch.int32), 2, 5, 500, None)
    np.testing.assert_array_equal(_gpu_build(mi), _oracle_build(mi))


def test_deterministic_and_overwrites_stale_live_words():
    mi = workloads.topk_mask(seed=3, B=2, Q=64, max_key_len=4000, K=256, key_starts=None)
    a = _gpu_build(mi, fill=np.uint32(0xFFFFFFFF))  # stale ones in live words must be cleared
    b = _gpu_build(mi, fill=np.uint32(0xFFFFFFFF))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, _oracle_build(mi, fill=np.uint32(0xFFFFFFFF)))


def test_cuda_graph_replay_tracks_new_indices():
    mi = workloads.topk_mask(seed=11, B=2, Q=128, max_key_len=2048, K=64, key_starts=(0, 9))
    d = mi.to("cuda")
    shape = binding.topk_mask_shape(2, 128, 2048, True)
    out = torch.zeros(shape, dtype=torch.int32, device="cuda")
    binding.build_topk_mask(d.topk, d.cu_q_lens, 128, 2048, d.key_starts, out=out)  # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            binding.build_topk_mask(d.topk, d.cu_q_lens, 128, 2048, d.key_starts, out=out)
    for seed in (12, 13):
        nxt = workloads.topk_mask(seed=seed, B=2, Q=128, max_key_len=2048, K=64, key_starts=(0, 9))
        d.topk.copy_(nxt.topk.cuda())
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        want = _oracle_build(nxt, fill=np.uint32(0))
        np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want)


def test_masked_dense_with_gpu_mask_equals_sparse_oracle():
    # the full mask workload's GPU-built rows, consumed by a dense attention over
    # all 8193 keys, give the same output as sparse attention over the indices
    mi = workloads.topk_mask()
    mask = _gpu_build(mi, fill=np.uint32(0))
    g = torch.Generator().manual_seed(1005)
    B, H, D, T = 4, 8, 64, 8193
    kv = torch.randn(B, T, D, generator=g).to(torch.bfloat16)
    sel = [0, 1, 777, 2047]
    q = torch.randn(B, len(sel), H, D, generator=g).to(torch.bfloat16)
    sink = torch.randn(H, generator=g)
    idx = torch.stack([mi.topk[b * 2048 + torch.tensor(sel)] for b in range(B)])  # [B, len(sel), K]
    dense = oracle.masked_dense_attn(q, kv, sink, mask[:, sel, :], D ** -0.5)
    sparse = oracle.sparse_attn(q, kv, sink, idx, D ** -0.5)
    np.testing.assert_allclose(dense, sparse, rtol=1e-10, atol=1e-12)
