"""GPU parity of the mask consumer (dense attention over the keys a bit-packed
mask admits) against the CPU oracle's ``masked_dense_attn``.

Bar, element by element, as for sparse_attn: |gpu - oracle| <= 1e-2 + 1e-2 |oracle|.
Masks are random 32-bit words (any bit pattern is a valid mask), masks the
oracle builds from top-k rows, and, at the full mask workload's size, the mask
the GPU builder writes (a consumer reads whatever the builder wrote)."""

import numpy as np
import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what=""):
    g = gpu.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    bad = np.abs(g - ref) > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first at "
                             f"{tuple(i)}: gpu={g[tuple(i)]} oracle={ref[tuple(i)]}")


def _inputs(B, S, H, D, T, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, S, H, D, generator=g).to(torch.bfloat16)
    kv = torch.randn(B, T, D, generator=g).to(torch.bfloat16)
    sink = torch.randn(H, generator=g)
    return q, kv, sink


def _random_mask(B, rows, words, density, seed):
    rng = np.random.default_rng(seed)
    bits = rng.random((B, rows, words * 32)) < density
    return np.packbits(bits, axis=-1, bitorder="little").view(np.uint32).reshape(B, rows, words)


def _gpu(q, kv, sink, mask_u32, scale, key_start_word=False, num_splits=0):
    m = torch.from_numpy(np.ascontiguousarray(mask_u32).view(np.int32)).cuda()
    o = binding.masked_dense_attn(q.cuda(), kv.cuda(), sink.cuda(), m, scale, key_start_word=key_start_word,
                                  num_splits=num_splits)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    return o


@pytest.mark.parametrize("B,S,H,D,T,density,splits", [
    (1, 3, 8, 64, 256, 0.3, 0),
    (2, 5, 8, 64, 777, 0.1, 0),
    (2, 4, 16, 128, 300, 0.6, 1),
    (1, 6, 128, 512, 1000, 0.25, 0),
    (3, 2, 128, 512, 2500, 0.05, 3),
    (2, 3, 64, 256, 4100, 0.5, 0),      # more keys than one split holds
    (1, 2, 8, 64, 9000, 0.2, 12),       # more splits than a cluster holds: separate combine kernel
    (1, 3, 128, 512, 129, 1.0, 0),      # every key admitted, ragged last tile
])
def test_random_masks(B, S, H, D, T, density, splits):
    q, kv, sink = _inputs(B, S, H, D, T, seed=B * 1000 + T)
    words = workloads.ceil_div(workloads.ceil_div(T, 32), 4) * 4
    mask = _random_mask(B, S + 1, words, density, seed=T)
    scale = D ** -0.5
    o = _gpu(q, kv, sink, mask, scale, num_splits=splits)
    assert_close(o, oracle.masked_dense_attn(q, kv, sink, mask, scale), f"B{B} S{S} H{H} D{D} T{T}")


@pytest.mark.parametrize("B,S,H,D,T,density,splits", [
    (3, 37, 8, 64, 1000, 0.25, 0),     # 16 tokens a unit, ragged last group, 3 requests
    (2, 11, 3, 64, 513, 0.3, 0),       # H = 3: 42 tokens on 126 of the 128 rows
    (2, 9, 24, 128, 700, 0.2, 2),      # 5 tokens of 24 heads, 2 key splits
    (1, 6, 1, 256, 2000, 0.1, 0),      # one head: 128 tokens a unit, 6 of them live
    (2, 5, 128, 128, 450, 0.5, 0),     # one token a unit
    (1, 40, 16, 64, 130, 1.0, 0),      # every key admitted, the last tile holds 2 keys
    (2, 33, 8, 64, 3000, 0.002, 0),    # most key tiles admit nothing and are skipped
])
def test_packed_query_groups(B, S, H, D, T, density, splits):
    # the consumer for D <= 256 packs 128 / H query tokens into one unit's
    # MMA rows; groups straddle neither requests nor the window
    q, kv, sink = _inputs(B, S, H, D, T, seed=7 * S + H)
    words = workloads.ceil_div(workloads.ceil_div(T, 32), 4) * 4
    mask = _random_mask(B, S + 3, words, density, seed=S + T)
    scale = D ** -0.5
    o = _gpu(q, kv, sink, mask, scale, num_splits=splits)
    assert_close(o, oracle.masked_dense_attn(q, kv, sink, mask, scale), f"B{B} S{S} H{H} D{D} T{T}")


def test_split_count_does_not_change_the_result():
    q, kv, sink = _inputs(1, 4, 128, 512, 3000, seed=5)
    mask = _random_mask(1, 4, 96, 0.3, seed=6)
    want = oracle.masked_dense_attn(q, kv, sink, mask, 0.05)
    for ns in (1, 2, 4, 7, 20):
        assert_close(_gpu(q, kv, sink, mask, 0.05, num_splits=ns), want, f"splits={ns}")


def test_empty_rows_and_infinite_sinks():
    B, S, H, D, T = 1, 4, 8, 64, 300
    q, kv, _ = _inputs(B, S, H, D, T, seed=7)
    mask = _random_mask(B, S, 12, 0.4, seed=8)
    mask[0, 1] = 0                       # query 1 admits nothing: o = 0
    sink = torch.tensor([0.5, float("inf"), float("-inf"), -3.0, 2.0, float("inf"), float("-inf"), 0.0])
    o = _gpu(q, kv, sink, mask, 0.125)
    want = oracle.masked_dense_attn(q, kv, sink, mask, 0.125)
    assert_close(o, want, "sinks")
    assert float(o[0, 1].float().abs().max()) == 0.0
    assert float(o[0, :, 1].float().abs().max()) == 0.0     # sink = +inf: every real weight is zero


def test_mask_built_from_topk_rows_matches_sparse_attention():
    # the builder's output consumed by the dense path equals sparse attention
    # over the same indices (oracle on both sides of the comparison chain)
    inp = workloads.random_attn(2, 5, 8, 64, 700, 90, p_invalid=0.2, seed=11)
    B, S = 2, 5
    cu = np.arange(0, B * S + 1, S, dtype=np.int32)
    mask = oracle.build_topk_mask(inp.topk_idxs.reshape(B * S, -1).numpy(), cu, B, S, 700)
    o = _gpu(inp.q, inp.kv, inp.attn_sink, mask, inp.softmax_scale)
    assert_close(o, oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale), "vs sparse")


@pytest.mark.parametrize("key_starts", [(0, 17), (40, -5), (1000, 3)])
def test_key_start_word_offsets_the_bit_test(key_starts):
    # a context chunk kv[b] of T keys at absolute position key_starts[b]; the
    # mask row covers absolute positions and its reserved word holds the start
    B, S, H, D, T = 2, 3, 8, 64, 400
    q, kv, sink = _inputs(B, S, H, D, T, seed=13)
    rng = np.random.default_rng(14)
    max_key = 1500
    topk = rng.integers(-3, max_key, size=(B * S, 160)).astype(np.int32)
    cu = np.arange(0, B * S + 1, S, dtype=np.int32)
    mask = oracle.build_topk_mask(topk, cu, B, S, max_key, key_starts=np.array(key_starts, np.int32))
    o = _gpu(q, kv, sink, mask, D ** -0.5, key_start_word=True)
    want = oracle.masked_dense_attn(q, kv, sink, mask, D ** -0.5, key_offset=list(key_starts))
    assert_close(o, want, f"key_starts={key_starts}")


@pytest.mark.parametrize("D,key_starts", [(64, (256, 384)), (128, (128, 0)), (256, (640, 64))])
def test_key_start_multiple_of_the_tile(D, key_starts):
    # key offsets that are multiples of the key tile take the packed
    # consumer's one-vector path for the mask words of every whole tile
    B, S, H, T = 2, 5, 8, 700
    q, kv, sink = _inputs(B, S, H, D, T, seed=19 + D)
    rng = np.random.default_rng(20)
    max_key = 1500
    topk = rng.integers(-3, max_key, size=(B * S, 300)).astype(np.int32)
    cu = np.arange(0, B * S + 1, S, dtype=np.int32)
    mask = oracle.build_topk_mask(topk, cu, B, S, max_key, key_starts=np.array(key_starts, np.int32))
    o = _gpu(q, kv, sink, mask, D ** -0.5, key_start_word=True)
    want = oracle.masked_dense_attn(q, kv, sink, mask, D ** -0.5, key_offset=list(key_starts))
    assert_close(o, want, f"D={D} key_starts={key_starts}")


def test_reserved_word_is_never_a_key_bit():
    # key_start = -1 fills the reserved word of row 0 with ones; the chunk's
    # keys reach its positions, and the consumer must admit none of them
    B, S, H, D, T = 1, 3, 8, 64, 300
    q, kv, sink = _inputs(B, S, H, D, T, seed=17)
    rng = np.random.default_rng(18)
    topk = rng.integers(-2, 200, size=(S, 70)).astype(np.int32)
    mask = oracle.build_topk_mask(topk, np.array([0, S], np.int32), B, S, 200, key_starts=np.array([-1], np.int32))
    assert mask[0, 0, -1] == 0xFFFFFFFF and 32 * (mask.shape[2] - 1) < T - 1
    o = _gpu(q, kv, sink, mask, D ** -0.5, key_start_word=True)
    assert_close(o, oracle.masked_dense_attn(q, kv, sink, mask, D ** -0.5, key_offset=[-1]), "reserved word")


def test_zero_and_negative_scale():
    q, kv, sink = _inputs(1, 2, 8, 64, 200, seed=15)
    mask = _random_mask(1, 2, 8, 0.3, seed=16)
    for scale in (0.0, -0.2):
        assert_close(_gpu(q, kv, sink, mask, scale), oracle.masked_dense_attn(q, kv, sink, mask, scale),
                     f"scale={scale}")


def test_full_mask_workload_consumed_on_the_gpu():
    # the mask workload at full size (4 requests x 2048 queries, 8193 keys):
    # the GPU builder's mask, consumed by the GPU dense path, compared on
    # every query row with the sparse oracle over the same top-k rows (the
    # keys a row admits are exactly its top-k indices; the oracle's
    # masked-dense and sparse forms are pinned equal)
    mi = workloads.topk_mask()
    d = mi.to("cuda")
    shape = binding.topk_mask_shape(mi.batch, mi.max_q_len, mi.max_key_len, True)
    mask = torch.zeros(shape, dtype=torch.int32, device="cuda")
    binding.build_topk_mask(d.topk, d.cu_q_lens, mi.max_q_len, mi.max_key_len, d.key_starts, out=mask)
    B, S, H, D, T = 4, 2048, 8, 64, 8193
    q, kv, sink = _inputs(B, S, H, D, T, seed=1005)
    o = binding.masked_dense_attn(q.cuda(), kv.cuda(), sink.cuda(), mask, D ** -0.5)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    want = oracle.sparse_attn(q, kv, sink, mi.topk.reshape(B, S, -1), D ** -0.5)
    assert_close(o, want, "mask workload, every row")
