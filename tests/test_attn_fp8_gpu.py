"""GPU parity of sparse_attn over an FP8 kv cache (584-byte V4 rows: E4M3
codes with E8M0 tile scales, bf16 RoPE dims) against the CPU oracle's
``sparse_attn_fp8``, which decodes every row exactly.

Bar, element by element: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| (the rows
widen to bf16 exactly, so the bf16 path's tolerance carries over)."""

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


def _run(inp: workloads.Fp8AttnInputs, num_splits=0, topk_length=None, sink=None, scale=None):
    d = inp.to("cuda")
    s = d.attn_sink if sink is None else sink.cuda()
    o = binding.sparse_attn_fp8(d.q, d.kv8, s, d.topk_idxs, inp.softmax_scale if scale is None else scale,
                                num_splits=num_splits,
                                topk_length=None if topk_length is None else topk_length.cuda())
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    return o


@pytest.mark.parametrize("B,S,H,T,K,p,splits", [
    (1, 2, 8, 100, 64, 0.1, 0),
    (2, 3, 128, 700, 200, 0.2, 0),
    (1, 4, 64, 3000, 1152, 0.05, 0),
    (2, 2, 128, 5000, 1152, 0.3, 2),
    (1, 1, 128, 9000, 2000, 0.0, 5),     # more splits than fit one cluster: separate combine
    (3, 1, 16, 300, 129, 0.5, 1),        # ragged last tile, one split
])
def test_random_fp8_cases(B, S, H, T, K, p, splits):
    inp = workloads.random_attn_fp8(B, S, H, T, K, p_invalid=p, seed=B * 97 + T)
    o = _run(inp, num_splits=splits)
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    assert_close(o, want, f"B{B} S{S} H{H} T{T} K{K}")


def test_split_count_invariance():
    inp = workloads.random_attn_fp8(1, 2, 128, 4000, 1152, p_invalid=0.1, seed=5)
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    for ns in (1, 2, 3, 4, 9):
        assert_close(_run(inp, num_splits=ns), want, f"splits={ns}")


def test_topk_length():
    inp = workloads.random_attn_fp8(2, 3, 32, 800, 300, p_invalid=0.1, seed=7)
    lens = torch.tensor([[0, 1, 300], [65, -4, 1000]], dtype=torch.int32)
    o = _run(inp, topk_length=lens)
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, topk_length=lens)
    assert_close(o, want, "topk_length")


def test_edges_all_invalid_sinks_and_scales():
    inp = workloads.random_attn_fp8(1, 3, 8, 200, 70, p_invalid=0.2, seed=9)
    inp.topk_idxs[0, 1] = -1                         # a token with no valid slot: o = 0
    sink = torch.tensor([0.0, float("inf"), float("-inf"), 1.5, -2.0, float("inf"), 0.3, float("-inf")])
    for scale in (inp.softmax_scale, 0.0, -0.05):
        o = _run(inp, sink=sink, scale=scale)
        want = oracle.sparse_attn_fp8(inp.q, inp.kv8, sink, inp.topk_idxs, scale)
        assert_close(o, want, f"scale={scale}")
        assert float(o[0, 1].float().abs().max()) == 0.0


def test_subnormal_codes_and_extreme_scales():
    # codes of every class (subnormal, normal, max 448, both signs) under
    # scales from 2^-40 to 2^10; all values stay inside bf16's normal range
    g = torch.Generator().manual_seed(11)
    inp = workloads.random_attn_fp8(1, 2, 8, 64, 64, p_invalid=0.0, seed=11)
    kv8 = inp.kv8.clone()
    codes = torch.tensor([0x01, 0x07, 0x08, 0x7E, 0x81, 0xFE, 0x00, 0x80], dtype=torch.uint8)
    kv8[0, :, :448] = codes[torch.randint(0, 8, (64, 448), generator=g)]
    kv8[0, :, 576:583] = torch.tensor([87, 100, 127, 137, 110, 120, 127], dtype=torch.uint8)
    inp.kv8 = kv8
    o = _run(inp)
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    assert_close(o, want, "extreme codes")


def test_full_v4_fp8_decode_every_token():
    inp = workloads.v4_ratio4_decode_fp8()
    o = _run(inp)
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    assert_close(o, want, "V4 ratio-4 decode, FP8 kv")
    assert binding.sa_sparse_attn_fp8_launch_count(32, 1, 128, 1152) == 1


@pytest.mark.parametrize("scale_byte", [134, 127, 135, 150])
def test_zero_and_subnormal_codes_at_the_fast_and_exact_paths(scale_byte):
    # only zero and subnormal codes (m * 2^-9) under one scale: at 2^7 the
    # values are m / 4, so a flushed subnormal would show; scale bytes above
    # 134 take the exact conversion path
    g = torch.Generator().manual_seed(scale_byte)
    inp = workloads.random_attn_fp8(1, 2, 16, 64, 64, p_invalid=0.0, seed=13)
    kv8 = inp.kv8.clone()
    sub = torch.tensor([0x00, 0x01, 0x02, 0x03, 0x04, 0x05, 0x06, 0x07,
                        0x80, 0x81, 0x82, 0x83, 0x84, 0x85, 0x86, 0x87], dtype=torch.uint8)
    kv8[0, :, :448] = sub[torch.randint(0, 16, (64, 448), generator=g)]
    kv8[0, :, 576:583] = scale_byte
    inp.kv8 = kv8
    dec = oracle.decode_kv_fp8(kv8)
    assert np.abs(dec[..., :448]).max() > 0
    o = _run(inp, scale=0.02)
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, 0.02)
    assert_close(o, want, f"subnormal codes, scale byte {scale_byte}")


def test_rows_no_valid_slot_points_at_are_never_read():
    # every row that no valid slot points at, row 0 included, holds NaN codes
    # and NaN scales; invalid slots (-1, past T) must contribute exact zeros,
    # never a NaN through P.V (the copy path does not copy their rows)
    inp = workloads.random_attn_fp8(2, 2, 16, 300, 130, p_invalid=0.3, seed=21)
    idx = inp.topk_idxs.clone()
    idx[0, 0, :5] = 300                       # past T: invalid
    idx[idx == 0] = 1                         # no valid slot points at row 0
    inp.topk_idxs = idx
    used = torch.zeros(2, 300, dtype=torch.bool)
    for b in range(2):
        v = idx[b][(idx[b] >= 0) & (idx[b] < 300)]
        used[b, v.long()] = True
    kv8 = inp.kv8.clone()
    kv8[~used] = 0xFF                         # E4M3 NaN codes, NaN bf16 RoPE values, E8M0 255 = NaN scales
    inp.kv8 = kv8
    assert not used[:, 0].any()
    o = _run(inp)
    assert torch.isfinite(o.float()).all()
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    assert_close(o, want, "NaN rows that no valid slot reads")


def test_even_last_row_of_the_cache_with_poison_after_it():
    # B*T odd: the cache's last row has an even index, and a 16-byte-aligned
    # window over its scale bytes would reach 8 bytes past the cache.  The
    # bytes after the cache hold NaN patterns; the last row is picked by
    # several slots of every token of the last request.
    B, S, H, T, K = 3, 2, 16, 101, 64
    inp = workloads.random_attn_fp8(B, S, H, T, K, p_invalid=0.1, seed=77)
    idx = inp.topk_idxs.clone()
    idx[B - 1, :, :6] = T - 1
    inp.topk_idxs = idx
    big = torch.full((B * T + 2, 584), 0xFF, dtype=torch.uint8, device="cuda")
    big[: B * T] = inp.kv8.reshape(B * T, 584).cuda()
    kv = big[: B * T].view(B, T, 584)
    d = inp.to("cuda")
    o = binding.sparse_attn_fp8(d.q, kv, d.attn_sink, d.topk_idxs, inp.softmax_scale)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    want = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    assert_close(o, want, "even last row of the cache")
