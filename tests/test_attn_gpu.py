"""GPU parity of sparse_attn against the CPU oracle.

Bar (bf16 inputs, fp32 accumulation, bf16 output), element by element:
    |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|
Small cases are compared in full; the full-size workloads on sampled tokens
(the oracle evaluates them one by one) plus properties that hold at any size.
"""

import math

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


def run_gpu(inp: workloads.AttnInputs, num_splits=0, out=None):
    d = inp.to("cuda")
    o = binding.sparse_attn(d.q, d.kv, d.attn_sink, d.topk_idxs, d.softmax_scale, out=out, num_splits=num_splits)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    return o


def run_oracle(inp, tokens=None):
    return oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, tokens=tokens)


def test_tiny_workload_full():
    inp = workloads.tiny()
    assert_close(run_gpu(inp), run_oracle(inp), "tiny")


@pytest.mark.parametrize("H,D,K,T,p", [
    (128, 512, 64, 300, 0.0),      # exactly one tile
    (128, 512, 200, 1000, 0.3),    # ragged last tile, many -1
    (128, 512, 1152, 3000, 0.1),   # the V4 slot count
    (16, 512, 130, 400, 0.05),     # few heads
    (1, 512, 7, 50, 0.0),          # one head, K < tile
    (128, 256, 300, 512, 0.2),
    (100, 128, 129, 256, 0.1),
    (8, 64, 65, 100, 0.5),
])
def test_random_shapes_full(H, D, K, T, p):
    inp = workloads.random_attn(2, 3, H, D, T, K, p_invalid=p, seed=H * 7 + D + K)
    assert_close(run_gpu(inp), run_oracle(inp), f"H={H} D={D} K={K}")


def test_repeated_and_out_of_range_indices():
    inp = workloads.random_attn(2, 2, 128, 512, 100, 150, p_invalid=0.1, seed=3, distinct=False)
    inp.topk_idxs[0, 0, 5] = 100          # == T
    inp.topk_idxs[1, 1, 7] = 1 << 30
    inp.topk_idxs[0, 1, 9] = -12345
    assert_close(run_gpu(inp), run_oracle(inp), "repeats/out-of-range")


def test_all_invalid_tokens_give_exact_zero():
    inp = workloads.random_attn(2, 3, 128, 512, 200, 130, p_invalid=0.0, seed=4)
    inp.topk_idxs[0, 1] = -1
    inp.topk_idxs[1, 2, :] = 500          # all out of range
    o = run_gpu(inp)
    assert torch.count_nonzero(o[0, 1]) == 0 and torch.count_nonzero(o[1, 2]) == 0
    assert_close(o, run_oracle(inp), "all-invalid")


def test_sink_limits():
    inp = workloads.random_attn(1, 2, 128, 512, 300, 100, p_invalid=0.2, seed=5)
    inp.attn_sink[:64] = math.inf
    inp.attn_sink[64:] = -math.inf
    o = run_gpu(inp)
    assert torch.count_nonzero(o[:, :, :64]) == 0
    assert_close(o, run_oracle(inp), "sink=+-inf")


@pytest.mark.parametrize("scale", [0.0, -0.05, -1.0, 1e-4])
def test_zero_and_negative_scales_with_masked_slots(scale):
    # masked slots weigh exactly 0 whatever the sign of the scale
    inp = workloads.random_attn(2, 2, 128, 512, 500, 300, p_invalid=0.3, seed=41, scale=scale)
    for ns in (1, 2):
        assert_close(run_gpu(inp, num_splits=ns), run_oracle(inp), f"scale={scale} splits={ns}")


def test_single_valid_slot_closed_form():
    # one valid slot: o = sigmoid(x - sink) * row, checked against the oracle
    inp = workloads.random_attn(1, 2, 128, 512, 64, 70, p_invalid=0.0, seed=6)
    inp.topk_idxs[:] = -1
    inp.topk_idxs[0, 0, 33] = 5
    inp.topk_idxs[0, 1, 69] = 63
    assert_close(run_gpu(inp), run_oracle(inp), "K_valid=1")


def test_split_count_does_not_change_the_result():
    inp = workloads.random_attn(3, 1, 128, 512, 2000, 1152, p_invalid=0.1, seed=8)
    ref = run_oracle(inp)
    outs = []
    for ns in (1, 2, 3, 5, 18):
        o = run_gpu(inp, num_splits=ns)
        assert_close(o, ref, f"splits={ns}")
        outs.append(o.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 2e-2


@pytest.mark.parametrize("H,D,K,T,ns,p", [
    (100, 512, 700, 1500, 3, 0.1),    # 6-CTA cluster, rows split 34/34/32
    (128, 512, 1152, 2000, 4, 0.0),   # 8-CTA cluster
    (7, 512, 200, 300, 2, 0.3),       # fewer heads than splits x warps
    (128, 256, 1024, 1500, 8, 0.1),   # one head-dim CTA, 8 splits in a cluster
    (64, 64, 300, 500, 2, 0.2),
    (128, 512, 1152, 2000, 5, 0.1),   # 10 CTAs: too many for a cluster, separate combine
])
def test_split_combine_paths(H, D, K, T, ns, p):
    inp = workloads.random_attn(3, 2, H, D, T, K, p_invalid=p, seed=H + D + K + ns)
    assert_close(run_gpu(inp, num_splits=ns), run_oracle(inp), f"H={H} D={D} K={K} splits={ns}")


def test_split_with_no_active_tile_and_infinite_sinks():
    # the last splits of token (0, 0) see only invalid slots; two heads have sink = +inf
    inp = workloads.random_attn(2, 2, 128, 512, 1500, 1152, p_invalid=0.05, seed=31)
    inp.topk_idxs[0, 0, 300:] = -1
    inp.topk_idxs[1, 1, :700] = 5000     # out of range: the first splits are empty
    inp.attn_sink[3] = math.inf
    inp.attn_sink[77] = math.inf
    inp.attn_sink[5] = -math.inf
    for ns in (2, 3, 4):
        o = run_gpu(inp, num_splits=ns)
        assert torch.count_nonzero(o[:, :, 3]) == 0 and torch.count_nonzero(o[:, :, 77]) == 0
        assert_close(o, run_oracle(inp), f"empty splits, splits={ns}")


def test_launch_count_query():
    # splits x head-dim halves <= 8 CTAs combine in-kernel: one launch
    assert binding.sa_sparse_attn_launch_count(32, 1, 128, 512, 1152, 2) == 1
    assert binding.sa_sparse_attn_launch_count(32, 1, 128, 512, 1152, 4) == 1
    assert binding.sa_sparse_attn_launch_count(32, 1, 128, 512, 1152, 5) == 2
    assert binding.sa_sparse_attn_launch_count(32, 1, 128, 256, 1152, 8) == 1
    assert binding.sa_sparse_attn_launch_count(32, 1, 128, 512, 1152, 1) == 1
    assert binding.sa_sparse_attn_launch_count(0, 1, 128, 512, 1152, 2) == 0
    assert binding.sa_sparse_attn_launch_count(1, 1, 128, 96, 1152, 2) == 0


def test_deterministic():
    inp = workloads.random_attn(2, 2, 128, 512, 500, 300, p_invalid=0.1, seed=9)
    a, b = run_gpu(inp), run_gpu(inp)
    assert torch.equal(a, b)


def test_output_guard_bands_untouched():
    inp = workloads.random_attn(1, 3, 128, 512, 400, 200, p_invalid=0.1, seed=10)
    n = inp.q.numel()
    buf = torch.full((n + 2 * 4096,), -7.5, dtype=torch.bfloat16, device="cuda")
    view = buf[4096:4096 + n].view(inp.q.shape)
    run_gpu(inp, out=view)
    assert (buf[:4096] == -7.5).all() and (buf[4096 + n:] == -7.5).all()
    assert_close(view, run_oracle(inp), "guarded")


def test_cuda_graph_replay_with_new_invalid_tails():
    inp = workloads.v4_ratio128_decode(B=8)
    d = inp.to("cuda")
    out = torch.empty_like(d.q)
    binding.sparse_attn(d.q, d.kv, d.attn_sink, d.topk_idxs, d.softmax_scale, out=out)
    torch.cuda.synchronize()
    ws = binding.workspace_for(8, 1, 128, 512, d.topk_idxs.shape[-1])
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            binding.sparse_attn(d.q, d.kv, d.attn_sink, d.topk_idxs, d.softmax_scale, out=out, workspace=ws)
    for seed in (21, 22):
        nxt = workloads.v4_ratio128_decode(seed=seed, B=8)
        d.topk_idxs.copy_(nxt.topk_idxs.cuda())
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, nxt.topk_idxs, inp.softmax_scale)
        assert_close(out, ref, f"graph replay seed {seed}")


# ------------------------------------------------------------- full-size workloads

def test_v4_ratio4_decode_all_tokens():
    inp = workloads.v4_ratio4_decode()
    assert_close(run_gpu(inp), run_oracle(inp), "ratio-4 decode")


def test_v4_ratio128_decode_all_tokens():
    inp = workloads.v4_ratio128_decode()
    assert_close(run_gpu(inp), run_oracle(inp), "ratio-128 decode")


def test_v4_prefill_all_tokens():
    # every one of the 4096 tokens against the oracle (multithreaded over
    # tokens: about 15 s on 16 host cores)
    inp = workloads.v4_prefill()
    assert_close(run_gpu(inp)[0], run_oracle(inp)[0], "prefill (all tokens)")


# ------------------------------------------------------- wide-range partial logits

@pytest.mark.parametrize("pattern", ["dominant", "outlier", "cancel"])
@pytest.mark.parametrize("ns", [0, 3, 5])
def test_wide_range_partial_logits(pattern, ns):
    # At D = 512 the two halves of the head dim live on two CTAs, whose
    # partial logits are added before the softmax.  These inputs put huge
    # partials (positive, negative, or two that cancel) next to the keys that
    # carry the weight: any lossy step in that exchange shows up here.
    # ns = 0: the library's plan; 3: six CTAs combining in-cluster; 5: the
    # separate combine kernel.
    inp = workloads.wide_range_attn(pattern, B=2, S=2, T=2048, K=1152, seed=len(pattern) * 10 + ns)
    assert_close(run_gpu(inp, num_splits=ns), run_oracle(inp), f"wide range ({pattern}) splits={ns}")


# ------------------------------------------------------- per-token topk_length

def run_gpu_len(inp, lens, num_splits=0):
    d = inp.to("cuda")
    L = torch.as_tensor(lens, dtype=torch.int32).cuda().contiguous()
    o = binding.sparse_attn(d.q, d.kv, d.attn_sink, d.topk_idxs, d.softmax_scale, num_splits=num_splits,
                            topk_length=L)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    return o


@pytest.mark.parametrize("H,D,K,T,ns", [
    (128, 512, 1152, 2000, 0),
    (128, 512, 700, 1500, 2),     # fused split combine
    (100, 512, 700, 1500, 3),
    (128, 512, 1152, 2000, 5),    # separate combine kernel
    (16, 256, 300, 500, 1),
    (64, 64, 200, 300, 2),
])
def test_topk_length_random(H, D, K, T, ns):
    inp = workloads.random_attn(3, 2, H, D, T, K, p_invalid=0.1, seed=H + K + ns + 7)
    rng = np.random.default_rng(K + ns)
    lens = rng.integers(-2, K + 6, size=(3, 2)).astype(np.int32)
    lens[0, 0], lens[0, 1], lens[1, 0] = 0, 1, K        # the edge values
    ref = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, topk_length=lens)
    assert_close(run_gpu_len(inp, lens, ns), ref, f"topk_length H={H} D={D} K={K} splits={ns}")


def test_topk_length_cuts_through_valid_slots():
    inp = workloads.random_attn(2, 2, 128, 512, 800, 640, p_invalid=0.0, seed=77)
    lens = np.array([[50, 64], [65, 639]], dtype=np.int32)   # inside a tile, at and just past a boundary
    for ns in (1, 2):
        ref = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, topk_length=lens)
        assert_close(run_gpu_len(inp, lens, ns), ref, f"cut lengths splits={ns}")


def test_topk_length_of_the_valid_prefix_matches_minus_one_padding_exactly():
    # ratio-4 decode: each token's slots are a valid prefix then -1; passing
    # the prefix length runs the same tiles with the same arithmetic
    inp = workloads.v4_ratio4_decode()
    T = inp.kv.shape[1]
    valid = (inp.topk_idxs >= 0) & (inp.topk_idxs < T)
    lens = valid.sum(-1).to(torch.int32).numpy()
    # the workload's valid slots form a prefix of every token's slot list
    prefix = valid.int().cumprod(-1).sum(-1).numpy()
    assert (prefix == lens).all()
    a = run_gpu(inp)
    b = run_gpu_len(inp, lens)
    assert torch.equal(a, b)


@pytest.mark.parametrize("H,D,K,T,ns", [
    (128, 512, 2049, 4000, 0),     # one slot more than a work unit holds: at least 2 splits
    (128, 512, 5000, 8000, 1),     # an explicit single split is raised to the 3 the slots need
    (64, 64, 8192, 9000, 0),       # 4 units' worth of slots, separate or in-cluster combine
    (128, 256, 4100, 5000, 9),     # more splits than a cluster holds
])
def test_long_slot_lists_force_splits(H, D, K, T, ns):
    inp = workloads.random_attn(1, 2, H, D, T, K, p_invalid=0.1, seed=K + ns)
    assert_close(run_gpu(inp, num_splits=ns), run_oracle(inp), f"H={H} D={D} K={K} splits={ns}")
