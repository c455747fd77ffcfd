"""GPU parity of sparse_attn over two kv sources (the extra kv source of the
V4 kernels: a second cache with its own slot list and length, joining each
token's softmax after the main slots) against the CPU oracle.

Bar, element by element: |gpu - oracle| <= 1e-2 + 1e-2 |oracle|."""

import numpy as np
import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import binding, workloads

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


def assert_close(gpu, ref, what=""):
    g = gpu.float().cpu().numpy().astype(np.float64)
    bad = np.abs(g - ref) > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first at {tuple(i)}: "
                             f"gpu={g[tuple(i)]} oracle={ref[tuple(i)]}")


def _lens(B, S, K, seed):
    g = torch.Generator().manual_seed(seed)
    L = torch.randint(-2, K + 3, (B, S), generator=g, dtype=torch.int32)
    L.view(-1)[0] = K            # one full list, one empty one
    if L.numel() > 1:
        L.view(-1)[1] = 0
    return L


def _run(main, extra, len1=None, len2=None, ns=0, fp8=False):
    kv, kv2 = (main.kv8, extra.kv8) if fp8 else (main.kv, extra.kv)
    c = lambda t: None if t is None else t.cuda().contiguous()
    o = binding.sparse_attn_extra(main.q.cuda(), kv.cuda(), main.attn_sink.cuda(), main.topk_idxs.cuda(), kv2.cuda(),
                                  extra.topk_idxs.cuda(), main.softmax_scale, topk_length=c(len1),
                                  extra_topk_length=c(len2), num_splits=ns)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    f = oracle.sparse_attn_fp8 if fp8 else oracle.sparse_attn
    kw = dict(extra_kv8=extra.kv8) if fp8 else dict(extra_kv=extra.kv)
    want = f(main.q, kv, main.attn_sink, main.topk_idxs, main.softmax_scale, topk_length=len1,
             extra_idxs=extra.topk_idxs, extra_length=len2, **kw)
    return o, want


@pytest.mark.parametrize("H,D,T,K,T2,K2,ns", [
    (128, 512, 900, 600, 500, 300, 0),     # the plan
    (128, 512, 900, 640, 400, 130, 2),     # splits combined in the cluster
    (128, 512, 3000, 1152, 800, 128, 5),   # separate combine kernel
    (16, 256, 400, 200, 300, 70, 0),       # one CTA per unit
    (8, 64, 300, 65, 200, 100, 3),
])
def test_random_two_sources(H, D, T, K, T2, K2, ns):
    main = workloads.random_attn(2, 2, H, D, T, K, p_invalid=0.1, seed=H + K + ns)
    extra = workloads.random_attn(2, 2, H, D, T2, K2, p_invalid=0.1, seed=H + K2 + ns + 1)
    len1, len2 = _lens(2, 2, K, 3), _lens(2, 2, K2, 4)
    o, want = _run(main, extra, len1, len2, ns)
    assert_close(o, want, f"H={H} D={D} K={K} K2={K2} splits={ns}")
    o, want = _run(main, extra, ns=ns)          # no lengths
    assert_close(o, want, f"no lengths, H={H} D={D}")


def test_only_extra_slots_and_empty_extra_list():
    main = workloads.random_attn(2, 3, 128, 512, 600, 200, p_invalid=0.2, seed=5)
    extra = workloads.random_attn(2, 3, 128, 512, 300, 150, p_invalid=0.2, seed=6)
    none = workloads.AttnInputs(main.q, main.kv, main.attn_sink, torch.full_like(main.topk_idxs, -1),
                                main.softmax_scale)
    o, want = _run(none, extra)
    assert_close(o, want, "main list all -1")
    zero = torch.zeros((2, 3), dtype=torch.int32)
    o, want = _run(main, extra, len2=zero)
    assert_close(o, want, "empty extra lists")


def test_v4_window_as_the_extra_source():
    # a V4-shaped decode step: the indexer's compressed picks in the main
    # list, the 128 sliding-window rows from a separate window cache
    dec = workloads.v4_ratio4_decode(B=8)
    T = dec.kv.shape[1]
    main = workloads.AttnInputs(dec.q, dec.kv[:, 128:].contiguous(), dec.attn_sink,
                                torch.where(dec.topk_idxs[..., 128:] >= 0, dec.topk_idxs[..., 128:] - 128,
                                            torch.full_like(dec.topk_idxs[..., 128:], -1)).contiguous(),
                                dec.softmax_scale)
    extra = workloads.AttnInputs(dec.q, dec.kv[:, :128].contiguous(), dec.attn_sink,
                                 dec.topk_idxs[..., :128].contiguous(), dec.softmax_scale)
    o, want = _run(main, extra)
    assert_close(o, want, "window rows as the extra source")
    # equal, as a whole, to the one-source call over the original layout
    one = binding.sparse_attn(dec.q.cuda(), dec.kv.cuda(), dec.attn_sink.cuda(), dec.topk_idxs.cuda(),
                              dec.softmax_scale)
    torch.cuda.synchronize()
    assert_close(one, want, "one source, same rows")


@pytest.mark.parametrize("ns", [0, 2])
def test_fp8_two_sources(ns):
    main = workloads.random_attn_fp8(2, 2, 128, 700, 400, p_invalid=0.1, seed=31 + ns)
    extra = workloads.random_attn_fp8(2, 2, 128, 301, 150, p_invalid=0.1, seed=32 + ns)   # odd T2: odd rows
    len1, len2 = _lens(2, 2, 400, 8), _lens(2, 2, 150, 9)
    o, want = _run(main, extra, len1, len2, ns, fp8=True)
    assert_close(o, want, f"fp8 two sources splits={ns}")


@pytest.mark.parametrize("ns", [0, 2])
def test_fp8_even_last_rows_of_both_sources(ns):
    # both sources end on a row with an even index (B*T and B*T2 odd); the
    # bytes after each hold NaN patterns, and several slots of every token of
    # the last request pick each source's last row
    B, S, H = 3, 2, 128
    main = workloads.random_attn_fp8(B, S, H, 101, 96, p_invalid=0.1, seed=61 + ns)
    extra = workloads.random_attn_fp8(B, S, H, 51, 40, p_invalid=0.1, seed=62 + ns)
    i1, i2 = main.topk_idxs.clone(), extra.topk_idxs.clone()
    i1[B - 1, :, :5] = 100
    i2[B - 1, :, 3:9] = 50
    main.topk_idxs, extra.topk_idxs = i1, i2

    def poisoned(kv8):
        n = kv8.shape[0] * kv8.shape[1]
        big = torch.full((n + 2, 584), 0xFF, dtype=torch.uint8, device="cuda")
        big[:n] = kv8.reshape(n, 584).cuda()
        return big[:n].view(kv8.shape)

    o = binding.sparse_attn_extra(main.q.cuda(), poisoned(main.kv8), main.attn_sink.cuda(), i1.cuda(),
                                  poisoned(extra.kv8), i2.cuda(), main.softmax_scale, num_splits=ns)
    torch.cuda.synchronize()
    assert binding.sa_device_error(True) == 0
    want = oracle.sparse_attn_fp8(main.q, main.kv8, main.attn_sink, i1, main.softmax_scale,
                                  extra_idxs=i2, extra_kv8=extra.kv8)
    assert_close(o, want, f"fp8 even last rows splits={ns}")
