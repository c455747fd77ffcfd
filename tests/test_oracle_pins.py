"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped sink
term, the scale applied to the sink, a wrong sign, the wrong batch's kv, a
transposed operand, an off-by-one word or bit) fails at least one of them:

* values printed by the pages (tests/golden/*.txt, each with its source);
* closed forms: K = 1 (a logistic of logit - sink), identical kv rows,
  q = 0 (uniform weights);
* a library routine: torch's scaled_dot_product_attention in float64 with an
  additive mask, where the sink is an extra key whose value row is zero;
* invariants: slot permutation, moving invalid slots, sink limits;
* brute force: the mask decoded bit by bit against Python sets.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from deepseek_top_sparse_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


# ---------------------------------------------------------------- mask shape

def _golden_shapes():
    out = []
    with open(os.path.join(GOLDEN, "mask_shape.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("->")
            out.append((tuple(int(v) for v in lhs.split()), tuple(int(v) for v in rhs.split())))
    return out


@pytest.mark.parametrize("args,want", _golden_shapes())
def test_mask_shape_golden(args, want):
    b, q, k, r = args
    assert oracle.topk_mask_shape(b, q, k, bool(r)) == want


def test_mask_shape_rows_are_16_byte_aligned():
    for q in (0, 1, 127, 128, 129, 255, 256, 257, 4097):
        for k in (0, 1, 31, 32, 33, 127, 128, 129, 8193):
            for r in (False, True):
                _, rows, words = oracle.topk_mask_shape(3, q, k, r)
                assert words % 4 == 0 and words * 32 >= k + 32 * r
                assert words < (-(-k // 32) + r) + 4
                assert rows >= q and rows % 128 == 0


# ---------------------------------------------------------------- mask build

def _golden_example():
    kv = {}
    with open(os.path.join(GOLDEN, "mask_build_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *vals = line.split()
                kv[key] = [int(v) for v in vals]
    return kv


def test_mask_build_worked_example():
    ex = _golden_example()
    B, Q, KEYS = ex["batch"][0], ex["max_q_len"][0], ex["max_key_len"][0]
    shape = oracle.topk_mask_shape(B, Q, KEYS)
    out = np.zeros(shape, dtype=np.uint32)
    topk = np.array([ex["topk"]], dtype=np.int32)
    m = oracle.build_topk_mask(topk, np.array([0, 1], np.int32), B, Q, KEYS, out=out)
    assert m[:B, :Q].shape == (1, 1, 8)
    assert m[0, 0].tolist() == ex["row"]


def _decode_row(words, n_keys):
    return {k for k in range(n_keys) if (int(words[k >> 5]) >> (k & 31)) & 1}


@pytest.mark.parametrize("seed", range(6))
def test_mask_build_brute_force(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    q_lens = [int(rng.integers(0, 6)) for _ in range(B)]
    max_q = max(q_lens + [1]) + int(rng.integers(0, 2))
    keys = int(rng.integers(1, 200))
    K = int(rng.integers(1, 40))
    reserve = bool(rng.integers(0, 2))
    rows = sum(q_lens)
    # indices include -1, out-of-range values and duplicates on purpose
    topk = rng.integers(-3, keys + 5, size=(rows, K)).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ks = rng.integers(-2**31, 2**31 - 1, size=B).astype(np.int32) if reserve else None
    shape = oracle.topk_mask_shape(B, max_q, keys, reserve)
    out = np.full(shape, workloads.SENTINEL_U32, dtype=np.uint32)
    m = oracle.build_topk_mask(topk, cu, B, max_q, keys, key_starts=ks, out=out)
    n_live = -(-keys // 32)
    for b in range(B):
        for q in range(shape[1]):
            row = m[b, q]
            if q < q_lens[b]:
                want = {int(v) for v in topk[cu[b] + q] if 0 <= v < keys}
                assert _decode_row(row, keys) == want
                # bits beyond max_key_len inside the last live word stay clear
                assert all(((int(row[k >> 5]) >> (k & 31)) & 1) == 0 for k in range(keys, n_live * 32))
                tail = row[n_live:]
            else:
                tail = row  # rows past q_len are never written
            for wi, w in enumerate(tail):
                absolute = (n_live + wi) if q < q_lens[b] else wi
                if reserve and q == 0 and absolute == shape[2] - 1:
                    assert np.uint32(w) == np.uint32(ks[b]).astype(np.uint32)
                else:
                    assert w == workloads.SENTINEL_U32, (b, q, absolute)


def test_mask_build_rejects_wrong_shape():
    topk = np.zeros((1, 2), np.int32)
    bad = np.zeros((1, 128, 4), dtype=np.uint32)  # 129 keys need 8 words
    with pytest.raises(ValueError):
        oracle.build_topk_mask(topk, np.array([0, 1], np.int32), 1, 1, 129, out=bad)


# ---------------------------------------------------------------- attention

def _sdpa_reference(inp):
    """torch SDPA (float64, CPU) over the gathered rows of each token, the sink
    realised as one more key with additive logit attn_sink[h] and a zero value
    row, invalid slots masked with -inf."""
    q = inp.q.double()
    kv = inp.kv.double()
    idx = inp.topk_idxs.long()
    B, S, H, D = q.shape
    T, K = kv.shape[1], idx.shape[-1]
    out = torch.zeros(B, S, H, D, dtype=torch.float64)
    for b in range(B):
        for s in range(S):
            sel = idx[b, s]
            valid = (sel >= 0) & (sel < T)
            rows = torch.zeros(K + 1, D, dtype=torch.float64)
            rows[:K][valid] = kv[b, sel[valid]]
            bias = torch.full((H, 1, K + 1), 0.0, dtype=torch.float64)
            bias[:, 0, :K][:, ~valid] = -math.inf
            bias[:, 0, K] = inp.attn_sink.double()
            qh = q[b, s].unsqueeze(1)  # [H,1,D]
            k = rows.unsqueeze(0).expand(H, K + 1, D)
            v = k.clone()
            v[:, K] = 0.0
            out[b, s] = torch.nn.functional.scaled_dot_product_attention(
                qh, k, v, attn_mask=bias, scale=inp.softmax_scale)[:, 0]
    return out.numpy()


def _run(inp, **kw):
    return oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, **kw)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attn_matches_library_sdpa_with_sink(seed):
    inp = workloads.random_attn(2, 3, 4, 32, 40, 12, p_invalid=0.2, seed=seed, distinct=(seed != 2))
    # seed 2 draws indices with repeats: a repeated slot counts once per occurrence
    got = _run(inp)
    want = _sdpa_reference(inp)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_attn_uses_own_batch_kv_and_out_of_range_is_invalid():
    inp = workloads.random_attn(3, 2, 2, 16, 20, 8, p_invalid=0.0, seed=5)
    inp.topk_idxs[0, 0, 0] = 20      # == T: out of range, treated like -1
    inp.topk_idxs[1, 1, 3] = 1 << 30
    inp.topk_idxs[2, 0, 5] = -7
    np.testing.assert_allclose(_run(inp), _sdpa_reference(inp), rtol=1e-10, atol=1e-12)


def test_attn_k1_closed_form():
    # one valid slot: weights are [sigmoid(x - sink), 1 - that]; o = w * row
    D, H = 8, 3
    q = _bf(torch.tensor([0.5, -1.0, 2.0, 0.25, 1.5, -0.75, 0.0, 1.0]).repeat(H, 1)).reshape(1, 1, H, D)
    row = _bf(torch.tensor([1.0, 0.5, -0.5, 2.0, -1.0, 0.25, 3.0, -2.0]))
    kv = row.reshape(1, 1, D)
    sink = torch.tensor([-1.0, 0.0, 2.5], dtype=torch.float32)
    idx = torch.zeros(1, 1, 1, dtype=torch.int32)
    scale = 0.375
    o = oracle.sparse_attn(q, kv, sink, idx, scale)
    x = scale * float((q[0, 0, 0].double() * row.double()).sum())
    for h in range(H):
        w = 1.0 / (1.0 + math.exp(-(x - float(sink[h]))))
        np.testing.assert_allclose(o[0, 0, h], w * row.double().numpy(), rtol=1e-14, atol=1e-15)


def test_attn_identical_rows_closed_form():
    # n valid copies of one row v: o = n e^x / (n e^x + e^sink) * v
    D, H, K, n = 16, 2, 10, 7
    g = torch.Generator().manual_seed(3)
    v = _bf(torch.randn(D, generator=g))
    q = _bf(torch.randn(1, 1, H, D, generator=g))
    kv = v.reshape(1, 1, D).repeat(1, 5, 1)
    idx = torch.full((1, 1, K), -1, dtype=torch.int32)
    idx[0, 0, [0, 2, 3, 5, 6, 8, 9]] = torch.tensor([0, 1, 2, 3, 4, 0, 1], dtype=torch.int32)
    sink = torch.tensor([0.3, -2.0], dtype=torch.float32)
    scale = D ** -0.5
    o = oracle.sparse_attn(q, kv, sink, idx, scale)
    for h in range(H):
        x = scale * float((q[0, 0, h].double() * v.double()).sum())
        w = n * math.exp(x) / (n * math.exp(x) + math.exp(float(sink[h])))
        np.testing.assert_allclose(o[0, 0, h], w * v.double().numpy(), rtol=1e-13, atol=1e-15)


def test_attn_zero_query_gives_uniform_weights():
    inp = workloads.random_attn(1, 1, 2, 8, 30, 9, p_invalid=0.3, seed=11)
    inp.q.zero_()
    sel = inp.topk_idxs[0, 0]
    valid = sel[(sel >= 0)].long()
    rows = inp.kv[0, valid].double().sum(0).numpy()
    o = _run(inp)
    for h in range(2):
        want = rows / (len(valid) + math.exp(float(inp.attn_sink[h])))
        np.testing.assert_allclose(o[0, 0, h], want, rtol=1e-13, atol=1e-15)


def test_attn_all_invalid_gives_zero():
    inp = workloads.random_attn(1, 2, 3, 8, 10, 5, p_invalid=0.0, seed=2)
    inp.topk_idxs.fill_(-1)
    assert np.all(_run(inp) == 0.0)
    inp.attn_sink[:] = -math.inf  # no sink and no key: zero, not NaN
    assert np.all(_run(inp) == 0.0)


def test_attn_sink_limits():
    inp = workloads.random_attn(1, 2, 3, 8, 10, 5, p_invalid=0.2, seed=4)
    inp.attn_sink[:] = math.inf
    assert np.all(_run(inp) == 0.0)
    inp.attn_sink[:] = -math.inf
    got = _run(inp)
    # sink = -inf is plain softmax attention over the valid slots
    want = _sdpa_reference(inp)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
    # and the sink lowers every weight when finite (sum w_j < 1)
    inp.attn_sink[:] = 0.0
    assert not np.allclose(_run(inp), got)


def test_attn_invariant_to_slot_order_and_invalid_position():
    inp = workloads.random_attn(1, 3, 4, 16, 64, 24, p_invalid=0.25, seed=9)
    base = _run(inp)
    perm = torch.randperm(24, generator=torch.Generator().manual_seed(1))
    inp2 = workloads.AttnInputs(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs[..., perm].contiguous(),
                                inp.softmax_scale)
    np.testing.assert_allclose(_run(inp2), base, rtol=1e-12, atol=1e-14)
    # padding with extra -1 slots changes nothing
    pad = torch.full((1, 3, 40), -1, dtype=torch.int32)
    inp3 = workloads.AttnInputs(inp.q, inp.kv, inp.attn_sink, torch.cat([pad, inp.topk_idxs], -1),
                                inp.softmax_scale)
    np.testing.assert_allclose(_run(inp3), base, rtol=1e-12, atol=1e-14)


def test_attn_token_subset_matches_full():
    inp = workloads.random_attn(2, 5, 2, 16, 32, 8, seed=12)
    full = _run(inp)
    tok = np.array([7, 0, 3], dtype=np.int64)
    sub = _run(inp, tokens=tok)
    for i, t in enumerate(tok):
        np.testing.assert_array_equal(sub[i], full[t // 5, t % 5])


# ---------------------------------------------------------------- mask <-> attention

def test_masked_dense_equals_sparse_with_oracle_mask():
    inp = workloads.random_attn(2, 4, 3, 16, 70, 20, p_invalid=0.15, seed=21)
    B, S = 2, 4
    cu = np.arange(0, B * S + 1, S, dtype=np.int32)
    topk = inp.topk_idxs.reshape(B * S, -1).numpy()
    m = oracle.build_topk_mask(topk, cu, B, S, 70)
    dense = oracle.masked_dense_attn(inp.q, inp.kv, inp.attn_sink, m, inp.softmax_scale)
    np.testing.assert_allclose(dense, _run(inp), rtol=1e-12, atol=1e-14)


def test_masked_dense_key_offset_reads_absolute_positions():
    # a context chunk kv[start:] with a mask over absolute key positions: the
    # consumer adds key_start before the bit test
    inp = workloads.random_attn(1, 2, 2, 8, 50, 12, p_invalid=0.0, seed=31)
    start = 17
    topk = inp.topk_idxs.reshape(2, -1).numpy()
    m = oracle.build_topk_mask(topk, np.array([0, 2], np.int32), 1, 2, 50)
    chunk = inp.kv[:, start:].contiguous()
    got = oracle.masked_dense_attn(inp.q, chunk, inp.attn_sink, m, inp.softmax_scale, key_offset=[start])
    shifted = torch.where(inp.topk_idxs >= start, inp.topk_idxs - start, torch.full_like(inp.topk_idxs, -1))
    want = oracle.sparse_attn(inp.q, chunk, inp.attn_sink, shifted, inp.softmax_scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_masked_dense_offset_form_never_reads_the_reserved_word():
    # key_starts = -1 puts 0xFFFFFFFF into the reserved last word of row 0;
    # a chunk of 128 keys at position -1 reaches mask positions 96..126 of
    # that word.  The offset form admits exactly the row's indices shifted by
    # the start: sparse attention over idx + 1, nothing from the reserved word.
    inp = workloads.random_attn(1, 2, 2, 8, 128, 20, p_invalid=0.1, seed=41)
    idx = inp.topk_idxs.clone()
    idx[idx >= 64] = -1                          # the mask covers 64 keys
    m = oracle.build_topk_mask(idx.reshape(2, -1).numpy(), np.array([0, 2], np.int32), 1, 2, 64,
                               key_starts=np.array([-1], np.int32))
    assert m.shape == (1, 128, 4) and m[0, 0, 3] == 0xFFFFFFFF
    got = oracle.masked_dense_attn(inp.q, inp.kv, inp.attn_sink, m, inp.softmax_scale, key_offset=[-1])
    shifted = torch.where(idx >= 0, idx + 1, idx)
    want = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, shifted, inp.softmax_scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_tiny_workload_shape_and_structure():
    inp = workloads.tiny()
    assert inp.shape == dict(B=1, S=4, H=8, D=64, T=256, K=64)
    idx = inp.topk_idxs
    for s in range(4):
        v = idx[0, s][idx[0, s] >= 0]
        assert len(set(v.tolist())) == len(v)
    assert 0 < int((idx < 0).sum()) < 64
    assert inp.softmax_scale == 0.125


# --------------------------------------------------- per-token topk_length
# A slot counts only below the token's length (clamped to [0, K]); these pins
# tie the length path to the -1 path, to the closed forms and to the clamps.

def _rand_case(seed, B=2, S=3, H=4, D=32, T=40, K=24, p_invalid=0.1):
    return workloads.random_attn(B, S, H, D, T, K, p_invalid=p_invalid, seed=seed)


@pytest.mark.parametrize("seed", range(3))
def test_topk_length_k_equals_no_length(seed):
    inp = _rand_case(200 + seed)
    B, S, K = inp.topk_idxs.shape
    full = np.full((B, S), K, dtype=np.int32)
    a = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    b = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, topk_length=full)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("seed", range(3))
def test_topk_length_equals_minus_one_padding(seed):
    inp = _rand_case(210 + seed)
    B, S, K = inp.topk_idxs.shape
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, K + 1, size=(B, S)).astype(np.int32)
    padded = inp.topk_idxs.clone()
    for b in range(B):
        for s in range(S):
            padded[b, s, lens[b, s]:] = -1
    a = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, topk_length=lens)
    b_ = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, padded, inp.softmax_scale)
    assert np.array_equal(a, b_)


def test_topk_length_zero_gives_zero_and_one_gives_sigmoid_closed_form():
    inp = _rand_case(220, p_invalid=0.0)
    B, S, K = inp.topk_idxs.shape
    zero = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale,
                              topk_length=np.zeros((B, S), np.int32))
    assert not zero.any()
    one = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale,
                             topk_length=np.ones((B, S), np.int32))
    q = inp.q.double().numpy()
    kv = inp.kv.double().numpy()
    sink = inp.attn_sink.double().numpy()
    for b in range(B):
        for s in range(S):
            row = kv[b, int(inp.topk_idxs[b, s, 0])]
            x = inp.softmax_scale * q[b, s] @ row                      # [H]
            w = 1.0 / (1.0 + np.exp(sink - x))                         # sigmoid(x - sink)
            np.testing.assert_allclose(one[b, s], w[:, None] * row[None, :], rtol=1e-12, atol=1e-14)


def test_topk_length_is_clamped_to_zero_and_k():
    inp = _rand_case(230)
    B, S, K = inp.topk_idxs.shape
    neg = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale,
                             topk_length=np.full((B, S), -7, np.int32))
    assert not neg.any()
    big = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale,
                             topk_length=np.full((B, S), K + 100, np.int32))
    assert np.array_equal(big, oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, inp.topk_idxs, inp.softmax_scale))


# ---------------------------------------------------------------- FP8 kv rows (V4 format)

def test_e4m3_decode_matches_the_format_definition():
    # OCP 8-bit floating point, E4M3: bias 7, 3 mantissa bits, subnormals at
    # exponent 0, no infinities, S.1111.111 = NaN, largest finite 448
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
             0x40: 2.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0, 0x77: 240.0, 0x30: 0.5}
    for code, want in cases.items():
        assert oracle.e4m3_to_float(code) == want, hex(code)
    assert math.copysign(1.0, oracle.e4m3_to_float(0x80)) == -1.0
    assert math.isnan(oracle.e4m3_to_float(0x7F)) and math.isnan(oracle.e4m3_to_float(0xFF))


def test_e4m3_decode_matches_torch_float8_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_to_float(c) for c in range(256)])
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(lib))
    np.testing.assert_array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])


def test_e8m0_decode():
    assert oracle.e8m0_to_float(127) == 1.0
    assert oracle.e8m0_to_float(128) == 2.0
    assert oracle.e8m0_to_float(0) == 2.0 ** -127
    assert oracle.e8m0_to_float(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_to_float(255))


def _hand_row():
    row = np.zeros(oracle.FP8_ROW_BYTES, dtype=np.uint8)
    row[576:583] = 127                     # every tile scale 2^0 ...
    row[0] = 0x38                          # dim 0: 1.0
    row[63] = 0xC0                         # dim 63: -2.0 (tile 0)
    row[64] = 0x38                         # dim 64: 1.0 x 2^2 (tile 1)
    row[577] = 129
    row[447] = 0x30                        # dim 447: 0.5 x 2^-1 (tile 6)
    row[582] = 126
    row[448:450] = (0x80, 0x3F)            # dim 448: bf16 1.0, little-endian
    row[574:576] = (0x00, 0xC0)            # dim 511: bf16 -2.0
    row[583] = 0xFF                        # padding byte: ignored
    want = np.zeros(512)
    want[0], want[63], want[64], want[447], want[448], want[511] = 1.0, -2.0, 4.0, 0.25, 1.0, -2.0
    return row, want


def test_fp8_row_layout_hand_built():
    row, want = _hand_row()
    np.testing.assert_array_equal(oracle.decode_kv_fp8(row[None, :])[0], want)


def test_fp8_attention_single_slot_closed_form():
    # K = 1: o = sigmoid(x - sink) * kv_row, x = scale * q . kv_row
    row, kv_row = _hand_row()
    g = torch.Generator().manual_seed(41)
    q = torch.randn(1, 1, 3, 512, generator=g).to(torch.bfloat16)
    sink = torch.tensor([0.3, -1.0, 2.0])
    kv8 = torch.from_numpy(np.stack([np.zeros_like(row), row])[None])     # [1, 2, 584]
    idx = torch.tensor([[[1]]], dtype=torch.int32)
    got = oracle.sparse_attn_fp8(q, kv8, sink, idx, 0.1)
    qd = q.double().numpy()[0, 0]
    for h in range(3):
        x = 0.1 * float(qd[h] @ kv_row)
        w = 1.0 / (1.0 + math.exp(-(x - float(sink[h]))))
        np.testing.assert_allclose(got[0, 0, h], w * kv_row, rtol=1e-14, atol=1e-300)


def test_fp8_attention_equals_bf16_attention_on_the_decoded_rows():
    # the generated codes and scales decode to values that bf16 holds exactly,
    # so attention over the FP8 rows must equal attention over those values
    inp = workloads.random_attn_fp8(2, 3, 8, 90, 40, p_invalid=0.2, seed=43)
    dec = oracle.decode_kv_fp8(inp.kv8)
    kv_bf16 = torch.from_numpy(dec).to(torch.bfloat16)
    np.testing.assert_array_equal(kv_bf16.double().numpy(), dec)       # exact in bf16
    want = oracle.sparse_attn(inp.q, kv_bf16, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    got = oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale)
    np.testing.assert_array_equal(got, want)
    lens = torch.tensor([[5, 40, 0], [17, -3, 60]], dtype=torch.int32)
    np.testing.assert_array_equal(
        oracle.sparse_attn_fp8(inp.q, inp.kv8, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, topk_length=lens),
        oracle.sparse_attn(inp.q, kv_bf16, inp.attn_sink, inp.topk_idxs, inp.softmax_scale, topk_length=lens))


# ---------------------------------------------------------------- mask windows and live ends

def _mask_case(seed, B=3, max_q=300, keys=700, K=40):
    rng = np.random.default_rng(seed)
    q_lens = [int(rng.integers(0, max_q + 1)) for _ in range(B)]
    topk = rng.integers(-3, keys + 3, size=(sum(q_lens), K)).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return rng, q_lens, topk, cu


def test_mask_window_of_every_query_is_the_whole_mask():
    _, q_lens, topk, cu = _mask_case(61)
    full = oracle.build_topk_mask(topk, cu, 3, 300, 700, key_starts=np.array([5, 0, 9], np.int32))
    win = oracle.build_topk_mask_window(topk, cu, 3, 0, 300, 700, key_starts=np.array([5, 0, 9], np.int32))
    np.testing.assert_array_equal(win, full)


def test_mask_windows_tile_the_whole_mask():
    # windows of 128 queries, stacked, give the live rows of the whole mask;
    # each window carries the reserved word in its own row 0
    _, q_lens, topk, cu = _mask_case(62)
    ks = np.array([7, 1, 2], np.int32)
    full = oracle.build_topk_mask(topk, cu, 3, 300, 700, key_starts=ks)
    W = full.shape[2]
    for q0 in range(0, 300, 128):
        win = oracle.build_topk_mask_window(topk, cu, 3, q0, 128, 700, key_starts=ks)
        assert win.shape == (3, 128, W)
        for b in range(3):
            assert win[b, 0, W - 1] == np.uint32(ks[b])
            for i in range(128):
                q = q0 + i
                if q < q_lens[b]:
                    lw = (700 + 31) // 32
                    np.testing.assert_array_equal(win[b, i, :lw], full[b, q, :lw])


def test_mask_live_end_brute_force():
    # only the words below each request's live end are written; they hold the
    # bits of the indices below the end; every other word keeps the sentinel
    rng, q_lens, topk, cu = _mask_case(63, keys=500)
    ends = np.array([0, 77, 1000], np.int32)          # empty, ragged, past max_key_len
    shape = oracle.topk_mask_shape(3, 300, 500)
    out = np.full(shape, 0xA5A5A5A5, dtype=np.uint32)
    oracle.build_topk_mask_window(topk, cu, 3, 0, 300, 500, key_ends=ends, out=out)
    for b in range(3):
        end = min(int(ends[b]), 500)
        lw = (end + 31) // 32
        for q in range(shape[1]):
            row = out[b, q]
            if q >= q_lens[b]:
                assert (row == 0xA5A5A5A5).all()
                continue
            want = set(int(k) for k in topk[cu[b] + q] if 0 <= k < end)
            got = {w * 32 + j for w in range(lw) for j in range(32) if (int(row[w]) >> j) & 1}
            assert got == want
            assert (row[lw:] == 0xA5A5A5A5).all()


def test_masked_dense_live_end_drops_the_keys_past_it():
    inp = workloads.random_attn(2, 3, 4, 16, 90, 30, p_invalid=0.1, seed=64)
    cu = np.array([0, 3, 6], np.int32)
    m = oracle.build_topk_mask(inp.topk_idxs.reshape(6, -1).numpy(), cu, 2, 3, 90)
    ends = np.array([41, 90], np.int64)
    got = oracle.masked_dense_attn(inp.q, inp.kv, inp.attn_sink, m, inp.softmax_scale, key_ends=ends)
    idx = inp.topk_idxs.clone()
    idx[0][idx[0] >= 41] = -1
    want = oracle.sparse_attn(inp.q, inp.kv, inp.attn_sink, idx, inp.softmax_scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_masked_dense_key_offset_and_live_end_together():
    # kv[b] is the chunk of mask positions start .. start + T - 1; the live end
    # is in mask positions, so a chunk key t counts iff t + start < end
    inp = workloads.random_attn(1, 3, 2, 8, 60, 15, p_invalid=0.0, seed=65)
    start, end = 11, 40
    topk = inp.topk_idxs.reshape(3, -1).numpy()
    m = oracle.build_topk_mask(topk, np.array([0, 3], np.int32), 1, 3, 60)
    chunk = inp.kv[:, start:].contiguous()
    got = oracle.masked_dense_attn(inp.q, chunk, inp.attn_sink, m, inp.softmax_scale, key_offset=[start],
                                   key_ends=[end])
    keep = (inp.topk_idxs >= start) & (inp.topk_idxs < end)
    shifted = torch.where(keep, inp.topk_idxs - start, torch.full_like(inp.topk_idxs, -1))
    want = oracle.sparse_attn(inp.q, chunk, inp.attn_sink, shifted, inp.softmax_scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------- extra kv source (R25)

def _extra_case(seed, B=2, S=3, H=4, D=32, T=40, K=24, T2=30, K2=20, p_invalid=0.15, fp8=False):
    """A main and an extra source with their own slot lists and lengths."""
    g = torch.Generator().manual_seed(seed)
    if fp8:
        main = workloads.random_attn_fp8(B, S, H, T, K, p_invalid=p_invalid, seed=seed)
        extra = workloads.random_attn_fp8(B, S, H, T2, K2, p_invalid=p_invalid, seed=seed + 1)
    else:
        main = workloads.random_attn(B, S, H, D, T, K, p_invalid=p_invalid, seed=seed)
        extra = workloads.random_attn(B, S, H, D, T2, K2, p_invalid=p_invalid, seed=seed + 1)
    len1 = torch.randint(-2, K + 3, (B, S), generator=g, dtype=torch.int32)
    len2 = torch.randint(-2, K2 + 3, (B, S), generator=g, dtype=torch.int32)
    return main, extra, len1, len2


def _concatenated(main_kv, extra_kv, idx, idx2, len1, len2):
    """The same problem as one source: kv rows [main | extra] per batch, slots
    [main | extra] per token with the extra indices shifted past the main rows
    and every slot at or past its list's length (or out of its source's range)
    set to -1."""
    T, T2 = main_kv.shape[1], extra_kv.shape[1]
    kv = torch.cat([main_kv, extra_kv], dim=1)
    K, K2 = idx.shape[-1], idx2.shape[-1]
    a = idx.clone().long()
    a[(a < 0) | (a >= T) | (torch.arange(K) >= len1.clamp(0, K).long().unsqueeze(-1))] = -1
    e = idx2.clone().long()
    bad = (e < 0) | (e >= T2) | (torch.arange(K2) >= len2.clamp(0, K2).long().unsqueeze(-1))
    e = torch.where(bad, torch.full_like(e, -1), e + T)
    return kv, torch.cat([a, e], dim=-1).to(torch.int32)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_extra_source_equals_one_concatenated_source(seed):
    main, extra, len1, len2 = _extra_case(seed)
    got = oracle.sparse_attn(main.q, main.kv, main.attn_sink, main.topk_idxs, main.softmax_scale, topk_length=len1,
                             extra_kv=extra.kv, extra_idxs=extra.topk_idxs, extra_length=len2)
    kv, idx = _concatenated(main.kv, extra.kv, main.topk_idxs, extra.topk_idxs, len1, len2)
    want = oracle.sparse_attn(main.q, kv, main.attn_sink, idx, main.softmax_scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_extra_source_matches_library_sdpa_on_the_union():
    main, extra, len1, len2 = _extra_case(7)
    kv, idx = _concatenated(main.kv, extra.kv, main.topk_idxs, extra.topk_idxs, len1, len2)
    union = workloads.AttnInputs(main.q, kv, main.attn_sink, idx, main.softmax_scale)
    got = oracle.sparse_attn(main.q, main.kv, main.attn_sink, main.topk_idxs, main.softmax_scale, topk_length=len1,
                             extra_kv=extra.kv, extra_idxs=extra.topk_idxs, extra_length=len2)
    np.testing.assert_allclose(got, _sdpa_reference(union), rtol=1e-10, atol=1e-12)


def test_extra_source_alone_and_swapped_roles():
    main, extra, len1, len2 = _extra_case(11, p_invalid=0.0)
    none = torch.full_like(main.topk_idxs, -1)
    alone = oracle.sparse_attn(main.q, main.kv, main.attn_sink, none, main.softmax_scale,
                               extra_kv=extra.kv, extra_idxs=extra.topk_idxs)
    want = oracle.sparse_attn(main.q, extra.kv, main.attn_sink, extra.topk_idxs, main.softmax_scale)
    np.testing.assert_allclose(alone, want, rtol=1e-12, atol=1e-12)
    # the two sources are interchangeable: one softmax over both slot lists
    a = oracle.sparse_attn(main.q, main.kv, main.attn_sink, main.topk_idxs, main.softmax_scale, topk_length=len1,
                           extra_kv=extra.kv, extra_idxs=extra.topk_idxs, extra_length=len2)
    b = oracle.sparse_attn(main.q, extra.kv, main.attn_sink, extra.topk_idxs, main.softmax_scale, topk_length=len2,
                           extra_kv=main.kv, extra_idxs=main.topk_idxs, extra_length=len1)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_extra_source_empty_list_changes_nothing():
    main, extra, len1, _ = _extra_case(13)
    zero = torch.zeros_like(len1)
    got = oracle.sparse_attn(main.q, main.kv, main.attn_sink, main.topk_idxs, main.softmax_scale, topk_length=len1,
                             extra_kv=extra.kv, extra_idxs=extra.topk_idxs, extra_length=zero)
    want = oracle.sparse_attn(main.q, main.kv, main.attn_sink, main.topk_idxs, main.softmax_scale, topk_length=len1)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("seed", [21, 22])
def test_extra_fp8_source_equals_one_concatenated_source(seed):
    main, extra, len1, len2 = _extra_case(seed, H=4, T=30, K=20, T2=25, K2=18, fp8=True)
    got = oracle.sparse_attn_fp8(main.q, main.kv8, main.attn_sink, main.topk_idxs, main.softmax_scale,
                                 topk_length=len1, extra_kv8=extra.kv8, extra_idxs=extra.topk_idxs, extra_length=len2)
    kv8 = torch.cat([main.kv8, extra.kv8], dim=1)
    _, idx = _concatenated(main.kv8, extra.kv8, main.topk_idxs, extra.topk_idxs, len1, len2)
    want = oracle.sparse_attn_fp8(main.q, kv8, main.attn_sink, idx, main.softmax_scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
