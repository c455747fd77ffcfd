"""Seeded synthetic inputs for top-k sparse attention and the top-k mask.

This module only draws random numbers and lays out index patterns; it holds
none of the method's arithmetic, so the CPU oracle (tests) and the CUDA
library both consume exactly the same bits from it.  Everything is generated
on the CPU with ``torch.Generator().manual_seed(seed)`` and may be moved to a
device afterwards.

Shapes and index structure follow the workloads the pages describe for
DeepSeek V4 ("DeepSeek V4 源码剖析, 第5章", §5.1 and §5.14): q [B,S,128,512]
bf16, a shared kv [B,T,512] bf16, a float32 sink per head, int32 top-k indices
[B,S,K] with -1 for an invalid slot, K = 128 window rows + 1024 indexer picks
on a ratio-4 layer, 128 window rows + every compressed row on a ratio-128
layer.  The kv layout puts the window rows first and the compressed rows after
them; indexer picks are random distinct compressed rows (unsorted, as a top-k
selection returns them).  The mask workload follows the vLLM PR 52217/48770
pages: per-request top-k rows scattered into a padded uint32 bitmask.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

SENTINEL_U32 = 0xA5A5A5A5


@dataclass
class AttnInputs:
    q: torch.Tensor          # [B,S,H,D] bf16
    kv: torch.Tensor         # [B,T,D]   bf16
    attn_sink: torch.Tensor  # [H]       float32
    topk_idxs: torch.Tensor  # [B,S,K]   int32, -1 = invalid slot
    softmax_scale: float
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, S, H, D = self.q.shape
        return dict(B=B, S=S, H=H, D=D, T=self.kv.shape[1], K=self.topk_idxs.shape[-1])

    def to(self, device):
        return AttnInputs(self.q.to(device), self.kv.to(device), self.attn_sink.to(device),
                          self.topk_idxs.to(device), self.softmax_scale, self.name, dict(self.meta))


@dataclass
class MaskInputs:
    topk: torch.Tensor       # [sum q_len, K] int32
    cu_q_lens: torch.Tensor  # [B+1] int32
    batch: int
    max_q_len: int
    max_key_len: int
    key_starts: torch.Tensor | None  # [B] int32 or None
    name: str = ""

    def to(self, device):
        return MaskInputs(self.topk.to(device), self.cu_q_lens.to(device), self.batch, self.max_q_len,
                          self.max_key_len, None if self.key_starts is None else self.key_starts.to(device),
                          self.name)


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def _randn_bf16(shape, g) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _distinct(n_pool: int, k: int, g) -> torch.Tensor:
    """k distinct values of [0, n_pool) in random order."""
    return torch.randperm(n_pool, generator=g)[:k].to(torch.int32)


def random_attn(B, S, H, D, T, K, *, p_invalid=0.1, seed=0, distinct=True, scale=None) -> AttnInputs:
    """Generic case: per token, K slots drawn from [0,T) (distinct when K<=T),
    each set to -1 with probability p_invalid."""
    g = _gen(seed)
    q = _randn_bf16((B, S, H, D), g)
    kv = _randn_bf16((B, T, D), g)
    sink = torch.randn((H,), generator=g, dtype=torch.float32)
    idx = torch.empty((B, S, K), dtype=torch.int32)
    for b in range(B):
        for s in range(S):
            if distinct and K <= T:
                idx[b, s] = _distinct(T, K, g)
            else:
                idx[b, s] = torch.randint(0, max(T, 1), (K,), generator=g, dtype=torch.int32)
    if p_invalid > 0:
        drop = torch.rand((B, S, K), generator=g) < p_invalid
        idx[drop] = -1
    return AttnInputs(q, kv, sink, idx, float(scale if scale is not None else D ** -0.5),
                      name=f"random B={B} S={S} H={H} D={D} T={T} K={K}")


def wide_range_attn(pattern: str, B=2, S=2, H=128, D=512, T=2048, K=1152, *, p_invalid=0.05,
                    seed=0) -> AttnInputs:
    """Inputs whose partial logits span a wide range (stress cases for any
    lossy step between the two head-dim halves of a row).  Every token takes
    one or two "special" rows in each block of 32 slots, ordinary rows in the
    other slots; the picks of a token are distinct.

    pattern "dominant": q drawn x30; the special rows (the first T/8 of kv)
      are drawn x8, every other row x0.01, so one or two keys of each block
      carry huge positive or negative logits next to near-zero ones.
    pattern "outlier": every head's q is u + N(0, 0.25) for one shared
      direction u ~ N(0,1)^D; the special rows (the first T/16) are -c.u with
      c uniform in [100, 300] (huge negative logits, weight ~0), the others
      N(0,1): the keys that carry the weight sit next to an outlier.
    pattern "cancel": q as for "outlier"; the special rows are
      c.[u_0, -u_1] + N(0,1), u_0 / u_1 the two halves of u: the partial
      logit over each half of the head dim is huge and the two nearly cancel,
      so the sum is ordinary and those keys carry weight.
    """
    g = _gen(seed)
    n_special = T // 8 if pattern == "dominant" else T // 16
    if pattern == "dominant":
        q = (torch.randn((B, S, H, D), generator=g) * 30).to(torch.bfloat16)
        base = torch.randn((B, T, D), generator=g)
        mult = torch.full((T, 1), 0.01)
        mult[:n_special] = 8.0
        kv = (base * mult).to(torch.bfloat16)
    elif pattern in ("outlier", "cancel"):
        u = torch.randn((D,), generator=g)
        q = (u + 0.5 * torch.randn((B, S, H, D), generator=g)).to(torch.bfloat16)
        kv32 = torch.randn((B, T, D), generator=g)
        c = 100 + 200 * torch.rand((B, n_special, 1), generator=g)
        if pattern == "outlier":
            kv32[:, :n_special] = -c * u
        else:
            signed = torch.cat([u[: D // 2], -u[D // 2:]])
            kv32[:, :n_special] = c * signed + kv32[:, :n_special]
        kv = kv32.to(torch.bfloat16)
    else:
        raise ValueError(pattern)
    sink = torch.randn((H,), generator=g, dtype=torch.float32)
    idx = torch.empty((B, S, K), dtype=torch.int32)
    j = torch.arange(K)
    special = j % 32 == 3
    if pattern == "dominant":
        special |= j % 32 == 20
    n_sp = int(special.sum())
    assert n_sp <= n_special and K - n_sp <= T - n_special, "not enough distinct rows"
    for b in range(B):
        for s in range(S):
            row = torch.empty((K,), dtype=torch.int32)
            row[special] = _distinct(n_special, n_sp, g)
            row[~special] = n_special + _distinct(T - n_special, K - n_sp, g)
            idx[b, s] = row
    if p_invalid > 0:
        idx[torch.rand((B, S, K), generator=g) < p_invalid] = -1
    return AttnInputs(q, kv, sink, idx, D ** -0.5,
                      name=f"wide-range ({pattern}) B={B} S={S} H={H} D={D} T={T} K={K}")


FP8_ROW_BYTES = 584      # one row of the FP8 kv cache: 448 codes + 64 bf16 + 8 scale bytes


@dataclass
class Fp8AttnInputs:
    q: torch.Tensor          # [B,S,H,512] bf16
    kv8: torch.Tensor        # [B,T,584]   uint8 rows of the FP8 kv format
    attn_sink: torch.Tensor  # [H]         float32
    topk_idxs: torch.Tensor  # [B,S,K]     int32, -1 = invalid slot
    softmax_scale: float
    name: str = ""
    meta: dict = field(default_factory=dict)

    def to(self, device):
        return Fp8AttnInputs(self.q.to(device), self.kv8.to(device), self.attn_sink.to(device),
                             self.topk_idxs.to(device), self.softmax_scale, self.name, dict(self.meta))


def fp8_kv_rows(B: int, T: int, g) -> torch.Tensor:
    """uint8 [B, T, 584]: bytes 0..447 are E4M3 codes with a random sign,
    exponent field uniform in [4, 9] and mantissa uniform in [0, 7] (so never
    the NaN pattern; magnitudes 2^-3 .. 7.5); bytes 448..575 are 64 N(0,1)
    bf16 values, little-endian; bytes 576..582 are E8M0 scale bytes uniform in
    [124, 127] (2^-3 .. 1); byte 583 is zero padding."""
    sign = torch.randint(0, 2, (B, T, 448), generator=g, dtype=torch.int32)
    expo = torch.randint(4, 10, (B, T, 448), generator=g, dtype=torch.int32)
    mant = torch.randint(0, 8, (B, T, 448), generator=g, dtype=torch.int32)
    codes = (sign * 128 + expo * 8 + mant).to(torch.uint8)
    rope = _randn_bf16((B, T, 64), g).contiguous().view(torch.uint8).reshape(B, T, 128)
    scales = torch.randint(124, 128, (B, T, 7), generator=g, dtype=torch.int32).to(torch.uint8)
    pad = torch.zeros((B, T, 1), dtype=torch.uint8)
    return torch.cat([codes, rope, scales, pad], dim=-1).contiguous()


def random_attn_fp8(B, S, H, T, K, *, p_invalid=0.1, seed=0) -> Fp8AttnInputs:
    """random_attn's index pattern over an FP8 kv cache (D = 512)."""
    g = _gen(seed)
    q = _randn_bf16((B, S, H, 512), g)
    kv8 = fp8_kv_rows(B, T, g)
    sink = torch.randn((H,), generator=g, dtype=torch.float32)
    idx = torch.empty((B, S, K), dtype=torch.int32)
    for b in range(B):
        for s in range(S):
            idx[b, s] = _distinct(T, K, g) if K <= T else torch.randint(0, T, (K,), generator=g, dtype=torch.int32)
    if p_invalid > 0:
        idx[torch.rand((B, S, K), generator=g) < p_invalid] = -1
    return Fp8AttnInputs(q, kv8, sink, idx, 512 ** -0.5, name=f"random fp8 B={B} S={S} H={H} T={T} K={K}")


def v4_ratio4_decode_fp8(seed=1006, B=32, H=128, window=128, topk=1024, ratio=4, long_ctx=65536, short_lo=128,
                         short_hi=4096) -> Fp8AttnInputs:
    """The ratio-4 decode batch (same context mix and slot structure as
    v4_ratio4_decode) over an FP8 kv cache of 584-byte rows."""
    g = _gen(seed)
    n_comp = long_ctx // ratio
    T = window + n_comp
    K = window + topk
    q = _randn_bf16((B, 1, H, 512), g)
    kv8 = fp8_kv_rows(B, T, g)
    sink = torch.randn((H,), generator=g, dtype=torch.float32)
    idx = torch.full((B, 1, K), -1, dtype=torch.int32)
    ctx = []
    for b in range(B):
        L = long_ctx if b >= B // 2 else int(torch.randint(short_lo, short_hi, (1,), generator=g))
        ctx.append(L)
        nw = min(window, L)
        idx[b, 0, :nw] = torch.arange(nw, dtype=torch.int32)
        pool = L // ratio
        nc = min(topk, pool)
        idx[b, 0, window:window + nc] = window + _distinct(pool, nc, g)
    return Fp8AttnInputs(q, kv8, sink, idx, 512 ** -0.5,
                         name=f"V4 ratio-4 decode, FP8 kv B={B} S=1 H={H} D=512 T={T} K={K}",
                         meta=dict(context=ctx))


def tiny(seed=1000) -> AttnInputs:
    """B=1,S=4,H=8,D=64,T=256,K=64: the first 64 of a random permutation of
    [0,256) per token, each slot -1 with probability 0.1, scale = 1/8."""
    out = random_attn(1, 4, 8, 64, 256, 64, p_invalid=0.1, seed=seed)
    out.name = "tiny B=1 S=4 H=8 D=64 T=256 K=64"
    return out


def v4_ratio4_decode(seed=1001, B=32, H=128, D=512, window=128, topk=1024, ratio=4,
                     long_ctx=65536, short_lo=128, short_hi=4096) -> AttnInputs:
    """Ratio-4 decode: T = window + long_ctx/ratio; K = window + topk.
    Context L_b = long_ctx for the upper half of the batch and uniform in
    [short_lo, short_hi) for the lower half.  Slots: the window rows
    0..window-1 (valid for min(window, L_b)), then min(topk, L_b//ratio)
    distinct random compressed rows from [window, window + L_b//ratio),
    then -1."""
    g = _gen(seed)
    n_comp = long_ctx // ratio
    T = window + n_comp
    K = window + topk
    q = _randn_bf16((B, 1, H, D), g)
    kv = _randn_bf16((B, T, D), g)
    sink = torch.randn((H,), generator=g, dtype=torch.float32)
    idx = torch.full((B, 1, K), -1, dtype=torch.int32)
    ctx = []
    for b in range(B):
        L = long_ctx if b >= B // 2 else int(torch.randint(short_lo, short_hi, (1,), generator=g))
        ctx.append(L)
        nw = min(window, L)
        idx[b, 0, :nw] = torch.arange(nw, dtype=torch.int32)
        pool = L // ratio
        nc = min(topk, pool)
        idx[b, 0, window:window + nc] = window + _distinct(pool, nc, g)
    return AttnInputs(q, kv, sink, idx, D ** -0.5,
                      name=f"V4 ratio-4 decode B={B} S=1 H={H} D={D} T={T} K={K}",
                      meta=dict(context=ctx))


def v4_prefill(seed=1002, S=4096, H=128, D=512, window=128, topk=1024, ratio=4) -> AttnInputs:
    """Prefill of one S-token chunk: kv rows 0..S-1 are the chunk's own
    tokens, rows S..S+S/ratio-1 the compressed rows.  Token s: window slots
    s-window+1..s ascending (-1 when negative), then min(topk, (s+1)//ratio)
    distinct random compressed rows from [S, S + (s+1)//ratio), then -1."""
    g = _gen(seed)
    n_comp = S // ratio
    T = S + n_comp
    K = window + topk
    q = _randn_bf16((1, S, H, D), g)
    kv = _randn_bf16((1, T, D), g)
    sink = torch.randn((H,), generator=g, dtype=torch.float32)
    idx = torch.full((1, S, K), -1, dtype=torch.int32)
    win = torch.arange(-window + 1, 1, dtype=torch.int32)
    for s in range(S):
        w = win + s
        idx[0, s, :window] = torch.where(w >= 0, w, torch.full_like(w, -1))
        pool = (s + 1) // ratio
        nc = min(topk, pool)
        if nc > 0:
            idx[0, s, window:window + nc] = S + _distinct(pool, nc, g)
    return AttnInputs(q, kv, sink, idx, D ** -0.5, name=f"V4 prefill B=1 S={S} H={H} D={D} T={T} K={K}")


def v4_ratio128_decode(seed=1003, B=64, H=128, D=512, window=128, end_pos=65536, ratio=128) -> AttnInputs:
    """Ratio-128 decode: K = T = window + end_pos/ratio.  Even b: every slot
    valid, idx = 0..K-1.  Odd b: end_b uniform in [1, end_pos); the first
    min(window, end_b) window slots and the first end_b//ratio compressed
    slots are valid, the rest -1."""
    g = _gen(seed)
    n_comp = end_pos // ratio
    T = window + n_comp
    K = T
    q = _randn_bf16((B, 1, H, D), g)
    kv = _randn_bf16((B, T, D), g)
    sink = torch.randn((H,), generator=g, dtype=torch.float32)
    idx = torch.full((B, 1, K), -1, dtype=torch.int32)
    ends = []
    for b in range(B):
        if b % 2 == 0:
            idx[b, 0] = torch.arange(K, dtype=torch.int32)
            ends.append(end_pos)
            continue
        e = int(torch.randint(1, end_pos, (1,), generator=g))
        ends.append(e)
        nw = min(window, e)
        idx[b, 0, :nw] = torch.arange(nw, dtype=torch.int32)
        nc = e // ratio
        idx[b, 0, window:window + nc] = window + torch.arange(nc, dtype=torch.int32)
    return AttnInputs(q, kv, sink, idx, D ** -0.5,
                      name=f"V4 ratio-128 decode B={B} S=1 H={H} D={D} T={T} K={K}", meta=dict(end=ends))


def topk_mask(seed=1004, B=4, Q=2048, max_key_len=8193, K=2048, key_starts=(0, 1, 31, 8192),
              q_lens=None) -> MaskInputs:
    """Mask build: request b has q_lens[b] (default Q) query rows; row q sits at
    absolute position p = max_key_len - Q + q and holds K distinct uniform
    indices from [0, p] (fewer candidates than K: -1 fill)."""
    g = _gen(seed)
    q_lens = [Q] * B if q_lens is None else list(q_lens)
    cu = [0]
    rows = []
    for b in range(B):
        for qi in range(q_lens[b]):
            p = max_key_len - Q + qi
            n = min(K, p + 1)
            r = torch.full((K,), -1, dtype=torch.int32)
            if n > 0:
                r[:n] = _distinct(p + 1, n, g)
            rows.append(r)
        cu.append(cu[-1] + q_lens[b])
    topk = torch.stack(rows) if rows else torch.empty((0, K), dtype=torch.int32)
    ks = None if key_starts is None else torch.tensor(list(key_starts)[:B], dtype=torch.int32)
    return MaskInputs(topk, torch.tensor(cu, dtype=torch.int32), B, max(q_lens) if q_lens else 0,
                      max_key_len, ks, name=f"topk mask B={B} Q={Q} keys={max_key_len} K={K}")


CONFIGS = {
    "tiny": tiny,
    "v4_ratio4_decode": v4_ratio4_decode,
    "v4_prefill": v4_prefill,
    "v4_ratio128_decode": v4_ratio128_decode,
}


def count_valid(idx: torch.Tensor, T: int) -> int:
    """Number of slots with 0 <= idx < T (the work a sparse kernel must do)."""
    return int(((idx >= 0) & (idx < T)).sum())


def ceil_div(a: int, b: int) -> int:
    return -(-a // b) if b else 0


def nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()
