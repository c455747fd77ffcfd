"""Host-only checks of the C ABI: the library builds and loads, exports every
function include/*.h declares, and the host-side paths (shape query, argument
validation) behave as documented.  No kernel is launched here."""

import ctypes
import glob
import os
import re
import subprocess

import pytest

import oracle
from deepseek_top_sparse_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(sa_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_three_operations():
    names = _declared_functions()
    for required in ("sa_sparse_attn_fwd", "sa_topk_mask_shape", "sa_build_topk_mask"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib_path = binding.load().__dict__.get("_name") or binding.library_path()
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing
    lib = binding.load()
    for n in _declared_functions():
        assert hasattr(lib, n)


def test_binding_exposes_c_names():
    for n in binding.EXPORTS:
        assert callable(getattr(binding, n))
    assert set(binding.EXPORTS) == set(_declared_functions())


def test_selftest_validates_its_limit_on_the_host():
    # argument checks happen before any device work (no GPU needed)
    assert binding.sa_selftest_wait_timeout(0) == -1
    assert binding.sa_selftest_wait_timeout(-5) == -1
    assert binding.sa_selftest_wait_drain(0, 1000)[0] == -1
    assert binding.sa_selftest_wait_drain(1025, 1000)[0] == -1
    assert binding.sa_selftest_wait_drain(4, 0)[0] == -1
    assert binding.sa_selftest_wait_drain(4, 1 << 29)[0] == -1


def test_status_strings():
    assert binding.sa_status_string(0) == "SA_OK"
    assert binding.sa_status_string(4) == "SA_ERR_WORKSPACE"
    assert binding.sa_status_string(99) == "SA_ERR_UNKNOWN"


def test_mask_shape_matches_oracle_and_golden():
    for b, q, k, r in [(2, 129, 129, 0), (2, 129, 129, 1), (1, 1, 129, 0), (4, 2048, 8193, 1), (3, 128, 32, 0),
                       (3, 129, 33, 0), (1, 257, 96, 1), (1, 513, 97, 1), (2, 0, 10, 0), (0, 5, 0, 1)]:
        assert binding.sa_topk_mask_shape(b, q, k, r) == oracle.topk_mask_shape(b, q, k, bool(r))
    assert binding.sa_topk_mask_shape(2, 129, 129, 0) == (2, 256, 8)


def test_mask_shape_rejects_negative_and_null():
    with pytest.raises(binding.SAError):
        binding.sa_topk_mask_shape(-1, 1, 1, 0)
    assert binding.load().sa_topk_mask_shape(1, 1, 1, 0, None) == 1  # SA_ERR_INVALID_ARG


def _fwd(**over):
    args = dict(q=16, kv=16, attn_sink=16, topk_idxs=16, softmax_scale=0.125, o=32, B=1, S=1, H=8, D=64, T=10,
                K=4, num_splits=0, workspace=None, workspace_bytes=0, stream=None)
    args.update(over)
    return binding.sa_sparse_attn_fwd_splits(**args)


def test_attn_validation_happens_before_any_device_work():
    # none of these reach the device: sizes, pointers and alignment are checked first
    assert _fwd(D=96) == 2                # SA_ERR_SHAPE: D not in {64,128,256,512}
    assert _fwd(H=129) == 2               # more than 128 heads
    assert _fwd(K=0) == 2
    assert _fwd(T=0) == 2
    assert _fwd(B=1 << 20, T=1 << 12) == 2  # B*T >= 2^31
    assert _fwd(B=1 << 17, S=1 << 7, H=128, T=1) == 2  # B*S*H >= 2^31
    assert _fwd(B=-1) == 1
    assert _fwd(softmax_scale=float("nan")) == 1
    assert _fwd(num_splits=65) == 1
    assert _fwd(q=None) == 1
    assert _fwd(o=None) == 1
    assert _fwd(q=8) == 3                 # q not 16-byte aligned
    assert _fwd(o=40) == 3
    assert _fwd(topk_idxs=2) == 3
    assert _fwd(B=0) == 0                 # nothing to do
    assert _fwd(S=0) == 0


def test_topk_length_entry_validates_like_the_others():
    f = binding.sa_sparse_attn_fwd_topk_length
    base = dict(q=16, kv=16, attn_sink=16, topk_idxs=16, topk_length=16, softmax_scale=0.125, o=32, B=1, S=1,
                H=8, D=64, T=10, K=4, num_splits=0, workspace=None, workspace_bytes=0, stream=None)
    assert f(**dict(base, topk_length=2)) == 3      # not 4-byte aligned
    assert f(**dict(base, D=96)) == 2
    assert f(**dict(base, q=None)) == 1
    assert f(**dict(base, B=0)) == 0


def test_mask_validation_happens_before_any_device_work():
    f = binding.sa_build_topk_mask
    shape = binding.sa_topk_mask_shape(1, 1, 129, 0)
    assert f(16, 1, 16, 1, 1, 129, 2, None, 16, (1, 128, 4), None) == 2   # wrong shape
    no_reserve = binding.sa_topk_mask_shape(1, 1, 128, 0)                # (1, 128, 4)
    assert f(16, 1, 16, 1, 1, 128, 2, 16, 16, no_reserve, None) == 2      # key_starts needs a reserved word
    assert f(16, 1, 16, -1, 1, 129, 2, None, 16, shape, None) == 1
    assert f(16, 1, None, 1, 1, 129, 2, None, 16, shape, None) == 1       # cu_q_lens NULL
    assert f(16, 1, 16, 1, 1, 129, 2, None, 8, shape, None) == 3          # mask not 16-byte aligned
    assert f(16, 0, 16, 1, 0, 129, 2, None, 16, binding.sa_topk_mask_shape(1, 0, 129, 0), None) == 0  # empty
    assert binding.load().sa_build_topk_mask(16, 1, 16, 1, 1, 129, 2, None, 16, None, None) == 1


def test_workspace_size_is_zero_without_splits_and_for_bad_sizes():
    assert binding.sa_sparse_attn_workspace_size(1, 1, 8, 96, 4, 1) == 0
    assert binding.sa_sparse_attn_workspace_size(1, 1, 8, 64, 4, 1) == 0
    # explicit split counts size the partials: tokens*splits*H*D fp32 (256-aligned) + tokens*splits*H fp32
    n = binding.sa_sparse_attn_workspace_size(2, 3, 8, 64, 256, 2)
    o_bytes = 2 * 3 * 2 * 8 * 64 * 4
    assert n == (o_bytes + 255) // 256 * 256 + 2 * 3 * 2 * 8 * 4
    # never more splits than 64-slot tiles
    assert binding.sa_sparse_attn_workspace_size(1, 1, 8, 64, 64, 8) == 0


def test_masked_dense_entry_validates_before_any_device_work():
    f = binding.sa_masked_dense_attn_fwd
    base = dict(q=16, kv=16, attn_sink=16, mask=16, mask_rows=4, mask_words=8, key_start_word=0,
                softmax_scale=0.125, o=32, B=1, S=2, H=8, D=64, T=200, num_splits=0, workspace=None,
                workspace_bytes=0, stream=None)
    assert f(**dict(base, mask_words=6)) == 2         # rows must be whole 16-byte vectors
    assert f(**dict(base, mask_words=0)) == 2
    assert f(**dict(base, mask_rows=1)) == 2          # fewer mask rows than queries
    assert f(**dict(base, D=96)) == 2
    assert f(**dict(base, T=0)) == 2
    assert f(**dict(base, key_start_word=2)) == 1
    assert f(**dict(base, softmax_scale=float("inf"))) == 1
    assert f(**dict(base, mask=None)) == 1
    assert f(**dict(base, mask=8)) == 3               # mask not 16-byte aligned
    assert f(**dict(base, q=24)) == 3
    assert f(**dict(base, B=0)) == 0
    # an explicit split count gives sparse_attn's workspace layout for that many splits
    assert binding.sa_masked_dense_attn_workspace_size(2, 3, 8, 64, 256, 2) == \
        binding.sa_sparse_attn_workspace_size(2, 3, 8, 64, 256, 2)
    assert binding.sa_masked_dense_attn_workspace_size(1, 1, 8, 96, 256, 2) == 0


def test_fp8_entry_validates_before_any_device_work():
    f = binding.sa_sparse_attn_fwd_fp8
    base = dict(q=16, kv_fp8=16, attn_sink=16, topk_idxs=16, topk_length=None, softmax_scale=0.05, o=32, B=1, S=1,
                H=128, T=10, K=4, num_splits=0, workspace=None, workspace_bytes=0, stream=None)
    assert f(**dict(base, H=129)) == 2
    assert f(**dict(base, K=0)) == 2
    assert f(**dict(base, T=0)) == 2
    assert f(**dict(base, kv_fp8=None)) == 1
    assert f(**dict(base, kv_fp8=8)) == 3          # not 16-byte aligned
    assert f(**dict(base, topk_length=2)) == 3
    assert f(**dict(base, softmax_scale=float("nan"))) == 1
    assert f(**dict(base, B=0)) == 0
    assert binding.sa_sparse_attn_fp8_launch_count(1, 1, 128, 0, 0) == 0


def test_mask_chunk_rows_plan():
    # the whole mask when it fits the 64 MiB cap; else the largest window of
    # 256-row multiples (or 128 rows) whose mask fits
    f = binding.sa_topk_mask_chunk_rows
    assert f(4, 2048, 8193, 1, 0) == 2048                    # 8.5 MB: global mask
    assert f(4, 2048, 8193, 1, 1 << 20) == 128               # 256 rows would be 1.06 MB
    assert f(4, 2048, 8193, 1, 100000) == 0                  # not even 128 rows fit
    assert f(1, 100000, 1 << 20, 0, 0) == 512                # 32 MiB per 256 rows of 2^15 words
    assert f(2, 300, 700, 0, 60000) == 256
    assert f(0, 300, 700, 0, 0) == 0


def test_window_entries_validate_before_any_device_work():
    f = binding.sa_masked_dense_attn_fwd_window
    base = dict(q=16, kv=16, attn_sink=16, mask=16, mask_rows=128, mask_words=8, key_start_word=0, key_ends=None,
                softmax_scale=0.1, o=32, B=1, S_total=10, q0=4, S=4, H=8, D=64, T=200, num_splits=0,
                workspace=None, workspace_bytes=0, stream=None)
    assert f(**dict(base, q0=7)) == 2                        # q0 + S > S_total
    assert f(**dict(base, q0=-1)) == 1
    assert f(**dict(base, key_ends=2)) == 3
    assert f(**dict(base, B=0)) == 0
    g = binding.sa_build_topk_mask_window
    shape = binding.sa_topk_mask_shape(2, 16, 100, 0)
    assert g(16, 4, 16, 2, -1, 16, 100, 8, None, None, 16, shape, None) == 1
    assert g(16, 4, 16, 2, 0, 16, 100, 8, None, None, 16, (2, 128, 8), None) == 2   # wrong shape
    assert g(16, 4, 16, 2, 0, 16, 100, 8, None, 6, 16, shape, None) == 3             # key_ends misaligned


def test_windowed_call_checks_every_window_before_launching():
    f = binding.sa_topk_masked_attn_fwd
    base = dict(q=16, kv=16, attn_sink=16, topk=16, topk_rows=300, cu_q_lens=16, key_starts=None, key_ends=None,
                softmax_scale=0.1, o=32, B=2, max_q_len=300, H=8, D=64, T=700, max_key_len=700, K=50, cap_bytes=30000,
                mask_buf=256, mask_buf_bytes=1 << 20, workspace=None, workspace_bytes=0, stream=None)
    assert f(**dict(base, T=0)) == 2                    # the consumer's shape error, nothing launched
    assert f(**dict(base, D=96)) == 2
    assert f(**dict(base, q=8)) == 3                    # q misaligned
    assert f(**dict(base, cap_bytes=1000)) == 2         # no window fits the cap
    assert f(**dict(base, mask_buf_bytes=100)) == 4     # mask buffer smaller than one window
    assert f(**dict(base, B=0)) == 0


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    # no fallback: with the CUDA library absent the binding raises instead of
    # computing anything some other way
    from deepseek_top_sparse_gb300 import build as sa_build

    monkeypatch.setattr(sa_build, "LIB", str(tmp_path / "libsa.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        binding.load(build_if_missing=False)


def test_extra_source_arguments_are_checked_on_the_host():
    # argument checks happen before any device work (no GPU needed)
    buf = ctypes.create_string_buffer(64)
    base = ctypes.addressof(buf)
    a16 = (base + 15) // 16 * 16
    args = dict(q=a16, kv=a16, attn_sink=a16, topk_idxs=a16, topk_length=None, extra_kv=a16, extra_topk_idxs=a16,
                extra_topk_length=None, softmax_scale=0.1, o=a16, B=1, S=1, H=8, D=64, T=4, K=2, T2=4, K2=2,
                num_splits=0, workspace=None, workspace_bytes=0, stream=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return binding.sa_status_string(binding.sa_sparse_attn_fwd_extra(*a.values()))

    assert call(K2=-1) == "SA_ERR_INVALID_ARG"
    assert call(K=0, K2=0) == "SA_ERR_SHAPE"
    assert call(K2=3, T2=0) == "SA_ERR_SHAPE"
    assert call(extra_kv=None) == "SA_ERR_INVALID_ARG"
    assert call(extra_kv=a16 + 4) == "SA_ERR_ALIGNMENT"
    assert call(extra_topk_idxs=a16 + 2) == "SA_ERR_ALIGNMENT"
    assert call(B=1 << 20, T=1 << 11, T2=1 << 11) == "SA_ERR_SHAPE"


def test_gather_probe_validates_before_any_device_work():
    f = binding.sa_probe_row_gather
    ok = dict(table=4096, rows=1024, row_bytes=1024, part_bytes=512, idx=8192, ctas=4, tiles=2, stream=None)
    bad = [dict(table=None), dict(idx=None), dict(rows=0), dict(rows=1 << 31), dict(ctas=0), dict(ctas=65536),
           dict(tiles=0), dict(tiles=(1 << 20) + 1), dict(part_bytes=8), dict(part_bytes=768),
           dict(part_bytes=65536), dict(row_bytes=256), dict(row_bytes=1032 - 1)]
    for b in bad:
        args = dict(ok, **b)
        assert f(**args) == 1, b                              # SA_ERR_INVALID_ARG
    assert f(**dict(ok, table=4096 + 8)) == 3                 # SA_ERR_ALIGNMENT
