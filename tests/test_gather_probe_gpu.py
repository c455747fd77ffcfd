"""The random-row gather probe (sa_probe_row_gather): it runs to completion on
every documented row-part size, with index values outside the table read as
row 0, leaves the device error word clear, and reports a rate that a copy
engine can physically reach (so the timed launch really moved the bytes)."""

import pytest
import torch

from deepseek_top_sparse_gb300 import binding

pytestmark = pytest.mark.gpu


def _rate_gbs(table, row_bytes, part, idx, ctas, tiles, flush):
    flush.zero_()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st = torch.cuda.current_stream()
    a.record(st)
    binding.probe_row_gather(table, row_bytes, part, idx, ctas, tiles)
    b.record(st)
    b.synchronize()
    return ctas * tiles * 32768 / (a.elapsed_time(b) * 1e-3) * 1e-9


@pytest.mark.parametrize("part", [16, 512, 1024, 32768])
def test_probe_runs_and_reports_a_physical_rate(part):
    dev = torch.device("cuda")
    row_bytes = max(1024, part)
    rows = (256 << 20) // row_bytes                       # 256 MB: more than L2
    table = torch.zeros(rows * row_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    tiles = 8
    n = ctas * tiles * (32768 // part)
    g = torch.Generator(device=dev).manual_seed(5)
    idx = torch.randint(0, rows, (n,), generator=g, device=dev, dtype=torch.int32)
    idx[::97] = -1                                        # outside the table: row 0
    idx[::89] = rows + 3
    rate = _rate_gbs(table, row_bytes, part, idx, ctas, tiles, flush)
    assert binding.sa_device_error(True) == 0
    assert 1.0 < rate < 20000.0                           # GB/s: moved, and no faster than the SMs can load


def test_probe_rejects_a_mismatched_index_count():
    dev = torch.device("cuda")
    table = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    idx = torch.zeros(10, dtype=torch.int32, device=dev)
    with pytest.raises(ValueError):
        binding.probe_row_gather(table, 1024, 1024, idx, 1, 1)
