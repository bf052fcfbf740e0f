"""cp_measure_stream_read and cp_measure_record_read: the read kernels that
measure the host link (zero-copy from pinned memory, streaming and record by
record) and HBM reads for the rooflines."""
import pytest
import torch

import trellis_row_decode_gb300 as cp

pytestmark = pytest.mark.gpu


def test_stream_read_device_and_pinned_host():
    dev = torch.ones(1 << 24, dtype=torch.uint8, device="cuda")
    host = torch.ones(1 << 24, dtype=torch.uint8).pin_memory()
    for buf in (dev, host, dev[: 4096 + 16]):
        cp.measure_stream_read(buf)
    torch.cuda.synchronize()
    assert bool((dev == 1).all()) and bool((host == 1).all())       # nothing written


def test_stream_read_rejects_unusable_buffers():
    L = cp.lib()
    dev = torch.ones(4096, dtype=torch.uint8, device="cuda")
    assert L.cp_measure_stream_read(None, 4096, None) == cp.CP_ERR_INVALID_ARG
    assert L.cp_measure_stream_read(dev.data_ptr() + 8, 4080, None) == cp.CP_ERR_INVALID_ARG
    assert L.cp_measure_stream_read(dev.data_ptr(), 4095, None) == cp.CP_ERR_INVALID_ARG
    pageable = torch.ones(4096, dtype=torch.uint8)                  # not page-locked
    assert L.cp_measure_stream_read(pageable.data_ptr(), 4096, None) == cp.CP_ERR_INVALID_ARG


def test_record_read_device_and_pinned_host():
    """Sorted distinct rows including the table's last record (its last piece
    would pass the table's end) and ids past the table (skipped): the call
    queues, completes and writes nothing."""
    R, n_rows = 258, 4097
    dev = torch.full((n_rows * R,), 7, dtype=torch.uint8, device="cuda")
    host = torch.full((n_rows * R,), 7, dtype=torch.uint8).pin_memory()
    rows = torch.tensor([0, 1, 2, 17, 1000, 4095, 4096, 4097, 1 << 40], dtype=torch.int64,
                        device="cuda")
    for t in (dev, host):
        cp.measure_record_read(t, R, rows)
        cp.measure_record_read(t, R, rows[:1])
    torch.cuda.synchronize()
    assert bool((dev == 7).all()) and bool((host == 7).all())


def test_record_read_rejects_unusable_buffers():
    rows = torch.zeros(4, dtype=torch.int64, device="cuda")
    pageable = torch.ones(4096, dtype=torch.uint8)                  # not page-locked
    with pytest.raises(cp.CPError):
        cp.measure_record_read(pageable, 258, rows)
    with pytest.raises(ValueError):
        cp.measure_record_read(torch.ones(4096, dtype=torch.uint8, device="cuda"), 258, rows.cpu())
