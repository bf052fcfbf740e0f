"""cp_measure_stream_read: the streaming-read kernel that measures the host link
(zero-copy from pinned memory) and HBM reads for the rooflines."""
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
