"""cp_lookup_decode_host_noalloc: the host-resident decode for callers that cannot
allocate device memory (its scratch is a static device array inside libcp).

Collected last on purpose.  It must agree bit for bit with cp_lookup_decode_host
and with the oracle (the tolerance of every parity test here), on two calls in a
row that share the static scratch, whether run alone or after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import trellis_row_decode_gb300 as cp
from trellis_row_decode_gb300 import synth

from gpu_util import compare, oracle_decode

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def test_noalloc_matches_table_entry_point_on_consecutive_calls():
    d, k, n_rows = 1024, 4, 20011
    rec = synth.gen_records(11, torch.arange(n_rows), d, k).reshape(-1).contiguous().pin_memory()
    table = cp.load_table(rec, n_rows, d, k)            # the existing host-resident entry point
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    free_before = None
    for call, (seed, n) in enumerate([(5, 40000), (6, 65536)]):
        idx_np = synth.zipf_indices(seed, n, n_rows)
        idx_np[3] = -1                                   # one out-of-range id per call
        idx = torch.from_numpy(idx_np).cuda()
        ref = cp.lookup_decode_host(table, idx)
        assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB
        status.zero_()
        out = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
        if call == 1:
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        cp.lookup_decode_host_noalloc(rec, n_rows, d, k, idx, out, status)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] >= free_before - (2 << 20)
        assert np.array_equal(_bits(out), _bits(ref)), f"call {call}: output differs"
        n_bad, ulp = compare(_bits(out).view(np.uint16),
                             oracle_decode(11, d, k, idx_np, n_rows, cp.default_lut()))
        assert n_bad == 0, f"call {call}: {n_bad} elements differ from the oracle ({ulp} ulp)"
        assert int(status.item()) & 1 == 1
        assert not out[3].view(torch.int16).any()
    table.close()


def test_noalloc_rejects_more_than_its_capacity():
    d, k, n_rows = 256, 4, 100
    rec = synth.gen_records(1, torch.arange(n_rows), d, k).reshape(-1).contiguous().pin_memory()
    n = 65537
    idx = torch.zeros(n, dtype=torch.int64, device="cuda")
    out = torch.full((n, d), 3.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lut = cp.default_lut()
    rc = cp.lib().cp_lookup_decode_host_noalloc(rec.data_ptr(), n_rows, d, k, lut.ctypes.data,
                                                idx.data_ptr(), n, out.data_ptr(),
                                                status.data_ptr(), None)
    assert rc == cp.CP_ERR_INVALID_ARG
    assert b"65536" in cp.lib().cp_last_error()
    torch.cuda.synchronize()
    assert bool((out.float() == 3.0).all())              # nothing was queued


def test_noalloc_rejects_a_short_records_buffer():
    """The wrapper refuses a pinned buffer smaller than n_rows records, before any launch."""
    d, k, n_rows = 256, 4, 100
    rec = torch.zeros(n_rows * synth.record_bytes(d, k) - 2, dtype=torch.uint8).pin_memory()
    idx = torch.zeros(4, dtype=torch.int64, device="cuda")
    out = torch.empty((4, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        cp.lookup_decode_host_noalloc(rec, n_rows, d, k, idx, out, status)


def test_noalloc_tables_of_different_sizes_in_turn():
    """Calls on tables with different numbers of row ranges share the static
    scratch in turn (its counters must be back at zero after each call)."""
    d, k = 512, 4
    lut = cp.default_lut()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tables = {}
    for n_rows in (300, 50021):
        tables[n_rows] = synth.gen_records(3, torch.arange(n_rows), d, k).reshape(-1) \
            .contiguous().pin_memory()
    for call, (n_rows, seed, n) in enumerate([(50021, 1, 30000), (300, 2, 5000),
                                              (50021, 3, 65536), (300, 4, 777)]):
        idx_np = synth.zipf_indices(seed, n, n_rows)
        idx = torch.from_numpy(idx_np).cuda()
        out = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
        cp.lookup_decode_host_noalloc(tables[n_rows], n_rows, d, k, idx, out, status)
        torch.cuda.synchronize()
        n_bad, ulp = compare(_bits(out).view(np.uint16), oracle_decode(3, d, k, idx_np, n_rows, lut))
        assert n_bad == 0, f"call {call}: {n_bad} elements differ from the oracle ({ulp} ulp)"
    assert int(status.item()) == 0
