"""Hot-row cache of host-resident tables (cp_table_set_cache): outputs unchanged, bit
for bit, whichever rows are cached; argument errors are rejected on the host."""
import numpy as np
import pytest
import torch

import trellis_row_decode_gb300 as cp
from trellis_row_decode_gb300 import synth

from gpu_util import bits, compare, oracle_decode

pytestmark = pytest.mark.gpu
SEED = 17


def _host_table(n_rows, d, k):
    rec = synth.gen_records(SEED, torch.arange(n_rows), d, k).reshape(-1).contiguous()
    return rec, rec.pin_memory()


def test_cache_keeps_outputs_identical():
    d, k, n_rows, n = 1024, 4, 20011, 50000
    rec_cpu, host = _host_table(n_rows, d, k)
    table = cp.load_table(host, n_rows, d, k)
    dev = cp.load_table(rec_cpu.cuda(), n_rows, d, k)
    idx_np = synth.zipf_indices(4, n, n_rows)
    idx_np[7] = -3
    idx = torch.from_numpy(idx_np).cuda()
    ref = bits(cp.lookup_decode(dev, idx))
    plain = bits(cp.lookup_decode_host(table, idx))
    assert np.array_equal(plain, ref)
    vals, counts = np.unique(idx_np[idx_np >= 0], return_counts=True)
    hot = vals[np.argsort(-counts)][:1000]
    for rows in (np.unique(np.concatenate([hot, [n_rows - 1]])),      # hot ids + the last row
                 np.random.default_rng(1).choice(n_rows, 3000, replace=False),
                 np.arange(n_rows)):                                    # everything cached
        cp.set_cache(table, rows)
        got = bits(cp.lookup_decode_host(table, idx))
        assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB
        assert np.array_equal(got, ref)
    cp.set_cache(table, [])                                            # removed
    assert np.array_equal(bits(cp.lookup_decode_host(table, idx)), ref)
    n_bad, ulp = compare(ref.reshape(n, d), oracle_decode(SEED, d, k, idx_np, n_rows,
                                                          cp.default_lut()))
    assert n_bad == 0, f"{n_bad} elements differ (max {ulp} ulp)"


def test_cache_argument_errors():
    d, k, n_rows = 512, 4, 1000
    rec_cpu, host = _host_table(n_rows, d, k)
    table = cp.load_table(host, n_rows, d, k)
    with pytest.raises(cp.CPError):
        cp.set_cache(table, [1, 2, 2])                                 # duplicate
    with pytest.raises(cp.CPError):
        cp.set_cache(table, [5, n_rows])                               # out of range
    dev = cp.load_table(rec_cpu.cuda(), n_rows, d, k)
    with pytest.raises(cp.CPError):
        cp.set_cache(dev, [1, 2])                                      # device-resident table
    soa = torch.empty(cp.soa_bytes(n_rows, d, k), dtype=torch.uint8, pin_memory=True)
    t2 = cp.load_table(host, n_rows, d, k, layout=cp.CP_LAYOUT_SOA, soa=soa)
    with pytest.raises(cp.CPError):
        cp.set_cache(t2, [1, 2])                                       # SoA layout
    cp.lib().cp_test_inject_failure(1, 1)
    with pytest.raises(cp.CPError) as ei:
        cp.set_cache(table, [1, 2])
    assert ei.value.status == cp.CP_ERR_NO_MEMORY


def test_cache_full_size_top_ranks():
    """51 GB host table, the 2^20 hottest Zipf ranks cached in HBM."""
    w = synth.WORKLOADS["host_prefill"]
    R = w.rec_bytes
    host = torch.empty(w.n_rows * R, dtype=torch.uint8, pin_memory=True)
    chunk = 1 << 22
    stage = torch.empty(chunk * R, dtype=torch.uint8, device="cuda")
    for r0 in range(0, w.n_rows, chunk):
        r1 = min(w.n_rows, r0 + chunk)
        rows = torch.arange(r0, r1, dtype=torch.int64, device="cuda")
        stage[: (r1 - r0) * R].view(r1 - r0, R).copy_(synth.gen_records(synth.SEED_TABLE, rows, w.d, w.k))
        host[r0 * R: r1 * R].copy_(stage[: (r1 - r0) * R])
    del stage
    table = cp.load_table(host, w.n_rows, w.d, w.k)
    idx_np = w.indices()
    idx = torch.from_numpy(idx_np).cuda()
    plain = bits(cp.lookup_decode_host(table, idx))
    hot = synth.feistel_bijection(np.arange(1 << 20), w.n_rows, synth.SEED_INDEX)
    cp.set_cache(table, hot)
    got = bits(cp.lookup_decode_host(table, idx))
    assert cp.get_status(table) == cp.CP_OK
    assert np.array_equal(got, plain)
    n_bad, ulp = 0, 0
    for j in range(0, idx_np.size, 1 << 16):
        b, u = compare(got[j:j + (1 << 16)],
                       oracle_decode(synth.SEED_TABLE, w.d, w.k, idx_np[j:j + (1 << 16)],
                                     w.n_rows, cp.default_lut()))
        n_bad, ulp = n_bad + b, max(ulp, u)
    assert n_bad == 0, f"{n_bad} elements differ (max {ulp} ulp)"
    table.close()
