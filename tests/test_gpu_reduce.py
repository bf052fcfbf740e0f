"""GPU parity of cp_lookup_decode_reduce (decode fused with a weighted group readout)
against the oracle's composition, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import trellis_row_decode_gb300 as cp
from trellis_row_decode_gb300 import synth

from gpu_util import NT, bits, compare, device_table

pytestmark = pytest.mark.gpu
SEED = 13


def _oracle(seed, d, k, idx, n_rows, lut, group, w):
    idx = np.asarray(idx, np.int64)
    valid = (idx >= 0) & (idx < n_rows)
    uniq, inv = np.unique(np.where(valid, idx, 0), return_inverse=True)
    rec = synth.gen_records(seed, torch.from_numpy(uniq), d, k).numpy()
    local = np.where(valid, inv, -1).astype(np.int64)
    out, _ = oracle.lookup_decode_reduce(rec, len(uniq), d, k, rec.shape[1], lut, local, group,
                                         w, n_threads=NT)
    return out


@pytest.mark.parametrize("layout", [cp.CP_LAYOUT_AOS, cp.CP_LAYOUT_SOA])
@pytest.mark.parametrize("k", [3, 4, 5, 6])
@pytest.mark.parametrize("d", [256, 512, 1024])
def test_reduce_parity(d, k, layout):
    lut = cp.default_lut()
    n_rows, group, n_groups = 2003, 24, 211
    rec = device_table(SEED, n_rows, d, k)
    soa = None
    if layout == cp.CP_LAYOUT_SOA:
        soa = torch.empty(cp.soa_bytes(n_rows, d, k), dtype=torch.uint8, device="cuda")
    table = cp.load_table(rec, n_rows, d, k, lut, layout=layout, soa=soa)
    idx = synth.zipf_indices(3, n_groups * group, n_rows)
    idx[:2] = [n_rows - 1, n_rows - 1]
    w = np.random.default_rng(d + k).standard_normal(idx.size).astype(np.float32)
    for weights in (None, w):
        wt = None if weights is None else torch.from_numpy(weights).cuda()
        out = cp.lookup_decode_reduce(table, torch.from_numpy(idx).cuda(), group, wt)
        torch.cuda.synchronize()
        ref = _oracle(SEED, d, k, idx, n_rows, lut, group, weights)
        n, ulp = compare(bits(out), ref)
        assert n == 0, f"{n} elements differ (max {ulp} ulp)"


@pytest.mark.parametrize("group", [1, 7, 48])
def test_reduce_group_sizes_and_out_of_range(group):
    lut = cp.default_lut()
    d, k, n_rows = 512, 4, 999
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k, lut)
    n_groups = 1000 // group + 3
    idx = synth.uniform_indices(group, n_groups * group, n_rows)
    idx[::11] = -5
    w = np.linspace(-2, 2, idx.size).astype(np.float32)
    out = cp.lookup_decode_reduce(table, torch.from_numpy(idx).cuda(), group,
                                  torch.from_numpy(w).cuda())
    assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB
    n, ulp = compare(bits(out), _oracle(SEED, d, k, idx, n_rows, lut, group, w))
    assert n == 0, f"{n} elements differ (max {ulp} ulp)"


def test_reduce_group_one_equals_plain_decode():
    d, k, n_rows = 1024, 4, 500
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k)
    idx = torch.from_numpy(synth.zipf_indices(1, 4000, n_rows)).cuda()
    a = cp.lookup_decode_reduce(table, idx, 1)
    b = cp.lookup_decode(table, idx)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_reduce_rejects_unsupported_geometry():
    d, k, n_rows = 64, 4, 10
    table = cp.load_table(device_table(SEED, n_rows, d, k), n_rows, d, k)
    with pytest.raises(cp.CPError):
        cp.lookup_decode_reduce(table, torch.zeros(8, dtype=torch.int64, device="cuda"), 4)


def test_reduce_full_size():
    """DeepSeek-scale table (51 GB), 4096 tokens x 2 layers x 24 rows, random gates:
    every one of the 8,192 output rows against the oracle."""
    w_ = synth.WORKLOADS["deepseek_prefill"]
    lut = cp.default_lut()
    rec = device_table(synth.SEED_TABLE, w_.n_rows, w_.d, w_.k)
    table = cp.load_table(rec, w_.n_rows, w_.d, w_.k, lut)
    idx = w_.indices()
    gates = np.random.default_rng(9).random(idx.size).astype(np.float32)
    out = cp.lookup_decode_reduce(table, torch.from_numpy(idx).cuda(), 24,
                                  torch.from_numpy(gates).cuda())
    torch.cuda.synchronize()
    assert cp.get_status(table) == cp.CP_OK
    ref = _oracle(synth.SEED_TABLE, w_.d, w_.k, idx, w_.n_rows, lut, 24, gates)
    n, ulp = compare(bits(out), ref)
    assert n == 0, f"{n} elements differ (max {ulp} ulp)"
    table.close()
    del rec
    torch.cuda.empty_cache()
