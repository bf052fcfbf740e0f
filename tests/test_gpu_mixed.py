"""GPU parity of mixed-rate tables (cp_table_load_mixed + cp_lookup_decode), bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import trellis_row_decode_gb300 as cp
from trellis_row_decode_gb300 import synth

from gpu_util import bits, compare

pytestmark = pytest.mark.gpu
SEED = 23


def _device_mixed(n_rows, d):
    ks = synth.mixed_rates(SEED, torch.arange(n_rows, device="cuda"))
    offs = synth.mixed_offsets(ks, d)
    total = int(offs[-1].item())
    buf = torch.empty(total, dtype=torch.uint8, device="cuda")
    synth.fill_mixed_records(buf, SEED, ks, offs, d)
    return buf, offs, ks


def _oracle_mixed(d, idx, n_rows):
    """Oracle rows for the lookups idx: the records of the distinct ids are
    regenerated on the host (grouped by rate), concatenated with their offsets,
    and decoded by the oracle's mixed-rate lookup."""
    idx = np.asarray(idx, np.int64)
    valid = (idx >= 0) & (idx < n_rows)
    uniq, inv = np.unique(np.where(valid, idx, 0), return_inverse=True)
    ks = synth.mixed_rates(SEED, torch.from_numpy(uniq)).numpy()
    sizes = ks.astype(np.int64) * (d // 16) + 2
    offs = np.zeros(uniq.size + 1, np.uint64)
    offs[1:] = np.cumsum(sizes)
    buf = np.empty(int(offs[-1]), np.uint8)
    for k in (3, 4, 5, 6):
        sel = np.nonzero(ks == k)[0]
        if sel.size == 0:
            continue
        rec = synth.gen_records(SEED, torch.from_numpy(uniq[sel]), d, k).numpy()
        pos = offs[sel].astype(np.int64)[:, None] + np.arange(rec.shape[1])[None, :]
        buf[pos.ravel()] = rec.ravel()
    local = np.where(valid, inv, -1).astype(np.int64)
    out, _ = oracle.lookup_decode_mixed(buf, offs, d, cp.default_lut(), local)
    return out


@pytest.mark.parametrize("d", [256, 512, 1024, 2048, 96])
def test_mixed_parity(d):
    n_rows, n = 3001, 6007
    buf, offs, _ = _device_mixed(n_rows, d)
    table = cp.load_mixed_table(buf, offs, d)
    idx = synth.zipf_indices(2, n, n_rows)
    idx[:4] = [n_rows - 1, -1, n_rows, 0]
    out = cp.lookup_decode(table, torch.from_numpy(idx).cuda())
    assert cp.get_status(table) == cp.CP_ERR_INDEX_OOB
    nb, ulp = compare(bits(out), _oracle_mixed(d, idx, n_rows))
    assert nb == 0, f"{nb} elements differ (max {ulp} ulp)"


def test_mixed_rejects_bad_tables():
    d, n_rows = 256, 100
    buf, offs, _ = _device_mixed(n_rows, d)
    bad = offs.clone()
    bad[5] += 2                                            # rows 4 and 5 change length
    with pytest.raises(cp.CPError) as ei:
        cp.load_mixed_table(buf, bad, d)
    assert ei.value.status == cp.CP_ERR_FORMAT
    with pytest.raises(cp.CPError):
        cp.load_mixed_table(buf, offs, 48)                 # d not a multiple of 32


def test_mixed_full_size():
    """2^24 rows x d=1024, rates uniform over b = 1.5..3, Zipf replay of 196,608 ids:
    every output row against the oracle."""
    n_rows, d = 1 << 24, 1024
    buf, offs, _ = _device_mixed(n_rows, d)
    table = cp.load_mixed_table(buf, offs, d)
    idx = synth.zipf_indices(synth.SEED_INDEX, 196608, n_rows)
    out = cp.lookup_decode(table, torch.from_numpy(idx).cuda())
    assert cp.get_status(table) == cp.CP_OK
    got = bits(out)
    nb, ulp = 0, 0
    for j in range(0, idx.size, 1 << 16):
        b, u = compare(got[j:j + (1 << 16)], _oracle_mixed(d, idx[j:j + (1 << 16)], n_rows))
        nb, ulp = nb + b, max(ulp, u)
    assert nb == 0, f"{nb} elements differ (max {ulp} ulp)"
    table.close()
