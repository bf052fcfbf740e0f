"""Pins for the oracle's mixed-rate lookup-decode (one bit rate per row)."""
import numpy as np
import torch

from trellis_row_decode_gb300 import synth


def _mixed(seed, n_rows, d):
    ks = synth.mixed_rates(seed, torch.arange(n_rows)).numpy()
    recs = [synth.gen_records(seed, torch.tensor([r]), d, int(k)).numpy()[0] for r, k in enumerate(ks)]
    offs = np.zeros(n_rows + 1, np.uint64)
    offs[1:] = np.cumsum([len(x) for x in recs])
    return ks, np.concatenate(recs), offs


def test_uniform_rate_equals_plain_decode(orc, lut):
    d, k, n_rows = 256, 4, 30
    rec = synth.gen_records(1, torch.arange(n_rows), d, k).numpy()
    offs = (np.arange(n_rows + 1) * rec.shape[1]).astype(np.uint64)
    idx = np.random.default_rng(0).integers(0, n_rows, 80)
    a, _ = orc.lookup_decode(rec, n_rows, d, k, rec.shape[1], lut, idx)
    b, bad = orc.lookup_decode_mixed(rec.reshape(-1), offs, d, lut, idx)
    assert bad == 0 and np.array_equal(a, b)


def test_each_row_decodes_at_its_own_rate(orc, lut):
    d, n_rows = 512, 40
    ks, flat, offs = _mixed(3, n_rows, d)
    assert set(ks.tolist()) == {3, 4, 5, 6}
    idx = np.arange(n_rows)
    out, bad = orc.lookup_decode_mixed(flat, offs, d, lut, idx)
    assert bad == 0
    for r in range(n_rows):
        rec = flat[int(offs[r]):int(offs[r + 1])]
        one, _ = orc.lookup_decode(rec[None, :], 1, d, int(ks[r]), rec.size, lut, np.array([0]))
        assert np.array_equal(out[r], one[0])
    # storage: b_r + 16/d bits per parameter for every row
    R = np.diff(offs.astype(np.int64))
    assert np.array_equal(R * 8 / d, ks / 2 + 16 / d)


def test_unusable_record_length_gives_zero_row(orc, lut):
    d, n_rows = 256, 4
    ks, flat, offs = _mixed(5, n_rows, d)
    bad_offs = offs.copy()
    bad_offs[2] = bad_offs[1] + 10                    # row 1: 10 bytes, no valid rate
    flat2 = np.concatenate([flat, np.zeros(64, np.uint8)])
    out, bad = orc.lookup_decode_mixed(flat2, bad_offs, d, lut, np.array([1, 0, -1]))
    assert bad == 2 and not out[0].any() and not out[2].any() and out[1].any()
