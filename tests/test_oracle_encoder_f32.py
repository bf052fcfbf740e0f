"""Pins for the oracle's fp32 encoder (the precision of the GPU encoder).

  * fp32 brute force over every code equals the exact fp32 tail-biting search in
    cost (bit for bit) and code (the group-wise minimum is exact because fp32
    addition is monotone);
  * the reported metric equals the fp32 distortion recomputed from the code;
  * the two-pass cost is >= the exact cost;
  * it agrees with the fp64 encoder up to fp32 rounding;
  * the records restore the norm within the bf16 bound.
"""
import numpy as np
import pytest

from trellis_row_decode_gb300 import synth


def _z(rng, d):
    e = rng.standard_normal(d)
    return (np.sqrt(d) * e / np.linalg.norm(e)).astype(np.float32)


@pytest.mark.parametrize("d,k,rows", [(8, 4, 2), (8, 5, 1), (8, 6, 1), (12, 4, 1)])
def test_f32_brute_force_equals_exact(orc, lut, d, k, rows):
    rng = np.random.default_rng(200 + d * 7 + k)
    for _ in range(rows):
        z = _z(rng, d)
        cb, cost_b = orc.encode_z_f32(z, d, k, lut, orc.BRUTE)
        cv, cost_v = orc.encode_z_f32(z, d, k, lut, orc.EXACT)
        assert np.float32(cost_b) == np.float32(cost_v)
        assert np.array_equal(cb, cv)
        assert np.float32(orc.distortion_f32(z, cv, d, k, lut)) == np.float32(cost_v)
        c2, cost_2 = orc.encode_z_f32(z, d, k, lut, orc.TWO_PASS)
        assert cost_2 >= cost_v
        assert np.float32(orc.distortion_f32(z, c2, d, k, lut)) == np.float32(cost_2)


def test_f32_close_to_f64(orc, lut):
    d, k = 256, 4
    e = synth.normal_rows(41, 12, d)
    rec64, _, cost64 = orc.encode_rows(e, d, k, lut, orc.TWO_PASS, n_threads=8)
    rec32, cost32 = orc.encode_rows_f32(e.astype(np.float32), d, k, lut, n_threads=8)
    assert np.allclose(cost32, cost64, rtol=2e-3)
    same = np.mean([np.array_equal(a[:-2], b[:-2]) for a, b in zip(rec32, rec64)])
    assert same >= 0.5


def test_f32_records_restore_norm(orc, lut):
    d, k = 256, 4
    e = synth.normal_rows(43, 8, d).astype(np.float32)
    rec, cost = orc.encode_rows_f32(e, d, k, lut, n_threads=8)
    out, _ = orc.lookup_decode(rec, 8, d, k, rec.shape[1], lut, np.arange(8))
    ehat = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rel = np.abs(np.linalg.norm(ehat, axis=1) / np.linalg.norm(e.astype(np.float64), axis=1) - 1)
    assert rel.max() <= 2.0 ** -8 + 1e-3
    assert np.all(cost > 0) and np.all(cost / d < 0.12)


def test_f32_zero_row(orc, lut):
    rec, cost = orc.encode_rows_f32(np.zeros((1, 64), np.float32), 64, 4, lut)
    assert not rec.any() and cost[0] == 0
