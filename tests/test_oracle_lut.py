"""Pins for the LUT construction (seeded Lloyd k-means on N(0,1) pairs).

  * the Box-Muller stream passes a Kolmogorov-Smirnov test against N(0,1);
  * with 2 centroids, Lloyd converges to the textbook optimum of the 2-D
    standard normal: two opposite points at distance sqrt(2/pi) from 0;
  * the committed LUT file is exactly what the generator writes (SHA-256);
  * its distortion on fresh pairs lies between the Gaussian rate-distortion
    bound 2^(-2R) at R = 4.5 bits/coordinate and the scalar 4.5-bit figure.
"""
import hashlib

import numpy as np
import pytest
from scipy import stats

from conftest import LUT_PATH

LUT_SHA256 = "cccfbe5f9765004137c22a927559426a059c85672a6e8f0116c43495ecd91743"


def test_normal_stream(orc):
    x = orc.normal_pairs(123, 0, 1 << 17).ravel()
    assert stats.kstest(x, "norm").pvalue > 1e-3
    assert abs(x.mean()) < 5 / np.sqrt(x.size)
    assert abs(x.var() - 1) < 0.02


def test_two_centroid_lloyd_reaches_textbook_optimum(orc):
    cent, _, mse = orc.lloyd_lut(77, 1 << 16, 2, 40, 4)
    r = np.linalg.norm(cent, axis=1)
    assert np.allclose(r, np.sqrt(2 / np.pi), rtol=0.03)
    assert np.allclose(cent[0], -cent[1], atol=0.03)
    # distortion per coordinate: (1 + 1 - 2/pi) / 2 = 1 - 1/pi
    assert abs(mse - (1 - 1 / np.pi)) < 0.01


def test_lloyd_independent_of_threads(orc):
    a = orc.lloyd_lut(5, 20000, 16, 5, 1)
    b = orc.lloyd_lut(5, 20000, 16, 5, 7)
    assert np.array_equal(a[0], b[0]) and a[2] == b[2]


def test_committed_lut_hash():
    assert hashlib.sha256(LUT_PATH.read_bytes()).hexdigest() == LUT_SHA256


@pytest.mark.slow
def test_committed_lut_regenerates(orc):
    from oracle import make_lut
    _, lut, _ = make_lut.generate()
    assert lut.astype("<u2").tobytes() == LUT_PATH.read_bytes()


def test_lut_distortion_on_fresh_pairs(orc, lut):
    v = orc.lut_values(lut)
    pts = orc.normal_pairs(999, 0, 1 << 15)
    d2 = ((pts[:, None, :] - v[None, :, :]) ** 2).sum(-1).min(1)
    mse = d2.mean() / 2
    assert 2.0 ** -9 < mse < 0.0055
    assert np.all(np.isfinite(v)) and np.abs(v).max() < 6
