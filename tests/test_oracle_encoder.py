"""Pins for the oracle's tail-biting TCQ encoder and the norm-restoring scale.

  * brute force over every code equals the exact tail-biting Viterbi, in cost
    (bit for bit, same fp64 summation order) and in the tie-broken code;
  * the Viterbi path metric equals D(c) recomputed from the decoded code;
  * the two-pass encoder returns a valid code whose cost is >= the exact one;
  * |alpha f(c)| = |e| after norm restoration ("how it differs":
    alpha = |e|_2 / |f(c)|_2);
  * encoded N(0,1) rows have lower relative MSE than 2-bit round-to-nearest
    and than the optimal 4-level scalar quantizer of N(0,1) (0.1175, Max 1960).
"""
import numpy as np
import pytest

from trellis_row_decode_gb300 import synth


def _z(rng, d):
    e = rng.standard_normal(d)
    return np.sqrt(d) * e / np.linalg.norm(e)


CASES = [  # (d, k, rows)
    (8, 4, 4),
    (8, 5, 2),
    (8, 6, 1),
    (12, 4, 1),
]


@pytest.mark.parametrize("d,k,rows", CASES)
def test_brute_force_equals_exact_viterbi(orc, lut, d, k, rows):
    rng = np.random.default_rng(100 + d * 7 + k)
    for _ in range(rows):
        z = _z(rng, d)
        cb, cost_b = orc.encode_z(z, d, k, lut, orc.BRUTE)
        cv, cost_v = orc.encode_z(z, d, k, lut, orc.EXACT)
        assert cost_b == cost_v                       # bitwise: same summation order
        assert np.array_equal(cb, cv)                 # same tie-broken code
        assert orc.distortion(z, cv, d, k, lut) == cost_v
        c2, cost_2 = orc.encode_z(z, d, k, lut, orc.TWO_PASS)
        assert cost_2 >= cost_v
        assert orc.distortion(z, c2, d, k, lut) == cost_2


def test_brute_force_short_code_k3(orc, lut):
    """Lc = 12 < 16: only brute force applies; its cost is the minimum of D."""
    d, k = 8, 3
    rng = np.random.default_rng(4)
    z = _z(rng, d)
    cb, cost = orc.encode_z(z, d, k, lut, orc.BRUTE)
    assert orc.distortion(z, cb, d, k, lut) == cost
    for c in rng.integers(0, 1 << 12, 300):
        code = np.array([c & 0xFF, c >> 8], dtype=np.uint8)
        assert orc.distortion(z, code, d, k, lut) >= cost
    with pytest.raises(ValueError):
        orc.encode_z(z, d, k, lut, orc.EXACT)


def test_exact_viterbi_handles_ties(orc, lut):
    """z = 0: every code costs sum |y|^2 of its states; ties are broken toward the smallest code."""
    d, k = 8, 4
    z = np.zeros(d)
    cb, cost_b = orc.encode_z(z, d, k, lut, orc.BRUTE)
    cv, cost_v = orc.encode_z(z, d, k, lut, orc.EXACT)
    assert cost_b == cost_v and np.array_equal(cb, cv)


def test_two_pass_metric_matches_distortion_d256(orc, lut):
    d, k = 256, 4
    rng = np.random.default_rng(8)
    z = _z(rng, d)
    code, cost = orc.encode_z(z, d, k, lut, orc.TWO_PASS)
    assert orc.distortion(z, code, d, k, lut) == cost
    assert cost / d < 0.12


@pytest.fixture(scope="session")
def encoded_rows(orc, lut):
    """64 N(0,1) rows, d=256, b=2, two-pass encoded (the tiny workload's round-trip set)."""
    d, k = 256, 4
    e = synth.normal_rows(synth.SEED_ENCODER_ROWS, 64, d)
    rec, alpha, cost = orc.encode_rows(e, d, k, lut, orc.TWO_PASS)
    return e, rec, alpha, cost


def test_normalised_row_has_norm_sqrt_d(encoded_rows):
    e, _, _, cost = encoded_rows
    d = e.shape[1]
    z = np.sqrt(d) * e / np.linalg.norm(e, axis=1, keepdims=True)
    assert np.allclose(np.sum(z * z, axis=1), d, rtol=1e-12)
    assert np.all(cost > 0)


def test_norm_restoration(orc, lut, encoded_rows):
    e, rec, alpha, _ = encoded_rows
    d, k = 256, 4
    cb = d * k // 16
    en = np.linalg.norm(e, axis=1)
    rel_exact, rel_stored = [], []
    for i in range(e.shape[0]):
        f = orc.decode_f(rec[i, :cb], d, k, lut)
        rel_exact.append(abs(np.linalg.norm(alpha[i] * f) / en[i] - 1))
        out, _ = orc.lookup_decode(rec, e.shape[0], d, k, rec.shape[1], lut, np.array([i]))
        ehat = out[0].astype(np.uint32) << 16
        ehat = ehat.view(np.float32).astype(np.float64)
        rel_stored.append(abs(np.linalg.norm(ehat) / en[i] - 1))
    assert max(rel_exact) <= 1e-3
    # bf16 alpha and bf16 outputs each round by at most 2^-9 relative
    assert max(rel_stored) <= 2.0 ** -8 + 1e-3
    assert np.mean(rel_stored) < 2.0 ** -9


def test_quality_beats_rtn_and_scalar_lloyd_max(orc, lut, encoded_rows):
    e, rec, _, _ = encoded_rows
    d, k = 256, 4
    out, _ = orc.lookup_decode(rec, e.shape[0], d, k, rec.shape[1], lut, np.arange(e.shape[0]))
    ehat = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    en2 = np.sum(e * e, axis=1)
    cp = np.mean(np.sum((e - ehat) ** 2, axis=1) / en2)
    rtn0 = np.mean([np.sum((r - orc.rtn2(r, 0)) ** 2) / np.sum(r * r) for r in e])
    rtn1 = np.mean([np.sum((r - orc.rtn2(r, 1)) ** 2) / np.sum(r * r) for r in e])
    assert cp < rtn0
    assert cp < rtn1
    assert cp < 0.1175
    assert rtn1 > 0.1175 * 0.9     # a 4-level scalar grid cannot beat Lloyd-Max by much


def test_rtn_hand_example(orc):
    e = np.array([3.0, -3.0, 1.0, -1.0, 0.2, -0.2, 2.0, -2.5])
    # absmax 3 -> step 2 (exact in bf16); levels -3, -1, 1, 3
    assert np.array_equal(orc.rtn2(e, 0), [3, -3, 1, -1, 1, -1, 3, -3])


def test_zero_row_encodes_to_zero(orc, lut):
    d, k = 16, 4
    rec, alpha, _ = orc.encode_rows(np.zeros((1, d)), d, k, lut, orc.TWO_PASS)
    assert not rec.any() and alpha[0] == 0.0


def test_golden_encoded_rows_regenerate(encoded_rows):
    """tests/golden/tiny_encoded_rows.txt is exactly what the oracle encoder writes."""
    import importlib.util
    from pathlib import Path
    p = Path(__file__).resolve().parent / "golden" / "make_golden.py"
    spec = importlib.util.spec_from_file_location("make_golden", p)
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    rec, alpha, cost = mg.load()
    _, rec2, alpha2, cost2 = encoded_rows
    assert np.array_equal(rec, rec2)
    assert np.array_equal(alpha, alpha2) and np.array_equal(cost, cost2)
