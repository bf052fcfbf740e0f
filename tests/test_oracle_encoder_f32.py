"""Pins for the oracle's fp32 encoder (the precision of the GPU encoder).

  * fp32 brute force over every code equals the exact fp32 tail-biting search in
    cost (bit for bit) and code (the group-wise minimum is exact because fp32
    addition is monotone);
  * the reported metric equals the fp32 distortion recomputed from the code;
  * the two-pass cost is >= the exact cost;
  * its first pass (a free-start Viterbi over the steps rotated by T/2) reaches
    the same minimum as an enumeration of every free-start path, follows a valid
    trellis path, and never exceeds the exact tail-biting cost (a relaxation);
  * the two-pass code's pre-window bits (cyclic positions [Lc - W, Lc)) are the
    top W bits of that path's state at the last step, the w the second pass is
    constrained to;
  * with the same w it matches the fp64 encoder up to fp32 rounding, and never
    beats the fp64 optimum for that w;
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


def _bits_value(code, lo, hi):
    """Integer made of code bits lo .. hi-1 (LSB-first stream), bit lo lowest."""
    return sum(((int(code[j >> 3]) >> (j & 7)) & 1) << (j - lo) for j in range(lo, hi))


@pytest.mark.parametrize("k", [3, 4])
def test_free_start_pass_equals_enumeration(orc, lut, k):
    """d = 8 (T = 4): the free-start pass's minimum equals the minimum over all
    2^(16 + k(T-1)) free-start paths, bit for bit (both accumulate in fp32 in the
    pass's step order), for rotations rho = 0, 1, 2."""
    d, T, W = 8, 4, 16 - k
    rng = np.random.default_rng(300 + k)
    for rho in (0, 1, 2):
        z = _z(rng, d)
        c, st = orc.free_start_f32(z, d, k, lut, rho)
        cb, stb = orc.free_start_f32(z, d, k, lut, rho, brute=True)
        assert np.float32(c) == np.float32(cb), (rho, c, cb)
        order = [(rho + i) % T for i in range(T)]
        for path in (st, stb):                 # each state is its predecessor shifted by k bits
            for a, b in zip(order, order[1:]):
                assert (int(path[a]) >> k) == (int(path[b]) & ((1 << W) - 1))


@pytest.mark.parametrize("d,k", [(8, 4), (8, 6), (12, 4), (16, 6)])
def test_free_start_is_a_relaxation(orc, lut, d, k):
    """Every tail-biting code is a free-start path, so the first pass's cost is at
    most the exact tail-biting cost, which is at most the two-pass cost."""
    rng = np.random.default_rng(400 + d + k)
    z = _z(rng, d)
    c_free, _ = orc.free_start_f32(z, d, k, lut)
    _, c_exact = orc.encode_z_f32(z, d, k, lut, orc.EXACT)
    _, c_two = orc.encode_z_f32(z, d, k, lut, orc.TWO_PASS)
    assert np.float32(c_free) <= np.float32(c_exact) <= np.float32(c_two)


@pytest.mark.parametrize("d,k", [(16, 4), (64, 3), (256, 4), (256, 6)])
def test_two_pass_w_comes_from_the_free_start_path(orc, lut, d, k):
    """The second pass is constrained to w = the top 16 - k bits of the best
    free-start path's state at the last step (original step T-1), which are the
    code bits at cyclic positions [Lc - W, Lc)."""
    T, W, Lc = d // 2, 16 - k, d * k // 2
    rng = np.random.default_rng(500 + d + k)
    for _ in range(3):
        z = _z(rng, d)
        _, st = orc.free_start_f32(z, d, k, lut)
        code, _ = orc.encode_z_f32(z, d, k, lut, orc.TWO_PASS)
        assert _bits_value(code, Lc - W, Lc) == int(st[T - 1]) >> k


def test_f32_matches_f64_up_to_rounding(orc, lut):
    """fp32 and fp64 two-pass encodings of the same rows: where both chose the same
    w, the fp32 code's cost evaluated in fp64 lies in [c64, c64 (1 + 1e-4)], c64
    the fp64 optimum for that w (the fp32 search sees every path's cost within
    fp32 rounding, so it cannot lose more; it cannot win, since c64 is optimal)."""
    d, k = 256, 4
    W, Lc = 16 - k, d * k // 2
    e = synth.normal_rows(41, 24, d)
    rec64, _, cost64 = orc.encode_rows(e, d, k, lut, orc.TWO_PASS, n_threads=8)
    rec32, cost32 = orc.encode_rows_f32(e.astype(np.float32), d, k, lut, n_threads=8)
    assert np.allclose(cost32, cost64, rtol=2e-3)
    same_w = 0
    for r in range(e.shape[0]):
        c32, c64 = rec32[r][:-2], rec64[r][:-2]
        if _bits_value(c32, Lc - W, Lc) != _bits_value(c64, Lc - W, Lc):
            continue
        same_w += 1
        z64 = np.sqrt(d) * e[r] / np.linalg.norm(e[r])
        d64_of_32 = orc.distortion(z64, c32, d, k, lut)
        assert d64_of_32 >= cost64[r] * (1 - 1e-12), (r, d64_of_32, cost64[r])
        assert d64_of_32 <= cost64[r] * (1 + 1e-4), (r, d64_of_32, cost64[r])
    assert same_w >= e.shape[0] // 2


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
