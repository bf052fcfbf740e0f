"""Pins for the oracle's decode fused with a weighted group readout.

  * group 1 with unit weights reduces to the plain lookup-decode, bit for bit;
  * power-of-two weights scale exactly (torch's fp32 product rounded to bf16);
  * a group of identical rows sums exactly (torch's fp32 product by the count);
  * the result is within the fp32-accumulation + bf16 bound of an fp64 sum;
  * out-of-range ids contribute zero rows and are counted.
"""
import numpy as np
import torch


def _records(rng, n_rows, d, k):
    cb = d * k // 16
    rec = rng.integers(0, 256, (n_rows, cb + 2)).astype(np.uint8)
    a = torch.from_numpy(rng.lognormal(0, 0.25, n_rows).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rec[:, cb] = a & 0xFF
    rec[:, cb + 1] = a >> 8
    return rec


def _f(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_group_one_is_plain_decode(orc, lut):
    rng = np.random.default_rng(1)
    d, k = 256, 4
    rec = _records(rng, 40, d, k)
    idx = rng.integers(0, 40, 100)
    plain, _ = orc.lookup_decode(rec, 40, d, k, rec.shape[1], lut, idx)
    red, _ = orc.lookup_decode_reduce(rec, 40, d, k, rec.shape[1], lut, idx, 1)
    assert np.array_equal(plain, red)


def test_power_of_two_weights_scale_exactly(orc, lut):
    rng = np.random.default_rng(2)
    d, k = 64, 6
    rec = _records(rng, 10, d, k)
    idx = np.arange(10)
    w = np.full(10, 4.0, np.float32)
    plain, _ = orc.lookup_decode(rec, 10, d, k, rec.shape[1], lut, idx)
    red, _ = orc.lookup_decode_reduce(rec, 10, d, k, rec.shape[1], lut, idx, 1, w)
    ref = (torch.from_numpy(_f(plain)) * 4.0).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(red.view(np.int16), ref)


def test_identical_rows_sum_exactly(orc, lut):
    rng = np.random.default_rng(3)
    d, k, g = 128, 4, 24
    rec = _records(rng, 5, d, k)
    idx = np.repeat(np.arange(5), g)
    plain, _ = orc.lookup_decode(rec, 5, d, k, rec.shape[1], lut, np.arange(5))
    red, _ = orc.lookup_decode_reduce(rec, 5, d, k, rec.shape[1], lut, idx, g)
    ref = (torch.from_numpy(_f(plain)) * float(g)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(red.view(np.int16), ref)


def test_within_bound_of_fp64_sum(orc, lut):
    rng = np.random.default_rng(4)
    d, k, g = 256, 5, 48
    rec = _records(rng, 300, d, k)
    idx = rng.integers(0, 300, g * 20)
    w = rng.standard_normal(idx.size).astype(np.float32)
    plain, _ = orc.lookup_decode(rec, 300, d, k, rec.shape[1], lut, idx)
    red, _ = orc.lookup_decode_reduce(rec, 300, d, k, rec.shape[1], lut, idx, g, w)
    rows = _f(plain).astype(np.float64).reshape(20, g, d)
    exact = np.einsum("gi,giq->gq", w.astype(np.float64).reshape(20, g), rows)
    absum = np.einsum("gi,giq->gq", np.abs(w.astype(np.float64)).reshape(20, g), np.abs(rows))
    got = _f(red).astype(np.float64)
    bound = g * 2.0 ** -24 * absum + 2.0 ** -8 * np.abs(exact) + 1e-30
    assert np.all(np.abs(got - exact) <= bound)


def test_out_of_range_ids_contribute_zero(orc, lut):
    rng = np.random.default_rng(5)
    d, k = 64, 4
    rec = _records(rng, 8, d, k)
    idx = np.array([1, 2, -1, 3, 8, 4])
    red, bad = orc.lookup_decode_reduce(rec, 8, d, k, rec.shape[1], lut, idx, 3)
    ok, _ = orc.lookup_decode_reduce(rec, 8, d, k, rec.shape[1], lut, np.array([1, 2, 3, 4]), 2)
    assert bad == 2
    # group 0 = rows 1, 2 (+ a zero row); group 1 = rows 3, 4 (+ a zero row in the middle)
    assert np.array_equal(red[0], ok[0]) and np.array_equal(red[1], ok[1])
