"""Pins for the oracle's trellis decoder f and the reconstruction alpha * f(c).

What pins what:
  * hand-derived states of periodic codes and hash outputs (tests/golden) fix
    the window's bit order, the cyclic read and the hash/index/sign bits;
  * the single-bit response fixes which windows see a given code bit;
  * cyclic rotation of the code by k bits rotates f(c) by 2 coordinates
    (tail-biting wrap);
  * the reconstruction matches torch's fp32 product rounded to bf16;
  * decoding a row alone equals decoding it inside a batch (independently
    addressable records);
  * record size equals b + 16/d bits per parameter.
"""
from pathlib import Path

import numpy as np
import pytest
import torch

GOLD = Path(__file__).resolve().parent / "golden" / "state_closed_forms.txt"


def _gold(kind):
    rows = []
    for line in GOLD.read_text().splitlines():
        if line.startswith(kind + " "):
            rows.append([int(v) for v in line.split()[1:]])
    return rows


def _pack(bits: np.ndarray) -> np.ndarray:
    return np.packbits(bits.astype(np.uint8), bitorder="little")


@pytest.mark.parametrize("d", [8, 16, 64, 256])
def test_periodic_code_constant_state(orc, d):
    for k, s_expect in _gold("periodic"):
        Lc = k * d // 2
        if Lc % 8:
            continue
        bits = (np.arange(Lc) % k == 0)
        st = orc.window_states(_pack(bits), d, k)
        assert np.all(st == s_expect), (k, d, st[:4])


def test_all_zero_and_all_one_codes(orc, lut):
    vals = orc.lut_values(lut)
    for d, k in [(8, 4), (256, 4), (1024, 6), (16, 3)]:
        Lc = k * d // 2
        f0 = orc.decode_f(np.zeros(Lc // 8, np.uint8), d, k, lut)
        assert np.array_equal(f0.reshape(-1, 2), np.tile(vals[0], (d // 2, 1)))
        f1 = orc.decode_f(np.full(Lc // 8, 0xFF, np.uint8), d, k, lut)
        # all ones: s = 0xFFFF -> entry 508, second coordinate negated
        assert np.array_equal(f1.reshape(-1, 2), np.tile([vals[508, 0], -vals[508, 1]], (d // 2, 1)))


def test_hash_closed_forms(orc):
    g = np.array(_gold("hash"), dtype=np.uint32)
    idx, neg = orc.state_hash(g[:, 0])
    assert np.array_equal(idx, g[:, 1])
    assert np.array_equal(neg, g[:, 2])


@pytest.mark.parametrize("d,k", [(16, 3), (8, 4), (32, 5), (8, 6), (256, 4), (64, 6)])
def test_single_bit_response(orc, d, k):
    Lc = k * d // 2
    T = d // 2
    for j in [0, 1, Lc // 2, Lc - 1]:
        bits = np.zeros(Lc, np.uint8)
        bits[j] = 1
        st = orc.window_states(_pack(bits), d, k)
        for t in range(T):
            # offset of bit j inside the window that ends at k(t+1), cyclically
            off = (j - (k * (t + 1) - 16)) % Lc
            expect = (1 << off) if off < 16 else 0
            assert st[t] == expect, (j, t, st[t], expect)


@pytest.mark.parametrize("d,k", [(16, 3), (8, 4), (256, 4), (1024, 3), (1024, 5), (512, 6)])
def test_tail_biting_rotation(orc, lut, d, k):
    rng = np.random.default_rng(d * 10 + k)
    Lc = k * d // 2
    bits = rng.integers(0, 2, Lc).astype(np.uint8)
    f = orc.decode_f(_pack(bits), d, k, lut)
    for shift_steps in [1, 3]:
        rot = np.roll(bits, -k * shift_steps)        # new bit j = old bit j + k*shift
        fr = orc.decode_f(_pack(rot), d, k, lut)
        assert np.array_equal(fr, np.roll(f, -2 * shift_steps))


def _records(rng, n_rows, d, k, alphas=None):
    cb = d * k // 16
    rec = rng.integers(0, 256, (n_rows, cb + 2)).astype(np.uint8)
    if alphas is None:
        alphas = torch.from_numpy(rng.lognormal(0, 0.25, n_rows).astype(np.float32)).to(
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rec[:, cb] = alphas & 0xFF
    rec[:, cb + 1] = alphas >> 8
    return rec


@pytest.mark.parametrize("d,k", [(256, 4), (64, 3), (128, 6), (1024, 5)])
def test_reconstruction_matches_torch_fp32_product(orc, lut, d, k):
    rng = np.random.default_rng(5)
    n_rows = 17
    rec = _records(rng, n_rows, d, k)
    idx = rng.integers(0, n_rows, 40)
    out, bad = orc.lookup_decode(rec, n_rows, d, k, rec.shape[1], lut, idx)
    assert bad == 0
    cb = d * k // 16
    for j, r in enumerate(idx):
        f = orc.decode_f(rec[r, :cb], d, k, lut)
        a = torch.tensor([int(rec[r, cb]) | (int(rec[r, cb + 1]) << 8)], dtype=torch.int32)
        a = a.to(torch.int16).view(torch.bfloat16).to(torch.float32)
        ref = (torch.from_numpy(f.astype(np.float32)) * a).to(torch.bfloat16)
        ref = ref.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out[j], ref)


def test_special_alphas(orc, lut):
    d, k = 64, 4
    rng = np.random.default_rng(9)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x7F7F,
                         0x3F80], dtype=np.uint16)
    rec = _records(rng, len(specials), d, k, specials)
    out, _ = orc.lookup_decode(rec, len(specials), d, k, rec.shape[1], lut,
                               np.arange(len(specials)))
    vals = out.view(np.uint16)
    f = [orc.decode_f(rec[i, :d * k // 16], d, k, lut) for i in range(len(specials))]
    assert np.all((vals[0] & 0x7FFF) == 0)                       # +0 * y = +-0
    assert np.all(((vals[0] >> 15) == 1) == np.signbit(f[0]))    # sign follows y
    assert np.all((vals[2] & 0x7FFF) == 0x7F80)                  # inf * y = +-inf
    assert np.all(vals[4] == 0x7FFF)                             # NaN -> canonical NaN
    one = vals[8].view(np.uint16)                                # alpha = 1.0
    ref = torch.from_numpy(f[8].astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(one, ref.numpy().view(np.uint16))


def test_batch_independence_and_order(orc, lut):
    d, k = 256, 4
    rng = np.random.default_rng(21)
    rec = _records(rng, 50, d, k)
    idx = rng.integers(0, 50, 300)                    # duplicates, arbitrary order
    out, _ = orc.lookup_decode(rec, 50, d, k, rec.shape[1], lut, idx, n_threads=4)
    for j in [0, 1, 77, 299]:
        single, _ = orc.lookup_decode(rec, 50, d, k, rec.shape[1], lut, idx[j:j + 1])
        assert np.array_equal(single[0], out[j])
    dup = np.nonzero(idx == idx[5])[0]
    assert all(np.array_equal(out[a], out[dup[0]]) for a in dup)


def test_out_of_range_ids_give_zero_rows(orc, lut):
    d, k = 64, 4
    rng = np.random.default_rng(2)
    rec = _records(rng, 10, d, k)
    idx = np.array([0, -1, 10, 3, 1 << 40, 9])
    out, bad = orc.lookup_decode(rec, 10, d, k, rec.shape[1], lut, idx)
    assert bad == 3
    assert not out[[1, 2, 4]].any()
    assert out[[0, 3, 5]].any()


@pytest.mark.parametrize("b,k", [(1.5, 3), (2, 4), (2.5, 5), (3, 6)])
@pytest.mark.parametrize("d", [256, 512, 1024])
def test_storage_bits_per_parameter(b, k, d):
    """Record bits / d = b + 16/d exactly ("how it works": one 16-bit scale per row)."""
    from trellis_row_decode_gb300.synth import record_bytes
    assert record_bytes(d, k) * 8 / d == b + 16 / d


def test_deepseek_table_size_matches_pages():
    """1.98e8 rows x 258 B = 51.08 GB, within 1% of the 50.7 GB the pages report."""
    from trellis_row_decode_gb300.synth import WORKLOADS
    w = WORKLOADS["deepseek_prefill"]
    assert w.rec_bytes == 258
    assert abs(w.table_bytes / 50.7e9 - 1) < 0.01
