"""Checks of the seeded input generators (shared by the CUDA path and the oracle)."""
import numpy as np
import torch

from trellis_row_decode_gb300 import synth


def test_lowbias32_matches_python_ints():
    def ref(x):
        x ^= x >> 16
        x = (x * 0x7FEB352D) & 0xFFFFFFFF
        x ^= x >> 15
        x = (x * 0x846CA68B) & 0xFFFFFFFF
        return x ^ (x >> 16)
    xs = [0, 1, 2, 0xFFFFFFFF, 0x12345678, 0x80000000, 987654321]
    got = synth.lowbias32(torch.tensor(xs, dtype=torch.int64)).tolist()
    assert got == [ref(x) for x in xs]


def test_records_are_row_local_and_deterministic():
    rows = torch.tensor([0, 5, 123456789012, 7], dtype=torch.int64)
    a = synth.gen_records(1, rows, 1024, 4)
    b = synth.gen_records(1, rows[[2]], 1024, 4)
    assert torch.equal(a[2], b[0])
    assert a.shape == (4, 258)
    assert not torch.equal(synth.gen_records(2, rows, 1024, 4), a)


def test_code_bits_look_uniform():
    c = synth.gen_codes(1, torch.arange(2000), 256).numpy()
    bits = np.unpackbits(c)
    assert abs(bits.mean() - 0.5) < 0.002


def test_alpha_lognormal():
    a = synth.gen_alpha(1, torch.arange(200000)).view(torch.bfloat16).float().numpy()
    la = np.log(a)
    assert abs(la.mean()) < 0.005 and abs(la.std() - 0.25) < 0.005


def test_fill_records_matches_gen_records():
    d, k, n = 256, 6, 1000
    buf = torch.empty(n * synth.record_bytes(d, k) + 16, dtype=torch.uint8)
    synth.fill_records(buf, 9, n, d, k, chunk_rows=300)
    view = buf[: n * synth.record_bytes(d, k)].view(n, -1)
    assert torch.equal(view[[0, 299, 300, 999]], synth.gen_records(9, torch.tensor([0, 299, 300, 999]), d, k))


def test_zipf_frequencies_match_closed_form():
    N = 1 << 20
    r = synth.zipf_ranks(4, 400000, N)
    HN = np.sum(1.0 / np.arange(1, N + 1))
    for rank in [1, 2, 3, 10]:
        p = 1.0 / (rank * HN)
        obs = np.mean(r == rank)
        assert abs(obs - p) < 5 * np.sqrt(p * (1 - p) / r.size), rank
    assert r.min() >= 1 and r.max() <= N


def test_feistel_is_a_bijection():
    for N in [1, 2, 7, 1000, 4096, 12345]:
        p = synth.feistel_bijection(np.arange(N), N, 3)
        assert np.array_equal(np.sort(p), np.arange(N))


def test_replay_shapes():
    w = synth.WORKLOADS["mid"]
    idx = w.indices()
    assert idx.shape == (196608,) and idx.dtype == np.int64
    assert idx.min() >= 0 and idx.max() < w.n_rows
    u = synth.WORKLOADS["tiny"].indices()
    assert len(np.unique(u)) < u.size         # duplicates present
