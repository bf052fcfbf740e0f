"""Seeded synthetic workloads for the CP lookup-decode: codes, scales, index streams.

This module holds input generators only -- none of the decode arithmetic.  The
same functions feed the CUDA path (tables built on the device) and the CPU
oracle (the same rows regenerated on the host), so every generator here is
counter-based and exact in integer arithmetic, or (the Zipf sampler) runs once
on the host and is shared as an array.

Recipes (the stand-ins for the pages' DeepSeek-tokenised web-text replay, which
is not available here):
  * code bits: uniform, 32-bit words from Wellons' "lowbias32" integer hash
    keyed by (seed, row, word);
  * alpha: lognormal(0, 0.25) via a 65,536-point inverse-CDF table rounded to
    bf16, indexed by 16 hash bits of (seed, row);
  * indices: i.i.d. Zipf(s) ranks on 1..N by rejection-inversion (Hoermann &
    Derflinger 1996), mapped to rows by a seeded 4-round Feistel bijection with
    cycle-walking, so hot rows land at scattered addresses; token-major layout,
    48 ids per token.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from statistics import NormalDist

import numpy as np
import torch

MASK32 = 0xFFFFFFFF
MASK64 = 0xFFFFFFFFFFFFFFFF


# ---------------------------------------------------------------------------
# Scalar seed derivation (Python ints).
# ---------------------------------------------------------------------------

def splitmix64_int(x: int) -> int:
    """SplitMix64 output for counter value x (Steele, Lea & Flood 2014)."""
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & MASK64
    return x ^ (x >> 31)


def _subkeys(seed: int, count: int) -> list[int]:
    return [splitmix64_int((seed << 8) + i) & MASK32 for i in range(count)]


# ---------------------------------------------------------------------------
# lowbias32 on int64 tensors holding values in [0, 2^32): every product stays
# below 2^49, so the arithmetic is exact on any device.
# ---------------------------------------------------------------------------

def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    lo = x * (c & 0xFFFF)
    hi = ((x * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & MASK32


def lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _row_keys(seed: int, rows: torch.Tensor) -> torch.Tensor:
    k = _subkeys(seed, 2)
    lo = rows & MASK32
    hi = rows >> 32
    return lowbias32(lowbias32(lo ^ k[0]) ^ hi ^ k[1])


def code_bytes(d: int, k: int) -> int:
    """Bytes of one row's code: d * b / 8 with b = k / 2."""
    assert (d * k) % 16 == 0
    return d * k // 16


def record_bytes(d: int, k: int) -> int:
    """AoS record: code then one bf16 scale."""
    return code_bytes(d, k) + 2


def gen_codes(seed: int, rows: torch.Tensor, cb: int) -> torch.Tensor:
    """uint8 [len(rows), cb]: uniform code bits for the given row ids."""
    rows = rows.to(torch.int64)
    nw = (cb + 3) // 4
    k = _subkeys(seed, 3)
    wkeys = lowbias32(torch.arange(nw, dtype=torch.int64, device=rows.device) ^ k[2])
    rk = _row_keys(seed, rows)
    words = lowbias32(rk[:, None] ^ wkeys[None, :])              # [rows, nw] in [0, 2^32)
    by = torch.stack([((words >> (8 * i)) & 0xFF).to(torch.uint8) for i in range(4)], dim=-1)
    return by.reshape(rows.numel(), nw * 4)[:, :cb]


_ALPHA_TABLE: dict[float, np.ndarray] = {}


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def alpha_table(sigma: float = 0.25) -> np.ndarray:
    """65,536 bf16 bit patterns: exp(sigma * Phi^-1((u + 0.5) / 65536))."""
    if sigma not in _ALPHA_TABLE:
        nd = NormalDist()
        q = np.array([nd.inv_cdf((u + 0.5) / 65536.0) for u in range(65536)], dtype=np.float64)
        _ALPHA_TABLE[sigma] = _f32_to_bf16_bits(np.exp(sigma * q).astype(np.float32))
    return _ALPHA_TABLE[sigma]


def gen_alpha(seed: int, rows: torch.Tensor, sigma: float = 0.25) -> torch.Tensor:
    """int16 tensor holding bf16 bit patterns, lognormal(0, sigma)."""
    k = _subkeys(seed, 4)
    u = lowbias32(_row_keys(seed, rows.to(torch.int64)) ^ k[3]) >> 16
    tab = torch.from_numpy(alpha_table(sigma).view(np.int16).copy()).to(rows.device)
    return tab[u]


def gen_records(seed: int, rows: torch.Tensor, d: int, k: int) -> torch.Tensor:
    """uint8 [len(rows), R] AoS records [code][alpha bf16 LE] for the given row ids."""
    cb = code_bytes(d, k)
    rec = torch.empty((rows.numel(), cb + 2), dtype=torch.uint8, device=rows.device)
    rec[:, :cb] = gen_codes(seed, rows, cb)
    a = gen_alpha(seed, rows).to(torch.int32) & 0xFFFF
    rec[:, cb] = (a & 0xFF).to(torch.uint8)
    rec[:, cb + 1] = (a >> 8).to(torch.uint8)
    return rec


def fill_records(buf: torch.Tensor, seed: int, n_rows: int, d: int, k: int,
                 chunk_rows: int = 1 << 20) -> None:
    """Fill a flat uint8 buffer (>= n_rows * R bytes, any device) with the table."""
    R = record_bytes(d, k)
    view = buf[: n_rows * R].view(n_rows, R)
    for r0 in range(0, n_rows, chunk_rows):
        r1 = min(n_rows, r0 + chunk_rows)
        rows = torch.arange(r0, r1, dtype=torch.int64, device=buf.device)
        view[r0:r1] = gen_records(seed, rows, d, k)


def mixed_rates(seed: int, rows: torch.Tensor) -> torch.Tensor:
    """Bits per step k in {3, 4, 5, 6} per row, uniform from hash bits (int64)."""
    k = _subkeys(seed, 6)
    return 3 + (lowbias32(_row_keys(seed, rows.to(torch.int64)) ^ k[5]) & 3)


def mixed_offsets(ks: torch.Tensor, d: int) -> torch.Tensor:
    """int64 [N + 1] byte offsets of records with rates ks (record = d*k/16 + 2 bytes)."""
    sizes = ks.to(torch.int64) * (d // 16) + 2
    off = torch.zeros(ks.numel() + 1, dtype=torch.int64, device=ks.device)
    off[1:] = torch.cumsum(sizes, 0)
    return off


def fill_mixed_records(buf: torch.Tensor, seed: int, ks: torch.Tensor, offsets: torch.Tensor,
                       d: int, chunk_rows: int = 1 << 18) -> None:
    """Write row r's record (rate ks[r]) at buf[offsets[r]:offsets[r+1]]."""
    n_rows = ks.numel()
    for r0 in range(0, n_rows, chunk_rows):
        r1 = min(n_rows, r0 + chunk_rows)
        for k in (3, 4, 5, 6):
            sel = torch.nonzero(ks[r0:r1] == k).flatten() + r0
            if sel.numel() == 0:
                continue
            rec = gen_records(seed, sel.to(torch.int64), d, k)
            R = rec.shape[1]
            dst = offsets[sel][:, None] + torch.arange(R, device=buf.device)[None, :]
            buf[dst.reshape(-1)] = rec.reshape(-1)


# ---------------------------------------------------------------------------
# Index streams (numpy, host).
# ---------------------------------------------------------------------------

def splitmix64_np(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint64) + np.uint64(0x9E3779B97F4A7C15)
    x = (x ^ (x >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    x = (x ^ (x >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return x ^ (x >> np.uint64(31))


def uniforms(seed: int, counters: np.ndarray) -> np.ndarray:
    """Doubles in [0, 1) from 53 hash bits of (seed, counter)."""
    key = np.uint64(splitmix64_int(seed))
    return (splitmix64_np(splitmix64_np(counters) ^ key) >> np.uint64(11)).astype(np.float64) \
        * (1.0 / 9007199254740992.0)


def zipf_ranks(seed: int, n: int, N: int, s: float = 1.0) -> np.ndarray:
    """n i.i.d. ranks in 1..N with P(r) proportional to r^-s (rejection-inversion)."""
    if s == 1.0:
        H = np.log
        Hinv = np.exp
    else:
        H = lambda x: (np.power(x, 1.0 - s) - 1.0) / (1.0 - s)          # noqa: E731
        Hinv = lambda u: np.power(1.0 + (1.0 - s) * u, 1.0 / (1.0 - s))  # noqa: E731
    h = lambda x: np.power(x, -s)                                        # noqa: E731
    H_x1 = H(np.float64(1.5)) - 1.0
    H_n = H(np.float64(N) + 0.5)
    s_const = 2.0 - Hinv(H(np.float64(2.5)) - h(np.float64(2.0)))
    out = np.zeros(n, dtype=np.int64)
    todo = np.arange(n, dtype=np.uint64)
    attempt = 0
    while todo.size:
        U = uniforms(seed, todo * np.uint64(64) + np.uint64(attempt))
        u = H_n + U * (H_x1 - H_n)
        x = Hinv(u)
        kk = np.clip(np.floor(x + 0.5), 1, N)
        ok = (kk - x <= s_const) | (u >= H(kk + 0.5) - h(kk))
        out[todo[ok].astype(np.int64)] = kk[ok].astype(np.int64)
        todo = todo[~ok]
        attempt += 1
        if attempt >= 64:
            raise RuntimeError("zipf sampler did not converge")
    return out


def feistel_bijection(x: np.ndarray, N: int, seed: int) -> np.ndarray:
    """Seeded bijection of [0, N): 4-round balanced Feistel on 2h bits, cycle-walking."""
    bits = max(2, int(N - 1).bit_length())
    bits += bits & 1
    half = bits // 2
    mask = np.uint64((1 << half) - 1)
    keys = [np.uint64(splitmix64_int((seed << 4) + i)) for i in range(4)]

    def perm(v: np.ndarray) -> np.ndarray:
        L = (v >> np.uint64(half)) & mask
        R = v & mask
        for kk in keys:
            F = splitmix64_np(R ^ kk) & mask
            L, R = R, L ^ F
        return (L << np.uint64(half)) | R

    y = perm(np.asarray(x, dtype=np.uint64))
    bad = y >= np.uint64(N)
    while bad.any():
        y[bad] = perm(y[bad])
        bad = y >= np.uint64(N)
    return y.astype(np.int64)


def zipf_indices(seed: int, n: int, N: int, s: float = 1.0) -> np.ndarray:
    """Row ids: Zipf ranks mapped through the seeded bijection."""
    return feistel_bijection(zipf_ranks(seed, n, N, s) - 1, N, seed)


def uniform_indices(seed: int, n: int, N: int) -> np.ndarray:
    c = splitmix64_np(np.arange(n, dtype=np.uint64) ^ np.uint64(splitmix64_int(seed)))
    return (c % np.uint64(N)).astype(np.int64)


# ---------------------------------------------------------------------------
# Named workloads.
# ---------------------------------------------------------------------------

SEED_TABLE, SEED_INDEX, SEED_ENCODER_ROWS = 1, 2, 3


@dataclass(frozen=True)
class Workload:
    name: str
    n_rows: int
    d: int
    k: int                       # bits per 2-coordinate step (2b)
    tokens: int
    rows_per_token: int
    dist: str                    # "zipf" or "uniform"
    zipf_s: float = 1.0
    residency: str = "device"
    notes: str = field(default="", compare=False)

    @property
    def n_lookups(self) -> int:
        return self.tokens * self.rows_per_token

    @property
    def rec_bytes(self) -> int:
        return record_bytes(self.d, self.k)

    @property
    def table_bytes(self) -> int:
        return self.n_rows * self.rec_bytes

    def indices(self, seed: int = SEED_INDEX) -> np.ndarray:
        if self.dist == "zipf":
            return zipf_indices(seed, self.n_lookups, self.n_rows, self.zipf_s)
        return uniform_indices(seed, self.n_lookups, self.n_rows)

    def algorithmic_bytes_per_lookup(self) -> int:
        """Record read + bf16 row written + int64 id read."""
        return self.rec_bytes + 2 * self.d + 8


DEEPSEEK_ROWS = 198_000_000

WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 4096, 256, 4, 4096, 1, "uniform"),
    "mid": Workload("mid", 1 << 24, 512, 4, 4096, 48, "zipf"),
    "sweep_b1.5": Workload("sweep_b1.5", 1 << 24, 1024, 3, 4096, 48, "zipf"),
    "sweep_b2": Workload("sweep_b2", 1 << 24, 1024, 4, 4096, 48, "zipf"),
    "sweep_b2.5": Workload("sweep_b2.5", 1 << 24, 1024, 5, 4096, 48, "zipf"),
    "sweep_b3": Workload("sweep_b3", 1 << 24, 1024, 6, 4096, 48, "zipf"),
    "deepseek_prefill": Workload("deepseek_prefill", DEEPSEEK_ROWS, 1024, 4, 4096, 48, "zipf"),
    "deepseek_decode": Workload("deepseek_decode", DEEPSEEK_ROWS, 1024, 4, 2048, 48, "zipf"),
    "host_prefill": Workload("host_prefill", DEEPSEEK_ROWS, 1024, 4, 4096, 48, "zipf",
                             residency="host"),
}


def normal_rows(seed: int, rows: int, d: int) -> np.ndarray:
    """N(0,1) rows by Box-Muller from the counter stream (inputs for the encoder)."""
    c = np.arange(rows * d, dtype=np.uint64)
    u1 = 1.0 - uniforms(seed, 2 * c)
    u2 = uniforms(seed, 2 * c + np.uint64(1))
    return (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)).reshape(rows, d)
