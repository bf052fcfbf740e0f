"""Shared helpers of the GPU tests: tables built on the device from the seeded
generators, oracle results computed from the same rows regenerated on the host."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import trellis_row_decode_gb300 as cp
from trellis_row_decode_gb300 import synth

NT = max(1, os.cpu_count() or 1)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def device_table(seed: int, n_rows: int, d: int, k: int, pad: int = 0) -> torch.Tensor:
    """Flat uint8 device buffer of n_rows AoS records (+ pad bytes)."""
    buf = torch.empty(n_rows * synth.record_bytes(d, k) + pad, dtype=torch.uint8, device="cuda")
    synth.fill_records(buf, seed, n_rows, d, k)
    return buf


def oracle_decode(seed: int, d: int, k: int, idx: np.ndarray, n_rows: int, lut) -> np.ndarray:
    """Oracle output for lookups idx on the synthetic table (rows regenerated on the host)."""
    idx = np.asarray(idx, dtype=np.int64)
    valid = (idx >= 0) & (idx < n_rows)
    uniq, inv = np.unique(np.where(valid, idx, 0), return_inverse=True)
    rec = synth.gen_records(seed, torch.from_numpy(uniq), d, k).numpy()
    local = np.where(valid, inv, -1).astype(np.int64)
    out, _ = oracle.lookup_decode(rec, len(uniq), d, k, rec.shape[1], lut, local, n_threads=NT)
    return out


def compare(got: np.ndarray, ref: np.ndarray) -> tuple[int, int]:
    """(# deviating elements, max ulp distance) between bf16 bit arrays; NaNs match NaNs."""
    g = got.astype(np.int32)
    r = ref.astype(np.int32)
    gnan = ((g & 0x7FFF) > 0x7F80)
    rnan = ((r & 0x7FFF) > 0x7F80)
    diff = (g != r) & ~(gnan & rnan)
    if not diff.any():
        return 0, 0
    # ulp distance on the monotone integer line of bf16
    def line(x):
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return int(diff.sum()), int(np.abs(line(g) - line(r))[diff].max())
