"""Write the shared reconstruction LUT of the CP trellis code as a data file.

The pages state that the reconstruction rule is stored once for the whole table
("2비트 코드와 공유 트렐리스로 n-gram 룩업 테이블을 4~8배 압축한다", section
어떻게 동작하나) and that the code is a Gaussian HYB bitshift trellis (section
무엇과 다른가).  They do not print the LUT; this format fixes it as 512 fp16
2-vectors from seeded Lloyd k-means (50 iterations) on 2^20 N(0,1) pairs drawn
by SplitMix64 + Box-Muller, initialised with the first 512 pairs, then rounded
to fp16 (ties to even).

Layout of the file: 512 entries x (y0, y1), fp16 little-endian, 2048 bytes.
Both the oracle and the CUDA library read this file; neither regenerates it at
run time.  Usage:  python -m oracle.make_lut [--check]
"""
from __future__ import annotations

import argparse
import hashlib
import sys
from pathlib import Path

import numpy as np

import oracle

LUT_SEED = 0x5EED
LUT_PAIRS = 1 << 20
LUT_ENTRIES = 512
LUT_ITERS = 50
LUT_PATH = (Path(__file__).resolve().parent.parent / "trellis_row_decode_gb300" / "data"
            / "cp_lut_v2_l16_512.bin")


def generate(n_threads: int | None = None):
    cent, lut, mse = oracle.lloyd_lut(LUT_SEED, LUT_PAIRS, LUT_ENTRIES, LUT_ITERS, n_threads)
    return cent, lut, mse


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--check", action="store_true", help="compare with the committed file")
    args = ap.parse_args()
    _, lut, mse = generate()
    blob = lut.astype("<u2").tobytes()
    print(f"mse/coord={mse:.6g} sha256={hashlib.sha256(blob).hexdigest()}")
    if args.check:
        ok = LUT_PATH.read_bytes() == blob
        print("match" if ok else "MISMATCH")
        return 0 if ok else 1
    LUT_PATH.parent.mkdir(parents=True, exist_ok=True)
    LUT_PATH.write_bytes(blob)
    print(f"wrote {LUT_PATH}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
