"""Write tests/golden/tiny_encoded_rows.txt with the CPU oracle.

The tiny workload carries 64 N(0,1) rows (d = 256, b = 2) compressed by the
oracle's two-pass tail-biting Viterbi encoder; the GPU parity tests decode
these records and check the round trip.  Each line: the AoS record in hex
(64 code bytes + bf16 alpha, little-endian), the alpha before bf16 rounding
(repr), and the search cost.  Run from the repo root:
    python tests/golden/make_golden.py
"""
from pathlib import Path
import sys

import numpy as np

ROOT = Path(__file__).resolve().parents[2]
sys.path.insert(0, str(ROOT))

import oracle  # noqa: E402
from trellis_row_decode_gb300 import synth  # noqa: E402

OUT = Path(__file__).resolve().parent / "tiny_encoded_rows.txt"
D, K, ROWS = 256, 4, 64


def compute():
    lut = np.fromfile(ROOT / "trellis_row_decode_gb300" / "data" / "cp_lut_v2_l16_512.bin",
                      dtype="<u2").reshape(512, 2)
    e = synth.normal_rows(synth.SEED_ENCODER_ROWS, ROWS, D)
    return oracle.encode_rows(e, D, K, lut, oracle.TWO_PASS)


def render(rec, alpha, cost) -> str:
    lines = [f"# d={D} k={K} rows={ROWS} seed={synth.SEED_ENCODER_ROWS} two-pass Viterbi"]
    for r, a, c in zip(rec, alpha, cost):
        lines.append(f"{bytes(r).hex()} {float(a)!r} {float(c)!r}")
    return "\n".join(lines) + "\n"


def load(path: Path = OUT):
    rec, alpha, cost = [], [], []
    for line in path.read_text().splitlines():
        if line.startswith("#"):
            continue
        h, a, c = line.split()
        rec.append(np.frombuffer(bytes.fromhex(h), dtype=np.uint8))
        alpha.append(float(a))
        cost.append(float(c))
    return np.stack(rec), np.array(alpha), np.array(cost)


if __name__ == "__main__":
    OUT.write_text(render(*compute()))
    print(f"wrote {OUT}")
