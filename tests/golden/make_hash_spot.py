"""Writes tests/golden/hash_spot.txt from the CPU oracle only (a regression table for the
producer values; the formula itself is this build's own definition)."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import hashfill as H  # noqa: E402

CASES = [
    ("bf16", 20261203, 0, 1, 0, 0, 256), ("bf16", 20261203, 1, 3, 255, 255, 256),
    ("bf16", 20261204, 3, 10, 4095, 4095, 4096), ("bf16", 20261204, 2, 7, 511, 0, 4096),
    ("bf16", 20261205, 7, 1, 7999, 8063, 8064), ("bf16", 20261205, 0, 10, 7936, 128, 8064),
    ("f32", 20261206, 0, 1, 0, 0, 1024), ("f32", 20261206, 7, 10, 1023, 1023, 1024),
    ("f32", 20261206, 4, 5, 128, 7, 1024), ("f32", 20261206, 5, 9, 896, 1000, 1024),
    ("u8", 20261206, 0, 1, 0, 0, 1 << 20), ("u8", 20261206, 0, 1, 2559, (1 << 20) - 1, 1 << 20),
    ("u8", 20261206, 0, 1, 1024, 0, 1 << 20), ("u8", 20261206, 0, 1, 2048, 12345, 1 << 20),
    ("bf16", 1, 0, 1, 0, 1, 2), ("bf16", 0, 0, 0, 0, 0, 1), ("f32", 0, 0, 0, 0, 0, 1),
    ("u8", 0xFFFFFFFF, 8, 4294967295, 3, 4, 5), ("bf16", 42, 2, 2, 17, 33, 200),
    ("f32", 42, 2, 2, 17, 33, 203),
]


def main():
    out = ["# Producer value spot table, written by make_hash_spot.py from oracle/hashfill.py.",
           "# dtype seed rank round row col N value(hex of the stored bits)"]
    for dtype, seed, rank, rnd, row, col, N in CASES:
        v = H.values_at(dtype, seed, rank, rnd, [row], [col], N)
        raw = v.view(np.uint8 if dtype == "u8" else (np.uint32 if dtype == "f32" else np.uint16))
        out.append(f"{dtype} {seed} {rank} {rnd} {row} {col} {N} {int(raw[0]):x}")
    with open(os.path.join(HERE, "hash_spot.txt"), "w") as f:
        f.write("\n".join(out) + "\n")


if __name__ == "__main__":
    main()
