"""Write the stored expected values that come from the oracle.

Calls only the CPU oracle (``oracle/``).  Run from the repository root:

    python tests/golden/make_golden.py

It writes ``probe_hash.txt``: the probe hash (the seeded 1024 x 1024 x 1024
block-scaled int8 GEMM without ReLU, hashed to 32 bytes) for a few seeds, and
a few small shapes, so that a GPU run can be checked against fixed bytes.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CASES = [
    (0, 1024, 1024, 1024),
    (1, 1024, 1024, 1024),
    (0, 1, 1, 1),
    (7, 17, 5, 33),
    (123456789, 300, 257, 1100),
]


def main():
    orc = oracle.load()
    lines = ["# probe hash written by tests/golden/make_golden.py from the CPU oracle",
             "# the kernel probe of \"Verification -- why you can trust the numbers\",",
             "# section \"Layer 3: the kernel probe\"; the page fixes neither the inputs",
             "# nor the hash, so these follow the oracle's readings: SplitMix64 inputs",
             "# in [-1, 1), a BLAKE2s-256 tree over C's little-endian f32 bytes",
             "# format: <seed> <M> <N> <K> <hash hex>"]
    for seed, M, N, K in CASES:
        h, st = orc.probe_hash(seed, M, N, K)
        assert st == 0
        lines.append(f"{seed} {M} {N} {K} {h.hex()}")
    with open(os.path.join(HERE, "probe_hash.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")
    print("\n".join(lines))


if __name__ == "__main__":
    main()
