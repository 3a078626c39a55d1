"""Writes tests/golden/tiny_topk.txt from the CPU oracle alone.

Run from the repository root: python tests/golden/make_golden.py
The tiny workload: 4 queries at positions 2044..2047 over 2048 keys, H=8,
D=64, f16 integers in {-3..3}, w in {0..3}, causal mask, top_k=64, seed 0.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import lid_inputs as li  # noqa: E402
import oracle  # noqa: E402


def main():
    inp = li.workload("tiny")
    idx, sc = oracle.topk_inputs(inp)
    path = os.path.join(ROOT, "tests", "golden", "tiny_topk.txt")
    with open(path, "w") as f:
        f.write("# CPU-oracle top-64 of the tiny workload (seed 0); written by make_golden.py\n")
        for t in range(inp.n_q):
            f.write(f"idx{t}: " + " ".join(str(int(x)) for x in idx[t]) + "\n")
            f.write(f"score{t}: " + " ".join(repr(float(x)) for x in sc[t]) + "\n")


if __name__ == "__main__":
    main()
