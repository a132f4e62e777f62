"""Write gumbel_regression.txt: (seed, layer, head, position) -> hash -> g.

A regression fixture for the oracle's frozen Gumbel values, not a pin from the
pages (they give no formula for the hash). It calls only the oracle:

    python tests/golden/make_gumbel_regression.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CASES = [(seed, layer, head, pos)
         for seed in (0, 1234, 2**63 + 5)
         for layer, head in ((0, 0), (1, 0), (0, 1), (31, 7), (27, 3))
         for pos in (0, 1, 4095, 123456)]


def main():
    out = os.path.join(HERE, "gumbel_regression.txt")
    with open(out, "w") as f:
        f.write("# Regression fixture (not a pin from the pages): the oracle's frozen Gumbel\n"
                "# values. Columns: seed layer head position hash(hex) g(float32 bits, hex).\n"
                "# Written by make_gumbel_regression.py from oracle/ alone.\n")
        for seed, layer, head, pos in CASES:
            h = oracle.gumbel_hash(seed, layer, head, pos)
            g = oracle.gumbel(seed, layer, head, pos, 1)
            f.write(f"{seed} {layer} {head} {pos} {h:016x} {int(g.view(np.uint32)[0]):08x}\n")


if __name__ == "__main__":
    main()
