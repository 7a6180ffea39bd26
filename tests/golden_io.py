"""Reader for the hand-packed block fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_block_cases(fname):
    cases, cur = [], None
    with open(os.path.join(GOLDEN, fname)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
                cases.append(cur)
            elif key == "bytes":
                cur["bytes"] = np.array([int(v, 16) for v in rest.split()], dtype=np.uint8)
            elif key == "expect":
                cur["expect"] = np.array([float(v) for v in rest.split()], dtype=np.float64)
    return cases
