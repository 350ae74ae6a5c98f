"""Reader for the hand-written hex fixtures under tests/golden/."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_hex(name):
    """Bytes of a fixture: whitespace-separated hex pairs; '#' starts a comment."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0]
            out += [int(tok, 16) for tok in line.split()]
    return np.asarray(out, dtype=np.uint8)
