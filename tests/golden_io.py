"""Loaders for the hand-worked fixtures under tests/golden/."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def hexbytes(s):
    return np.frombuffer(bytes.fromhex(s), dtype=np.uint8)


def nf4_codebook_fixture():
    """The frozen float32 NormalFloat levels, read from their bit patterns."""
    bits = []
    with open(os.path.join(GOLDEN, "nf4_codebook.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            bits.append(int(line.split()[1], 16))
    return np.asarray(bits, dtype=np.uint32).view(np.float32)
