"""Write ``nf4_codebook.txt``: the 16 NormalFloat levels as float32.

Calls only the oracle.  Run from the repository root:
``python tests/golden/make_nf4_codebook.py``.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import nf4_codebook  # noqa: E402


def main():
    cb = nf4_codebook()
    lines = ["# NormalFloat-4 levels (QLoRA construction), float32, ascending.",
             "# Written by make_nf4_codebook.py from oracle.nf4_codebook().",
             "# index  float32_bits  value"]
    for i, v in enumerate(cb):
        bits = int(np.float32(v).view(np.uint32))
        lines.append(f"{i:2d} 0x{bits:08x} {float(v):.9g}")
    with open(os.path.join(HERE, "nf4_codebook.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
