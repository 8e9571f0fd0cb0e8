"""The standard NF4 codebook for callers of the library.

The GEMV and the quantiser take the 16 levels as an argument; this helper
builds the usual NormalFloat-4 set (QLoRA, Dettmers et al. 2023): normal
quantiles taken asymmetrically so that zero is a level -- 8 positive levels
from probabilities evenly spaced from ``delta`` to 1/2 (9 points, 1/2
dropped), 7 negative ones likewise (8 points), plus 0 -- divided by the
largest so the ends are -1 and +1, with
``delta = 1 - (1/(2*15) + 1/(2*16)) / 2``.  The inverse normal CDF is
``torch.special.ndtri`` in float64.
"""
import torch


def normal_float_levels():
    """16 ascending float32 levels as a CPU tensor."""
    delta = 1.0 - 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    pos = torch.special.ndtri(torch.linspace(delta, 0.5, 9, dtype=torch.float64)[:-1])
    neg = -torch.special.ndtri(torch.linspace(delta, 0.5, 8, dtype=torch.float64)[:-1])
    top = pos.max()
    lv = torch.cat([pos / top, torch.zeros(1, dtype=torch.float64), neg / top])
    return torch.sort(lv).values.to(torch.float32)
