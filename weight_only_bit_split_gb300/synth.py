"""Seeded synthetic inputs for the decode-GEMV workloads.

This module only draws numbers and rounds them to a storage dtype; it holds
none of the GEMV or quantisation arithmetic, and both the CUDA path and the
CPU oracle take their inputs from it.

Recipe: ``torch.Generator(device).manual_seed(seed)`` and ``torch.randn``
(float32), scaled by the standard deviation, then cast to the storage dtype
(fp16 / bf16 casts round to nearest even).  The seed of a tensor is
``1_000_000 * workload + 1000 * tensor + copy`` with tensor 1 = weights,
2 = activations; ``copy`` numbers the rotated weight copies.

The workloads are the decode shapes of the pages: an 8B model's
projections (4096x4096 q/o, 1024x4096 k/v, 14336x4096 gate/up, 4096x14336
down), a 70B model's MLP matrix (28672x8192), a 128000-token vocabulary
head, and the rows of the standalone argmax / argmin (logit rows of 32K to
262K entries, batched rows, a 1M-entry distance row).  Weights ~ N(0,
0.02^2), activations and logit rows ~ N(0, 1).
"""
import torch

W_STD = 0.02
X_STD = 1.0
TENSOR_W = 1
TENSOR_X = 2

# workload id -> description (id is the seed's leading term)
WORKLOADS = {
    1: dict(name="fp16_gemv_4096x4096", fmt="f16", shapes=[(4096, 4096)], M=(1,)),
    2: dict(name="q4_0_q8_1_gemv_m1_8b_shapes", fmt="q4_0",
            shapes=[(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)], M=(1,)),
    3: dict(name="nf4_gemv_28672x8192", fmt="nf4", shapes=[(28672, 8192)], M=(1,)),
    4: dict(name="q4_0_q8_1_m_sweep", fmt="q4_0", shapes=[(4096, 4096), (14336, 4096)],
            M=(1, 2, 4, 8, 12, 16, 24, 32)),
    5: dict(name="bf16_lm_head_argmax_128000x4096", fmt="bf16", shapes=[(128000, 4096)],
            M=(1, 32)),
    # standalone argmax / argmin rows (M, N): vocabulary heads of the ArgCompare
    # discussion's model table, values ~ N(0, 1) stand in for logits
    6: dict(name="argcompare_rows", fmt="argcmp",
            shapes=[(1, 128000), (32, 128000), (1, 262144), (8, 32768), (4096, 8192),
                    (64, 1048576)], M=()),
}


def seed_of(workload, tensor, copy=0):
    return 1_000_000 * int(workload) + 1000 * int(tensor) + int(copy)


def normal(shape, std, seed, device="cpu", dtype=torch.float32):
    """N(0, std^2) samples of ``shape``, drawn in float32 then cast to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t if dtype == torch.float32 else t.to(dtype)


def weights(workload, shape, copy=0, device="cpu", dtype=torch.float32):
    return normal(shape, W_STD, seed_of(workload, TENSOR_W, copy), device, dtype)


def activations(workload, shape, copy=0, device="cpu", dtype=torch.float32):
    return normal(shape, X_STD, seed_of(workload, TENSOR_X, copy), device, dtype)
