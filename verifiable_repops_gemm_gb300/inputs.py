"""Seeded synthetic inputs with the shapes and value distributions of the
workloads (order-fixed GEMM sweep, decoder-layer GEMM set, contributor
gradients, tensors to commit).

This module holds no arithmetic of the method: it only draws random numbers.
Tests feed the same buffers to the CUDA library and to the oracle.

Recipes (seed -> tensor), all float32:
  uniform_pm1(shape, seed)  U[-1, 1): torch.rand * 2 - 1 (exact: rand returns
                            multiples of 2^-24)
  normal(shape, std, seed)  N(0, std^2): torch.randn * std
  contributor_ids(n, seed)  n random 32-byte identifiers (numpy PCG64)
Generation runs on the device the tensor is requested on; a given
(seed, device type) always gives the same values.
"""
import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def uniform_pm1(shape, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    return x.mul_(2.0).sub_(1.0)


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def contributor_ids(n: int, seed: int, nbytes: int = 32):
    rng = np.random.default_rng(int(seed))
    return [rng.bytes(nbytes) for _ in range(n)]


def integer_matrix(shape, lo: int, hi: int, seed: int, device="cpu") -> torch.Tensor:
    """Integers in [lo, hi] stored as float32 (exact-sum inputs)."""
    g = _gen(seed, device)
    return torch.randint(lo, hi + 1, shape, generator=g, device=device).to(torch.float32)


# Workload shapes -----------------------------------------------------------

SQUARE_SWEEP = (1024, 2048, 4096, 8192)
RAGGED = (4097, 1023, 3001)            # M, N, K
DECODER_TOKENS, DECODER_DIM = 4096, 2048
# (name, K = input dim, N = output dim): QKV (32 q heads + 2 x 8 kv heads of
# dim 64 = 3072), O, MLP up, MLP gate, MLP down
DECODER_LAYERS = (("qkv", 2048, 3072), ("o", 2048, 2048), ("up", 2048, 8192),
                  ("gate", 2048, 8192), ("down", 8192, 2048))
MEAN_CONTRIBUTORS, MEAN_LEN = 16, 1 << 28
MERKLE_ELEMS, MERKLE_LEAF = 1 << 30, 4096
