"""Seeded synthetic inputs shaped like the BitNet b1.58 workloads.

This module only draws random numbers; it holds none of the method's
arithmetic.  Tests feed the same host arrays to the CPU oracle and to the CUDA
library, so no random stream has to match across languages.

Recipe (all from a torch.Generator seeded with `seed`):
  * weights  : binary32 N(0, 0.02), shape [N, K] (out x in), drawn first;
  * tokens   : bf16 N(0, 1), shape [M, K] (binary32 draw rounded to bf16);
  * outliers : optional, a fraction `outlier_frac` of token entries (drawn
               after the values) is set to +-outlier_sigma.
A `device` of "cuda" draws with the device generator instead (used only for
the large benchmark weight sets, which the oracle never sees in full).
"""
import numpy as np
import torch

WEIGHT_STD = 0.02


def weights_f32(N: int, K: int, seed: int, std: float = WEIGHT_STD, device="cpu"):
    g = torch.Generator(device=device).manual_seed(seed)
    w = torch.randn((N, K), generator=g, dtype=torch.float32, device=device) * std
    return w if device != "cpu" else w.numpy()


def tokens_bf16(M: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_sigma: float = 20.0, device="cpu"):
    """bf16 activations as uint16 bit patterns (numpy) or a torch bf16 tensor
    on `device`."""
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn((M, K), generator=g, dtype=torch.float32, device=device)
    if outlier_frac > 0:
        pick = torch.rand((M, K), generator=g, device=device) < outlier_frac
        sign = torch.where(torch.rand((M, K), generator=g, device=device) < 0.5, -1.0, 1.0)
        x = torch.where(pick, sign * outlier_sigma, x)
    xb = x.to(torch.bfloat16)
    if device != "cpu":
        return xb
    return xb.view(torch.int16).numpy().view(np.uint16)


def ternary_codes(N: int, K: int, seed: int, zero_frac: float = 0.31):
    """Ternary weights drawn directly (int8 in {-1, 0, +1}; a fraction
    zero_frac of zeros, the rest +-1 with equal odds): a cheap stand-in for
    absmean-quantised N(0, sigma) weights, whose zero fraction is about 0.31,
    for tests that need many large matrices on the host."""
    g = torch.Generator().manual_seed(seed)
    u = torch.rand((N, K), generator=g)
    q = torch.where(u < zero_frac, 0, torch.where(u < (1 + zero_frac) / 2, -1, 1))
    return q.to(torch.int8).numpy()


def weight_scale(seed: int):
    """A positive binary32 scale near the absmean of N(0, 0.02) weights."""
    g = torch.Generator().manual_seed(seed)
    return np.float32(0.016 * (1.0 + 0.05 * torch.rand(1, generator=g).item()))


def gain_ones(H: int):
    return np.ones(H, np.float32)


def gain_random(H: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    return (1.0 + 0.1 * torch.randn(H, generator=g)).numpy().astype(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to binary32 (exact; a bit shift)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (nearest-even) via torch; input helper."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
