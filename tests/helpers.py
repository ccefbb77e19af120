"""Comparison helpers shared by the GPU parity tests."""

import numpy as np
import torch

# Tolerances against the fp64 oracle on identical seeded fp16 inputs.
O_ATOL = 2e-3     # forward output, max-abs
LSE_ATOL = 1e-4   # log-sum-exp, max-abs
GRAD_RTOL = 1e-2  # dQ, dK, dV relative Frobenius error

# bf16 inputs and outputs: the roundings that reach O and the gradients (P,
# dS and the outputs themselves) have a unit roundoff 2^-8 instead of 2^-11,
# so the fp16 output tolerance is scaled by 8.  lse comes from fp32 scores of
# exactly representable inputs and keeps its tolerance.  The gradient bound
# stays 1e-2.  Measured on GB300 (N 256-512, D 64-256): O max-abs up to
# 8.4e-3 (causal), gradients' relative error 2.3-2.5e-3, 8x the fp16 ones.
O_ATOL_BF16 = 8 * O_ATOL
GRAD_RTOL_BF16 = GRAD_RTOL


def max_abs(gpu: torch.Tensor, ref: np.ndarray) -> float:
    return float(np.max(np.abs(gpu.detach().double().cpu().numpy() - ref)))


def rel_fro(gpu: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu.detach().double().cpu().numpy()
    return float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))


def sample_heads(heads: int, k: int = 6):
    """Head indices spread over the whole range, first and last included."""
    if heads <= k:
        return list(range(heads))
    return sorted(set(int(round(x)) for x in np.linspace(0, heads - 1, k)))
