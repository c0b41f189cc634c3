"""Float64 oracle of RMSNorm and its gradient (test infrastructure only).

Method: the "RMSNorm" section of the "Megatron 训练" notes. RMSNorm is LayerNorm with the mean
computation removed; only the scale is controlled, because shift invariance is mostly redundant
in a Transformer. The page's formula was stripped. This reading keeps everything else of the
LayerNorm reading used for the SP block: per row of h elements, the mean square over the hidden
dimension (divide by h), eps inside the square root, a per-column gain gamma and no bias:

    r = 1 / sqrt(mean(x^2) + eps),   y = x * r * gamma.

Backward, from dy: with x_hat = x * r and g = dy * gamma,

    dx = r * (g - x_hat * mean(g * x_hat)),   dgamma = sum over rows of dy * x_hat.

Only the component along x_hat is removed (the mean direction stays, unlike LayerNorm's
gradient), since RMSNorm no longer subtracts the mean.
"""
from __future__ import annotations

import numpy as np


def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * gamma per row (last axis), float64."""
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    return x * r * np.asarray(gamma, np.float64)


def rmsnorm_backward(x, gamma, eps: float, dy):
    """Returns dx and dgamma (summed over all leading axes) of y = rmsnorm(x, gamma, eps)."""
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    xhat = x * r
    g = dy * np.asarray(gamma, np.float64)
    dx = r * (g - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    lead = tuple(range(x.ndim - 1))
    return dx, (dy * xhat).sum(axis=lead)
