"""Float64 oracle of the sequence-parallel MLP block (test infrastructure only).

Block order ("Megatron-SP 机制", section "通信插在层内什么位置？", the MLP half of the
placement diagram): input [b, s/t, h] per shard -> LayerNorm -> g: all-gather to
[b, s, h] -> FC1 (column-parallel) -> GeLU + FC2 (row-parallel) -> g-bar:
reduce-scatter to [b, s/t, h] -> dropout + residual add.

Readings taken where the pages are silent (the LayerNorm and dropout formulas
were stripped from the "Megatron 训练" notes, sections "LayerNorm" and "Dropout"):

* LayerNorm follows torch.nn.LayerNorm, which those notes name: per token,
  mean and biased variance (divide by h) over the hidden dimension,
  y = (x - mean) / sqrt(var + eps) * gamma + beta.
* Dropout follows torch.nn.Dropout, which those notes name: p is the drop
  probability and kept elements are scaled by 1/(1-p). The mask is a counter
  hash instead of torch's RNG state: element k of the logical [b, s, h] tensor
  (row-major flat index) is dropped iff splitmix64(seed XOR k) < T with
  T = floor(p * 2^64) evaluated in double precision. Indexing by the global
  flat index makes every shard's mask different, as the RNG-domain section of
  "Megatron-SP 机制" ("Dropout 的 RNG 为什么要分域管理？") requires, and makes the
  mask independent of t.
* splitmix64 is Steele, Lea and Flood's SplitMix64 step as published by Vigna
  (splitmix64.c): add the golden-gamma increment 0x9E3779B97F4A7C15, then the
  variant-13 mixer (xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27,
  multiply 0x94D049BB133111EB, xor-shift 31), all modulo 2^64.
* The residual operand is the block input x (pre-LayerNorm), the pre-norm reading
  of the placement diagram.
"""
from __future__ import annotations

import numpy as np

from . import collectives, mlp

_GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def layernorm(x, gamma, beta, eps: float) -> np.ndarray:
    """Per-row LayerNorm over the last axis, float64, biased variance."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def splitmix64(x) -> np.ndarray:
    """Vectorised SplitMix64 output for states ``x`` (uint64 array; arithmetic mod 2^64)."""
    z = np.asarray(x, dtype=np.uint64) + np.uint64(_GOLDEN_GAMMA)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
    return z ^ (z >> np.uint64(31))


def splitmix64_scalar(x: int) -> int:
    """The same function on one Python integer, with explicit reduction mod 2^64."""
    z = (x + _GOLDEN_GAMMA) & _MASK64
    z = ((z ^ (z >> 30)) * _MIX1) & _MASK64
    z = ((z ^ (z >> 27)) * _MIX2) & _MASK64
    return z ^ (z >> 31)


def drop_threshold(p: float) -> int:
    """T = floor(p * 2^64) with the product taken in double precision; 0 <= p < 1."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(float(p) * 18446744073709551616.0)


def drop_mask(flat_index, seed: int, p: float) -> np.ndarray:
    """True where the element with this global flat index is dropped."""
    k = np.asarray(flat_index, dtype=np.uint64) ^ np.uint64(seed & _MASK64)
    return splitmix64(k) < np.uint64(drop_threshold(p))


def pack_mask_bits(dropped: np.ndarray) -> np.ndarray:
    """Pack a flat boolean mask into uint32 words: bit i of word w is element 32*w + i."""
    flat = np.asarray(dropped, dtype=bool).reshape(-1)
    nwords = (flat.size + 31) // 32
    padded = np.zeros(nwords * 32, dtype=np.uint64)
    padded[:flat.size] = flat
    weights = np.uint64(1) << np.arange(32, dtype=np.uint64)
    return (padded.reshape(nwords, 32) * weights).sum(axis=1).astype(np.uint32)


def dropout_residual(x, y, seed: int, p: float, flat_index) -> np.ndarray:
    """out = x + (1 - drop) * y / (1 - p), float64."""
    dropped = drop_mask(flat_index, seed, p)
    scale = 1.0 / (1.0 - p)
    return np.asarray(x, np.float64) + np.where(dropped, 0.0, np.asarray(y, np.float64) * scale)


def sp_block(x, gamma, beta, eps, A, B, p: float, seed: int, kind: str) -> dict[str, np.ndarray]:
    """Unsharded composition on the logical [b, s, h] tensor (every step acts per token,
    so sharding along s only relabels rows). Returns LN output, MLP output o,
    block output and the drop mask, all in token order."""
    x = np.asarray(x, np.float64)
    b, s, h = x.shape
    rows = x.reshape(b * s, h)
    xn = layernorm(rows, gamma, beta, eps)
    o = mlp.forward(xn, A, B, kind)["O"]
    flat = np.arange(b * s * h, dtype=np.uint64).reshape(b * s, h)
    out = dropout_residual(rows, o, seed, p, flat)
    return {"xn": xn.reshape(b, s, h), "o": o.reshape(b, s, h), "out": out.reshape(b, s, h),
            "dropped": drop_mask(flat, seed, p).reshape(b, s, h)}


def sp_block_ranks(x_shards, gamma, beta, eps, A, B, p: float, seed: int, kind: str) -> np.ndarray:
    """The same block run the way t sequence/tensor-parallel ranks run it: per-rank
    LayerNorm on its [b, s/t, h] shard, all-gather along s, rank i computes the
    partial Y_i B_i on the full sequence, reduce-scatter along s, per-rank dropout
    (global flat indices) and residual. Returns the output shards [t, b, s/t, h]."""
    xs = [np.asarray(a, np.float64) for a in x_shards]
    t = len(xs)
    b, sl, h = xs[0].shape
    s = sl * t
    ln = [layernorm(a, gamma, beta, eps) for a in xs]
    gathered = collectives.all_gather(ln, axis=1)          # each rank: [b, s, h]
    partials = []
    for i, (Ai, Bi) in enumerate(mlp.shard_views(np.asarray(A, np.float64), np.asarray(B, np.float64), t)):
        Zi = gathered[i].reshape(b * s, h) @ Ai
        partials.append((mlp.gelu(Zi, kind) @ Bi).reshape(b, s, h))
    o_shards = collectives.reduce_scatter(partials, axis=1)  # rank j: [b, s/t, h]
    out = []
    for j in range(t):
        bi = np.arange(b, dtype=np.uint64)[:, None, None]
        li = np.arange(sl, dtype=np.uint64)[None, :, None]
        hi = np.arange(h, dtype=np.uint64)[None, None, :]
        flat = (bi * np.uint64(s) + np.uint64(j * sl) + li) * np.uint64(h) + hi
        out.append(dropout_residual(xs[j], o_shards[j], seed, p, flat))
    return np.stack(out)


def layernorm_backward(x, gamma, eps: float, dy):
    """Gradients of y = LayerNorm(x) * gamma + beta (per row, biased variance) given dy.

    Returns dx, dgamma (summed over rows), dbeta (summed over rows). With g = dy * gamma and
    x_hat the normalised row, dx = (g - mean(g) - x_hat * mean(g * x_hat)) / sqrt(var + eps):
    the gradient loses its components along 1 and along x_hat, as the "Megatron 训练" notes
    describe in their LayerNorm section (the formulas themselves were stripped).
    """
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mean) * rstd
    g = dy * np.asarray(gamma, np.float64)
    dx = rstd * (g - g.mean(axis=-1, keepdims=True) - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    lead = tuple(range(x.ndim - 1))
    return dx, (dy * xhat).sum(axis=lead), dy.sum(axis=lead)


def sp_block_backward(x, gamma, beta, eps, A, B, p: float, seed: int, kind: str, G_out) -> dict[str, np.ndarray]:
    """Backward of ``sp_block`` on the logical [b, s, h] tensor, from G_out = dl/d out.

    Chain (the SP backward of the "Efficient Large-Scale ... Megatron-LM" notes, section 3.5.1,
    run per token): the residual passes G_out to x; dropout passes G_out * keep / (1 - p) to
    the MLP output; the MLP backward gives dA, dB and the gradient at the LayerNorm output;
    LayerNorm's backward adds its part to dx and gives dgamma, dbeta.
    """
    x = np.asarray(x, np.float64)
    b, s, h = x.shape
    rows = x.reshape(b * s, h)
    G = np.asarray(G_out, np.float64).reshape(b * s, h)
    xn = layernorm(rows, gamma, beta, eps)
    flat = np.arange(b * s * h, dtype=np.uint64).reshape(b * s, h)
    keep = ~drop_mask(flat, seed, p)
    do = np.where(keep, G * (1.0 / (1.0 - p)), 0.0)
    grads = mlp.backward(xn, A, B, do, kind)
    dx_ln, dgamma, dbeta = layernorm_backward(rows, gamma, eps, grads["dX"])
    return {"dx": (G + dx_ln).reshape(b, s, h), "dgamma": dgamma, "dbeta": dbeta, "dA": grads["dA"],
            "dB": grads["dB"], "do": do.reshape(b, s, h), "dxn": grads["dX"].reshape(b, s, h)}
