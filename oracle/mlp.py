"""Float64 oracle of the tensor-parallel MLP block (test infrastructure only).

Notation of "024 | Megatron-LM: 按矩阵结构切分 Transformer", section 二, block
"前向少通信，反向为何仍要一次归约？": X is n x d, A is d x m split by columns into
A_i, B is m x d split by the matching rows into B_i, Z_i = X A_i, Y_i = phi(Z_i),
O = sum_i Y_i B_i, and with G = dl/dO:
    D_i = (G B_i^T) * phi'(Z_i),  dl/dA_i = X^T D_i,  dl/dB_i = Y_i^T G,
    dl/dX = sum_i D_i A_i^T.
Concatenating the shards gives the unsharded quantities, which is what the
method reaches up to rounding order; ``forward``/``backward`` therefore write the
unsharded definition out, with numpy's float64 matmul as the only library step.

The pages do not print the GeLU formula (the "激活函数" section of the
"Megatron 训练" notes only names torch.nn.functional.gelu). The reading taken:
  exact:  phi(x) = x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)),
          phi'(x) = Phi(x) + x * N(x), N the standard normal density;
  tanh:   phi(x) = x/2 * (1 + tanh(u)), u = sqrt(2/pi) * (x + 0.044715 x^3),
          phi'(x) = (1 + tanh u)/2 + x/2 * (1 - tanh^2 u) * sqrt(2/pi) * (1 + 3*0.044715 x^2),
the Hendrycks-Gimpel definition and its published tanh approximation.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

_SQRT2 = math.sqrt(2.0)
_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)
_TANH_C = 0.044715


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def gelu(x, kind: str) -> np.ndarray:
    """phi(x): exact ("erf") or tanh-approximated ("tanh") GeLU, float64."""
    x = _f64(x)
    if kind == "erf":
        return 0.5 * x * (1.0 + erf(x / _SQRT2))
    if kind == "tanh":
        return 0.5 * x * (1.0 + np.tanh(_SQRT_2_OVER_PI * (x + _TANH_C * x ** 3)))
    if kind == "relu":  # only for the counterexample of section 二 ("教学算例")
        return np.maximum(x, 0.0)
    raise ValueError(f"unknown activation {kind!r}")


def gelu_grad(x, kind: str) -> np.ndarray:
    """phi'(x) for the same variants, float64."""
    x = _f64(x)
    if kind == "erf":
        cdf = 0.5 * (1.0 + erf(x / _SQRT2))
        pdf = _INV_SQRT_2PI * np.exp(-0.5 * x * x)
        return cdf + x * pdf
    if kind == "tanh":
        th = np.tanh(_SQRT_2_OVER_PI * (x + _TANH_C * x ** 3))
        return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * _SQRT_2_OVER_PI * (1.0 + 3.0 * _TANH_C * x * x)
    if kind == "relu":
        return (x > 0.0).astype(np.float64)
    raise ValueError(f"unknown activation {kind!r}")


def forward(X, A, B, kind: str, b1=None, b2=None) -> dict[str, np.ndarray]:
    """Unsharded forward: Z = X A (+ b1), Y = phi(Z), O = Y B (+ b2), all float64.

    Biases follow the Megatron layers of the "Megatron 训练" notes: the column-parallel layer's
    bias b1 [m] is split with A's columns and added before the activation; the row-parallel
    layer's bias b2 [d] is added once, after the partial products are summed.
    """
    X, A, B = _f64(X), _f64(A), _f64(B)
    Z = X @ A
    if b1 is not None:
        Z = Z + _f64(b1)
    Y = gelu(Z, kind)
    O = Y @ B
    if b2 is not None:
        O = O + _f64(b2)
    return {"Z": Z, "Y": Y, "O": O}


def backward(X, A, B, G, kind: str, b1=None) -> dict[str, np.ndarray]:
    """Unsharded backward from G = dl/dO: D, dA = X^T D, dB = Y^T G, dX = D A^T, and the bias
    gradients db1 = sum over tokens of D, db2 = sum over tokens of G (the matmul-gradient rule
    of the "Megatron 训练" notes: a broadcast bias collects the sum of its rows' gradients)."""
    X, A, B, G = _f64(X), _f64(A), _f64(B), _f64(G)
    Z = X @ A
    if b1 is not None:
        Z = Z + _f64(b1)
    Y = gelu(Z, kind)
    D = (G @ B.T) * gelu_grad(Z, kind)
    return {"D": D, "dA": X.T @ D, "dB": Y.T @ G, "dX": D @ A.T, "db1": D.sum(axis=0), "db2": G.sum(axis=0)}


def shard_views(A, B, t: int):
    """A_i = A[:, i*m/t:(i+1)*m/t], B_i = B[i*m/t:(i+1)*m/t, :] (equal contiguous split).

    The SenseParrots note, section 2.1, states that every split is an even one; a
    width that t does not divide is rejected.
    """
    m = A.shape[1]
    if m % t:
        raise ValueError(f"m={m} is not divisible by t={t}")
    mt = m // t
    return [(A[:, i * mt:(i + 1) * mt], B[i * mt:(i + 1) * mt, :]) for i in range(t)]


def forward_sharded(X, A, B, t: int, kind: str, b1=None, b2=None) -> dict[str, np.ndarray]:
    """Per-shard forward: every shard reads the same X (f is the identity), shard i adds its
    slice of b1, and O = sum_i Y_i B_i in shard order 0..t-1 (the all-reduce of f-bar), with b2
    added once after the sum. Returns the concatenated Z_i, Y_i and the summed O."""
    X = _f64(X)
    m = _f64(A).shape[1]
    mt = m // t if t else m
    Zs, Ys, O = [], [], None
    for i, (Ai, Bi) in enumerate(shard_views(_f64(A), _f64(B), t)):
        Zi = X @ Ai
        if b1 is not None:
            Zi = Zi + _f64(b1)[i * mt:(i + 1) * mt]
        Yi = gelu(Zi, kind)
        Pi = Yi @ Bi
        O = Pi if O is None else O + Pi
        Zs.append(Zi)
        Ys.append(Yi)
    if b2 is not None:
        O = O + _f64(b2)
    return {"Z": np.concatenate(Zs, axis=1), "Y": np.concatenate(Ys, axis=1), "O": O}


def backward_sharded(X, A, B, G, t: int, kind: str, b1=None) -> dict[str, np.ndarray]:
    """Per-shard backward: D_i, dA_i, dB_i and db1_i are local; dX = sum_i D_i A_i^T is the one
    reduction the backward needs (the all-reduce in f's backward); db2 is the same on every
    shard (G is replicated)."""
    X, G = _f64(X), _f64(G)
    m = _f64(A).shape[1]
    mt = m // t
    Ds, dAs, dBs, db1s, dX = [], [], [], [], None
    for i, (Ai, Bi) in enumerate(shard_views(_f64(A), _f64(B), t)):
        Zi = X @ Ai
        if b1 is not None:
            Zi = Zi + _f64(b1)[i * mt:(i + 1) * mt]
        Yi = gelu(Zi, kind)
        Di = (G @ Bi.T) * gelu_grad(Zi, kind)
        Ds.append(Di)
        dAs.append(X.T @ Di)
        dBs.append(Yi.T @ G)
        db1s.append(Di.sum(axis=0))
        part = Di @ Ai.T
        dX = part if dX is None else dX + part
    return {"D": np.concatenate(Ds, axis=1), "dA": np.concatenate(dAs, axis=1),
            "dB": np.concatenate(dBs, axis=0), "dX": dX, "db1": np.concatenate(db1s), "db2": G.sum(axis=0)}


def forward_input_split(X, A, B, t: int, kind: str) -> np.ndarray:
    """The wrong split of section 二 ("若先把输入通道拆开..."): X split by columns and A
    by rows along d, the nonlinearity applied to each partial product before
    summing. Kept only so a test can show it differs from ``forward``."""
    X, A, B = _f64(X), _f64(A), _f64(B)
    d = X.shape[1]
    if d % t:
        raise ValueError(f"d={d} is not divisible by t={t}")
    dt = d // t
    return sum(gelu(X[:, i * dt:(i + 1) * dt] @ A[i * dt:(i + 1) * dt, :], kind) for i in range(t)) @ B
