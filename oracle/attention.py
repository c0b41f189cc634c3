"""Float64 oracle of the tensor-parallel self-attention block (test infrastructure only).

Method (the parallel multi-head attention code of the SenseParrots model-parallel note,
section 2.1.1, and the "Attention 层" section of the "Megatron 训练" notes): X [b, s, h] ->
QKV = X W_qkv with W_qkv [h, 3h] (column-parallel: shard i owns heads i*a/t .. (i+1)*a/t - 1),
each head's columns laid out as [q | k | v] x head_dim, heads one after another; per head
S = Q K^T * head_dim^-1/2, P = softmax(S) over the keys, O_head = P V; O concatenates the heads
to [b, s, h]; Y = O W_o with W_o [h, h] (row-parallel: shard i owns the rows of its heads, the
partial products are summed).

Readings where the pages are silent: no attention mask (the SenseParrots code applies none);
attention and projection dropout left out (probability 0 here); no biases.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _split_heads(QKV, heads: int):
    b, s, three_h = QKV.shape
    dh = three_h // (3 * heads)
    r = QKV.reshape(b, s, heads, 3, dh)
    return [np.transpose(r[:, :, :, c, :], (0, 2, 1, 3)) for c in range(3)]  # each [b, a, s, dh]


def softmax(S):
    S = _f64(S)
    e = np.exp(S - S.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def forward(X, Wqkv, Wo, heads: int) -> dict[str, np.ndarray]:
    """Unsharded forward; returns QKV [b,s,3h], P [b,a,s,s], O [b,s,h], Y [b,s,h]."""
    X, Wqkv, Wo = _f64(X), _f64(Wqkv), _f64(Wo)
    b, s, _ = X.shape
    width = Wqkv.shape[1] // 3          # heads * head_dim (h, or h/t on one shard)
    dh = width // heads
    QKV = X @ Wqkv
    q, k, v = _split_heads(QKV, heads)
    P = softmax(q @ np.swapaxes(k, -1, -2) * dh ** -0.5)
    O = np.transpose(P @ v, (0, 2, 1, 3)).reshape(b, s, width)
    return {"QKV": QKV, "P": P, "O": O, "Y": O @ Wo}


def backward(X, Wqkv, Wo, heads: int, G) -> dict[str, np.ndarray]:
    """Gradients from G = dl/dY: dX, dWqkv, dWo (and dQKV, dO)."""
    X, Wqkv, Wo, G = _f64(X), _f64(Wqkv), _f64(Wo), _f64(G)
    b, s, h = X.shape
    dh = h // heads
    f = forward(X, Wqkv, Wo, heads)
    q, k, v = _split_heads(f["QKV"], heads)
    P = f["P"]
    dO = G @ Wo.T                                                    # [b, s, h]
    dWo = f["O"].reshape(b * s, h).T @ G.reshape(b * s, h)
    dOh = np.transpose(dO.reshape(b, s, heads, dh), (0, 2, 1, 3))    # [b, a, s, dh]
    dv = np.swapaxes(P, -1, -2) @ dOh
    dP = dOh @ np.swapaxes(v, -1, -2)
    dS = P * (dP - (dP * P).sum(axis=-1, keepdims=True)) * dh ** -0.5
    dq = dS @ k
    dk = np.swapaxes(dS, -1, -2) @ q
    dQKV = np.stack([np.transpose(x, (0, 2, 1, 3)) for x in (dq, dk, dv)], axis=3).reshape(b, s, 3 * h)
    dX = dQKV @ Wqkv.T
    dWqkv = X.reshape(b * s, h).T @ dQKV.reshape(b * s, 3 * h)
    return {"dX": dX, "dWqkv": dWqkv, "dWo": dWo, "dQKV": dQKV, "dO": dO}


def forward_sharded(X, Wqkv, Wo, heads: int, t: int) -> np.ndarray:
    """The t-rank computation: rank i runs its heads with its column block of W_qkv and its row
    block of W_o; the partial outputs are summed in rank order (the row layer's all-reduce)."""
    X, Wqkv, Wo = _f64(X), _f64(Wqkv), _f64(Wo)
    h = X.shape[-1]
    if heads % t:
        raise ValueError(f"{heads} heads do not split evenly over {t} shards")
    hp = heads // t
    cq, co = 3 * h // t, h // t
    Y = None
    for i in range(t):
        part = forward(X, Wqkv[:, i * cq:(i + 1) * cq], np.eye(co), hp)["O"] @ Wo[i * co:(i + 1) * co, :]
        Y = part if Y is None else Y + part
    return Y
