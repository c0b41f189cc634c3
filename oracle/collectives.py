"""Host "ranks" for the three collectives of tensor and sequence parallelism (test infrastructure only).

A rank's buffer is one numpy array; a collective takes the list of every rank's
buffer and returns the list of what each rank holds afterwards. Sums run in rank
order 0..t-1, one addition at a time, in the buffers' own dtype, so that the
identity AllReduce(x) = AllGather(ReduceScatter(x)) of "Megatron-SP 机制"
(section "f/g 算子怎么定义？", the AR identity equation) can be checked bit for bit.
"""
from __future__ import annotations

import numpy as np


def _ordered_sum(parts):
    acc = parts[0].copy()
    for p in parts[1:]:
        acc = acc + p
    return acc


def all_reduce(parts: list[np.ndarray]) -> list[np.ndarray]:
    """Every rank receives sum_i parts[i]."""
    total = _ordered_sum(parts)
    return [total.copy() for _ in parts]


def reduce_scatter(parts: list[np.ndarray], axis: int = 0) -> list[np.ndarray]:
    """Rank j receives chunk j (along ``axis``, equal chunks) of sum_i parts[i]."""
    t = len(parts)
    size = parts[0].shape[axis]
    if size % t:
        raise ValueError(f"axis length {size} is not divisible by {t} ranks")
    c = size // t
    out = []
    for j in range(t):
        sl = [slice(None)] * parts[0].ndim
        sl[axis] = slice(j * c, (j + 1) * c)
        out.append(_ordered_sum([p[tuple(sl)] for p in parts]))
    return out


def all_gather(chunks: list[np.ndarray], axis: int = 0) -> list[np.ndarray]:
    """Every rank receives the concatenation of all ranks' chunks along ``axis``."""
    full = np.concatenate(chunks, axis=axis)
    return [full.copy() for _ in chunks]
