"""Seeded synthetic workloads for the tensor-parallel MLP and its sequence-parallel block.

This module only names the workload shapes and draws their inputs; it holds none
of the MLP's arithmetic. The CUDA path and the float64 oracle both take their
inputs from here, and from nowhere else.

Recipe (every workload, seed 0 unless a caller passes another):
  one ``numpy.random.default_rng(seed)``; float64 ``standard_normal`` draws in the
  order X, A, B, G (SP block: x, A, B), each scaled by its standard deviation,
  rounded to float32 (round-to-nearest-even) and then, for bf16 workloads, to
  bfloat16 (round-to-nearest-even on the float32 bits). The stored arrays hold the
  exactly representable rounded values, so the oracle reads the very numbers the
  GPU reads. Draws are made in row chunks; numpy's Generator fills a stream
  sequentially, so chunking does not change the values.

Shapes follow the notation of "Megatron-LM: Training Multi-Billion Parameter
Language Models Using Model Parallelism" (section 2, "forward little
communication"): n tokens, d model width, m intermediate width, t shards.
The second parameter of every N(0, .) is a standard deviation.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_CHUNK_ELEMS = 1 << 24  # float64 elements drawn per chunk (128 MiB)


@dataclass(frozen=True)
class MLPConfig:
    """One tensor-parallel MLP workload: O = sum_i gelu(X A_i) B_i and its gradients."""
    name: str
    n: int
    d: int
    m: int
    t: int
    dtype: str      # "f32" or "bf16"
    gelu: str       # "erf" or "tanh"
    x_std: float
    w_std: float
    g_std: float
    seed: int = 0

    @property
    def flops_fwd_bwd(self) -> int:
        """Six GEMMs of 2*n*d*m each: two forward, four backward."""
        return 12 * self.n * self.d * self.m


@dataclass(frozen=True)
class SPConfig:
    """One sequence-parallel block: LN -> gather -> MLP -> reduce-scatter -> dropout + residual."""
    name: str
    b: int
    s: int
    h: int
    m: int
    t: int
    gelu: str
    x_std: float
    w_std: float
    eps: float = 1e-5
    p_drop: float = 0.1
    seed: int = 0
    dtype: str = "bf16"

    @property
    def n(self) -> int:
        return self.b * self.s

    @property
    def flops_mlp_fwd(self) -> int:
        return 4 * self.n * self.h * self.m


WORKED_EXAMPLE = MLPConfig("worked_example_n3_d4_m8_t2_f32", 3, 4, 8, 2, "f32", "erf", 1.0, 1.0, 1.0)
SINGLE_BLOCK = MLPConfig("mlp_n512_d1024_m4096_t2_bf16", 512, 1024, 4096, 2, "bf16", "tanh", 1.0, 0.02, 1.0)
GPT_MLP = MLPConfig("gpt_mlp_n8192_h4096_m16384_t8_bf16", 8192, 4096, 16384, 8, "bf16", "tanh", 1.0, 0.02, 0.01)
SP_BLOCK = SPConfig("sp_block_b2_s4096_h4096_m16384_t8_bf16", 2, 4096, 4096, 16384, 8, "tanh", 1.0, 0.02)
LARGE_MLP = MLPConfig("large_mlp_n16384_h8192_m32768_t8_bf16", 16384, 8192, 32768, 8, "bf16", "tanh", 1.0, 0.01, 0.01)

@dataclass(frozen=True)
class AttnConfig:
    """One tensor-parallel self-attention workload (heads split across t shards)."""
    name: str
    b: int
    s: int
    h: int
    heads: int
    t: int
    x_std: float
    w_std: float
    g_std: float
    seed: int = 0
    dtype: str = "bf16"

    @property
    def n(self) -> int:
        return self.b * self.s

    @property
    def flops_fwd(self) -> int:
        """QKV (6nh^2) + scores and PV (4 b s^2 h) + output projection (2nh^2)."""
        return 8 * self.n * self.h * self.h + 4 * self.b * self.s * self.s * self.h


GPT_ATTENTION = AttnConfig("gpt_attention_b2_s2048_h4096_a32_t8_bf16", 2, 2048, 4096, 32, 8, 1.0, 0.02, 0.01)

MLP_CONFIGS = {c.name: c for c in (WORKED_EXAMPLE, SINGLE_BLOCK, GPT_MLP, LARGE_MLP)}
SP_CONFIGS = {SP_BLOCK.name: SP_BLOCK}


def round_to_bf16(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32 holding them."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    u = x32.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = ((u + bias) >> np.uint32(16)) << np.uint32(16)
    return r.astype(np.uint32).view(np.float32)


def bf16_bits(x32: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are already bf16-exact."""
    return (np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _draw(rng: np.random.Generator, shape: tuple[int, int], std: float, dtype: str) -> np.ndarray:
    rows, cols = shape
    out = np.empty(shape, dtype=np.float32)
    step = max(1, _CHUNK_ELEMS // max(cols, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        chunk = (rng.standard_normal((r1 - r0, cols)) * std).astype(np.float32)
        out[r0:r1] = round_to_bf16(chunk) if dtype == "bf16" else chunk
    return out


def mlp_inputs(cfg: MLPConfig, seed: int | None = None) -> dict[str, np.ndarray]:
    """X [n,d], A [d,m], B [m,d], G [n,d] as float32 arrays of dtype-exact values."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    X = _draw(rng, (cfg.n, cfg.d), cfg.x_std, cfg.dtype)
    A = _draw(rng, (cfg.d, cfg.m), cfg.w_std, cfg.dtype)
    B = _draw(rng, (cfg.m, cfg.d), cfg.w_std, cfg.dtype)
    G = _draw(rng, (cfg.n, cfg.d), cfg.g_std, cfg.dtype)
    return {"X": X, "A": A, "B": B, "G": G}


def sp_inputs(cfg: SPConfig, seed: int | None = None) -> dict[str, np.ndarray]:
    """x [b,s,h] in token order, A [h,m], B [m,h], gamma = 1, beta = 0 (float32)."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    x = _draw(rng, (cfg.b * cfg.s, cfg.h), cfg.x_std, cfg.dtype).reshape(cfg.b, cfg.s, cfg.h)
    A = _draw(rng, (cfg.h, cfg.m), cfg.w_std, cfg.dtype)
    B = _draw(rng, (cfg.m, cfg.h), cfg.w_std, cfg.dtype)
    gamma = np.ones(cfg.h, dtype=np.float32)
    beta = np.zeros(cfg.h, dtype=np.float32)
    return {"x": x, "A": A, "B": B, "gamma": gamma, "beta": beta}


def to_shards(x: np.ndarray, t: int) -> np.ndarray:
    """[b, s, h] token order -> [t, b, s/t, h]: shard j holds sequence positions j*s/t .. (j+1)*s/t - 1."""
    b, s, h = x.shape
    assert s % t == 0
    return np.ascontiguousarray(x.reshape(b, t, s // t, h).transpose(1, 0, 2, 3))


def from_shards(xs: np.ndarray) -> np.ndarray:
    """[t, b, s/t, h] -> [b, s, h] token order (inverse of ``to_shards``)."""
    t, b, sl, h = xs.shape
    return np.ascontiguousarray(xs.transpose(1, 0, 2, 3).reshape(b, t * sl, h))


def sample_indices(count: int, total: int, seed: int) -> np.ndarray:
    """Sorted distinct indices for sampled parity checks at full size."""
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(total, size=min(count, total), replace=False))


def attn_inputs(cfg: AttnConfig, seed: int | None = None) -> dict[str, np.ndarray]:
    """X [b, s, h], W_qkv [h, 3h], W_o [h, h], G [b, s, h] (same recipe as the MLP workloads)."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    X = _draw(rng, (cfg.b * cfg.s, cfg.h), cfg.x_std, cfg.dtype).reshape(cfg.b, cfg.s, cfg.h)
    Wqkv = _draw(rng, (cfg.h, 3 * cfg.h), cfg.w_std, cfg.dtype)
    Wo = _draw(rng, (cfg.h, cfg.h), cfg.w_std, cfg.dtype)
    G = _draw(rng, (cfg.b * cfg.s, cfg.h), cfg.g_std, cfg.dtype).reshape(cfg.b, cfg.s, cfg.h)
    return {"X": X, "Wqkv": Wqkv, "Wo": Wo, "G": G}


def norm_inputs(rows: int, h: int, dtype: str = "bf16", seed: int = 0, x_std: float = 1.0, x_mean: float = 0.5):
    """RMSNorm inputs: x [rows, h] ~ N(x_mean, x_std), gamma [h] ~ 1 + 0.1 N(0, 1) (fp32), dy
    [rows, h] ~ N(0, 1); x and dy hold values exact in `dtype`."""
    rng = np.random.default_rng(seed)
    x = _draw(rng, (rows, h), x_std, dtype) + np.float32(x_mean)
    if dtype == "bf16":
        x = round_to_bf16(x)
    gamma = (1.0 + 0.1 * rng.standard_normal(h)).astype(np.float32)
    dy = _draw(rng, (rows, h), 1.0, dtype)
    return {"x": x, "gamma": gamma, "dy": dy}

