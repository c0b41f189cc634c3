"""GPU parity of the tensor-parallel self-attention block (through the C ABI) against the
float64 oracle: projections, per-head softmax(Q K^T / sqrt(head_dim)) V, and all gradients."""
import numpy as np
import pytest
import torch

import tensor_transformer_mlp_gb300 as tp
from oracle import attention as oattn
from tensor_transformer_mlp_gb300 import workloads as wl

from helpers import TOL_BF16, assert_close, dev, host

pytestmark = pytest.mark.gpu


def run_case(cfg):
    inp = wl.attn_inputs(cfg)
    X = dev(inp["X"], "bf16")
    Wqkv, Wo, G = dev(inp["Wqkv"], "bf16"), dev(inp["Wo"], "bf16"), dev(inp["G"], "bf16")
    Y, saves = tp.attention_forward(X, Wqkv, Wo, cfg.heads, cfg.t)
    dX, dWqkv, dWo = tp.attention_backward(X, Wqkv, Wo, G, saves, cfg.heads, cfg.t)
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    f = oattn.forward(inp["X"], inp["Wqkv"], inp["Wo"], cfg.heads)
    g = oattn.backward(inp["X"], inp["Wqkv"], inp["Wo"], cfg.heads, inp["G"])
    b, s, h = cfg.b, cfg.s, cfg.h
    rep = {}
    assert_close("QKV", host(saves[0]).reshape(b, s, 3 * h), f["QKV"], TOL_BF16, rep)
    assert_close("P", host(saves[1]), f["P"], TOL_BF16, rep)
    assert_close("O", host(saves[2]).reshape(b, s, h), f["O"], TOL_BF16, rep)
    assert_close("Y", host(Y), f["Y"], TOL_BF16, rep)
    assert_close("dX", host(dX), g["dX"], TOL_BF16, rep)
    assert_close("dWqkv", host(dWqkv), g["dWqkv"], TOL_BF16, rep)
    assert_close("dWo", host(dWo), g["dWo"], TOL_BF16, rep)
    print(cfg.name, rep)


@pytest.mark.parametrize("shape", [(2, 64, 256, 4, 2), (1, 200, 128, 2, 1), (3, 136, 512, 8, 4), (2, 256, 384, 3, 3)])
def test_attention_small(shape):
    b, s, h, heads, t = shape
    run_case(wl.AttnConfig("attn-small", b, s, h, heads, t, 1.0, 0.05, 1.0, seed=s))


def test_attention_gpt_size():
    run_case(wl.GPT_ATTENTION)


def test_attention_empty_batch():
    h, heads = 128, 2
    X = torch.empty((0, 64, h), dtype=torch.bfloat16, device="cuda")
    Wqkv = torch.ones((h, 3 * h), dtype=torch.bfloat16, device="cuda")
    Wo = torch.ones((h, h), dtype=torch.bfloat16, device="cuda")
    Y, saves = tp.attention_forward(X, Wqkv, Wo, heads, 2)
    dX, dWqkv, dWo = tp.attention_backward(X, Wqkv, Wo, torch.empty_like(X), saves, heads, 2)
    torch.cuda.synchronize()
    assert Y.shape == (0, 64, h) and dX.shape == (0, 64, h)
    assert torch.count_nonzero(dWqkv) == 0 and torch.count_nonzero(dWo) == 0


def test_attention_smallest_head_dim_and_sequence():
    # head_dim 8 and s 8: the operand tiles are mostly fill, one row of a softmax is 8 wide
    run_case(wl.AttnConfig("attn-min", 3, 8, 32, 4, 2, 1.0, 0.2, 1.0, seed=5))


def test_attention_longest_sequence():
    # s = 8192, the largest the softmax kernels take (one row per CTA, 8 vectors per thread)
    run_case(wl.AttnConfig("attn-s8192", 1, 8192, 256, 2, 2, 1.0, 0.05, 1.0, seed=9))
