"""GPU parity of RMSNorm and its backward (through the C ABI) against the float64 oracle,
element by element on seeded inputs: ragged row counts, several widths, both dtypes, the
empty batch, in-place use, and the GPT attention block's input size."""
import numpy as np
import pytest
import torch

import tensor_transformer_mlp_gb300 as tp
from oracle import rmsnorm as orms
from tensor_transformer_mlp_gb300 import workloads as wl

from helpers import TOL_BF16, TOL_F32, assert_close, dev, host

pytestmark = pytest.mark.gpu

TOL = {"bf16": TOL_BF16, "f32": TOL_F32}


def _check(rows, h, dtype, eps, backward=True, seed=0):
    inp = wl.norm_inputs(rows, h, dtype, seed=seed)
    x, dy = dev(inp["x"], dtype), dev(inp["dy"], dtype)
    gamma = torch.from_numpy(inp["gamma"]).cuda()
    y = tp.rmsnorm(x, gamma, eps)
    rep = {}
    ref_y = orms.rmsnorm(inp["x"], inp["gamma"], eps)
    if backward:
        dx, dgamma = tp.rmsnorm_backward(x, gamma, dy, eps)
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    if rows == 0:
        assert y.shape == (0, h)
        if backward:
            assert torch.count_nonzero(dgamma) == 0
        return
    assert_close("y", host(y), ref_y, TOL[dtype], rep)
    if backward:
        ref_dx, ref_dg = orms.rmsnorm_backward(inp["x"], inp["gamma"], eps, inp["dy"])
        assert_close("dx", host(dx), ref_dx, TOL[dtype], rep)
        assert_close("dgamma", host(dgamma), ref_dg, TOL[dtype], rep)
    print(rows, h, dtype, rep)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,h", [(1, 8), (37, 256), (300, 1000 + 8), (129, 4096)])
def test_rmsnorm_parity(rows, h, dtype):
    _check(rows, h, dtype, 1e-5)


def test_rmsnorm_large_eps_and_width_8192():
    _check(64, 256, "bf16", 1e-1)
    _check(257, 8192, "bf16", 1e-5)   # forward and backward take h up to 8192 in bf16


def test_rmsnorm_backward_width_8192_f32():
    inp = wl.norm_inputs(33, 8192, "f32", seed=4)
    x, dy = dev(inp["x"], "f32"), dev(inp["dy"], "f32")
    gamma = torch.from_numpy(inp["gamma"]).cuda()
    dx, dgamma = tp.rmsnorm_backward(x, gamma, dy, 1e-5)
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    ref_dx, ref_dg = orms.rmsnorm_backward(inp["x"], inp["gamma"], 1e-5, inp["dy"])
    assert_close("dx", host(dx), ref_dx, TOL_F32)
    assert_close("dgamma", host(dgamma), ref_dg, TOL_F32)


def test_rmsnorm_empty_batch():
    _check(0, 64, "bf16", 1e-5)


def test_rmsnorm_in_place():
    inp = wl.norm_inputs(50, 512, "bf16", seed=3)
    x = dev(inp["x"], "bf16")
    gamma = torch.from_numpy(inp["gamma"]).cuda()
    tp.tpmlp_rmsnorm(x, gamma, 1e-5, x)
    torch.cuda.synchronize()
    assert_close("y in place", host(x), orms.rmsnorm(inp["x"], inp["gamma"], 1e-5), TOL_BF16)


def test_rmsnorm_gpt_attention_input():
    cfg = wl.GPT_ATTENTION
    _check(cfg.b * cfg.s, cfg.h, "bf16", 1e-5, seed=7)
