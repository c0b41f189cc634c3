"""tpmlp_backward_noalloc, the backward for callers that cannot allocate device memory.

Such a caller (a host that passes only one step's tensors and owns no allocator on the
device, or code that must not allocate once running) cannot provide the workspace that
tpmlp_backward wants; this entry point keeps that intermediate in a static device array
instead. The test calls it through the C ABI twice in a row, on different inputs, and
compares each result with tpmlp_backward given a torch-allocated workspace. This file is
named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import tensor_transformer_mlp_gb300 as tp
from tensor_transformer_mlp_gb300 import workloads as wl

from helpers import TOL_BF16, assert_close, host

pytestmark = pytest.mark.gpu

WORKSPACE_ERR = 7


def _noalloc(lib, X, A, B, G, Z, Y, dX, dA, dB, t, gelu):
    n, d = X.shape
    m = A.shape[1]
    return lib.tpmlp_backward_noalloc(X.data_ptr(), A.data_ptr(), B.data_ptr(), G.data_ptr(), Z.data_ptr(),
                                      Y.data_ptr(), dX.data_ptr(), dA.data_ptr(), dB.data_ptr(), n, d, m, t,
                                      tp._binding.GELU[gelu], tp._binding.DTYPE[X.dtype],
                                      torch.cuda.current_stream().cuda_stream)


def test_backward_noalloc_matches_backward_on_two_calls():
    lib = tp.load_library()
    cfg = wl.SINGLE_BLOCK  # D is 512 x 4096 bf16 = 4 MiB, inside the static scratch
    for call, seed in enumerate((0, 1)):
        inp = wl.mlp_inputs(cfg, seed=seed)
        X, A, B, G = (torch.from_numpy(inp[k]).cuda().to(torch.bfloat16) for k in "XABG")
        O, Z, Y = tp.forward(X, A, B, cfg.t, cfg.gelu)
        ref = tp.backward(X, A, B, G, Z, Y, cfg.t, cfg.gelu)
        dX = torch.full_like(X, float("nan"))
        dA = torch.full((cfg.d, cfg.m), float("nan"), dtype=torch.float32, device="cuda")
        dB = torch.full((cfg.m, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(lib, X, A, B, G, Z, Y, dX, dA, dB, cfg.t, cfg.gelu)
        assert st == 0, lib.tpmlp_last_error()
        torch.cuda.synchronize()
        tp.tpmlp_device_status()
        for name, got, want in (("dX", dX, ref[0]), ("dA", dA, ref[1]), ("dB", dB, ref[2])):
            assert_close(f"call {call} {name}", host(got), host(want), TOL_BF16)


def test_backward_noalloc_rejects_oversize():
    lib = tp.load_library()
    fake = 0x10000  # never dereferenced: the size check runs before anything else
    n, d, m = 16384, 8192, 32768  # D would be 1 GiB
    st = lib.tpmlp_backward_noalloc(*([fake] * 9), n, d, m, 8, 1, 1, None)
    assert st == WORKSPACE_ERR
    assert b"static scratch" in lib.tpmlp_last_error()
