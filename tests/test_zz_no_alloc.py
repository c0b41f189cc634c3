"""tpmlp_backward_noalloc, the backward for callers that cannot allocate device memory.

Such a caller (a host that passes only one step's tensors and owns no allocator on the
device, or code that must not allocate once running) cannot provide the workspace that
tpmlp_backward wants; this entry point keeps that intermediate in a static device array
instead. The tests call it through the C ABI and compare every output with tpmlp_backward
given a torch-allocated workspace: the kernels are the same and deterministic, so the results
must be bit-identical. The size limit's rejections need no GPU and live in test_abi_host.py.
This file is named so that pytest collects it last.
"""
import pytest
import torch

import tensor_transformer_mlp_gb300 as tp
from tensor_transformer_mlp_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc(lib, X, A, B, G, Z, Y, dX, dA, dB, t, gelu):
    n, d = X.shape
    m = A.shape[1]
    return lib.tpmlp_backward_noalloc(X.data_ptr(), A.data_ptr(), B.data_ptr(), G.data_ptr(), Z.data_ptr(),
                                      Y.data_ptr(), dX.data_ptr(), dA.data_ptr(), dB.data_ptr(), n, d, m, t,
                                      tp._binding.GELU[gelu], tp._binding.DTYPE[X.dtype],
                                      torch.cuda.current_stream().cuda_stream)


def _check_against_backward(lib, X, A, B, G, t, gelu, label):
    d, m = A.shape
    O, Z, Y = tp.forward(X, A, B, t, gelu)
    ref = tp.backward(X, A, B, G, Z, Y, t, gelu)
    dX = torch.full_like(X, float("nan"))
    dA = torch.full((d, m), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((m, d), float("nan"), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, X, A, B, G, Z, Y, dX, dA, dB, t, gelu)
    assert st == 0, lib.tpmlp_last_error()
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    for name, got, want in (("dX", dX, ref[0]), ("dA", dA, ref[1]), ("dB", dB, ref[2])):
        assert torch.equal(got, want), f"{label} {name}: differs from tpmlp_backward"


def _inputs(cfg, seed, dtype):
    inp = wl.mlp_inputs(cfg, seed=seed)
    return [torch.from_numpy(inp[k]).cuda().to(dtype) for k in "XABG"]


def test_backward_noalloc_matches_backward_on_two_calls():
    lib = tp.load_library()
    cfg = wl.SINGLE_BLOCK  # D is 512 x 4096 bf16 = 4 MiB, inside the static scratch
    for call, seed in enumerate((0, 1)):
        X, A, B, G = _inputs(cfg, seed, torch.bfloat16)
        _check_against_backward(lib, X, A, B, G, cfg.t, cfg.gelu, f"call {call}")


def test_backward_noalloc_f32():
    lib = tp.load_library()
    cfg = wl.WORKED_EXAMPLE
    X, A, B, G = _inputs(cfg, 0, torch.float32)
    _check_against_backward(lib, X, A, B, G, cfg.t, cfg.gelu, "fp32 worked example")


def test_backward_noalloc_at_the_size_limit():
    # n x m x 2 bytes = 8192 x 4096 x 2 = exactly the 64 MiB the static array holds.
    lib = tp.load_library()
    n, d, m, t = 8192, 64, 4096, 8
    g = torch.Generator(device="cpu").manual_seed(3)
    X = torch.randn(n, d, generator=g).to("cuda", torch.bfloat16)
    A = (torch.randn(d, m, generator=g) * 0.02).to("cuda", torch.bfloat16)
    B = (torch.randn(m, d, generator=g) * 0.02).to("cuda", torch.bfloat16)
    G = (torch.randn(n, d, generator=g) * 0.01).to("cuda", torch.bfloat16)
    assert lib.tpmlp_backward_workspace_size(n, m, 1) == 64 << 20
    _check_against_backward(lib, X, A, B, G, t, "tanh", "64 MiB")
