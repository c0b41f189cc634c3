"""GPU parity of the tensor-parallel MLP forward and backward (through the C ABI) against
the float64 oracle, element by element on seeded inputs; sampled rows and columns at the
full sizes the benchmark runs."""
import os

import numpy as np
import pytest
import torch

import tensor_transformer_mlp_gb300 as tp
from oracle import mlp as omlp
from tensor_transformer_mlp_gb300 import workloads as wl

from helpers import TOL_BF16, TOL_F32, assert_close, dev, host

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_example_seed0.txt")

# The plain bf16 GEMMs' kernel variants (tpmlp_set_gemm_variant): SM pairs choosing 256 x 512 or
# 256 x 256 tiles per shape (the default), the one-SM kernel, pairs without pacing, pairs on
# 256 x 256 tiles only, pairs on 256 x 512 tiles only, and two non-default tile bands. The
# parity cases that take the `gemm_variant` fixture run on each.
GEMM_VARIANTS = {"pair": (1, 1, 0), "one_sm": (0, 1, 0), "unpaced": (1, 0, 0), "pair256": (2, 1, 0), "wide": (3, 1, 0),
                 # non-default tile bands: 3 N-blocks walked along M; 5 pair-rows (ragged last band)
                 "nband3": (1, 1, -3), "wide_band5": (3, 1, 5)}


@pytest.fixture(params=list(GEMM_VARIANTS))
def gemm_variant(request):
    tp.tpmlp_set_gemm_variant(*GEMM_VARIANTS[request.param])
    try:
        yield request.param
    finally:
        tp.tpmlp_set_gemm_variant(*GEMM_VARIANTS["pair"])


def run_gpu(inp, t, gelu, dtype):
    X, A, B, G = (dev(inp[k], dtype) for k in "XABG")
    O, Z, Y = tp.forward(X, A, B, t, gelu)
    dX, dA, dB = tp.backward(X, A, B, G, Z, Y, t, gelu)
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    return {"O": O, "Z": Z, "Y": Y, "dX": dX, "dA": dA, "dB": dB}


def check_full(inp, t, gelu, dtype, tol):
    got = run_gpu(inp, t, gelu, dtype)
    ref = omlp.forward(inp["X"], inp["A"], inp["B"], gelu)
    ref.update(omlp.backward(inp["X"], inp["A"], inp["B"], inp["G"], gelu))
    report = {}
    for k in ("Z", "Y", "O", "dX", "dA", "dB"):
        assert_close(k, host(got[k]), ref[k], tol, report)
    print(report)
    return got


def _read_golden():
    arrays, lines = {}, [ln for ln in open(GOLDEN) if not ln.startswith("#")]
    i = 0
    while i < len(lines):
        name, r, c = lines[i].split()
        r, c = int(r), int(c)
        arrays[name] = np.array([[float(v) for v in lines[i + 1 + j].split()] for j in range(r)])
        i += 1 + r
    return arrays


def test_worked_example_f32():
    cfg = wl.WORKED_EXAMPLE
    inp = wl.mlp_inputs(cfg)
    got = check_full(inp, cfg.t, cfg.gelu, "f32", TOL_F32)
    gold = _read_golden()
    assert np.array_equal(gold["X"], inp["X"].astype(np.float64))
    for k in ("O", "dX", "dA", "dB"):
        assert_close("golden " + k, host(got[k]), gold[k], TOL_F32)


def test_single_block_bf16(gemm_variant):
    cfg = wl.SINGLE_BLOCK
    check_full(wl.mlp_inputs(cfg), cfg.t, cfg.gelu, "bf16", TOL_BF16)


@pytest.mark.parametrize("gelu", ["erf", "tanh"])
@pytest.mark.parametrize("shape", [(300, 200, 392, 7), (129, 72, 264, 3), (1, 8, 8, 1), (517, 1032, 776, 8)])
def test_ragged_bf16(shape, gelu, gemm_variant):
    n, d, m, t = shape
    cfg = wl.MLPConfig("ragged", n, d, m, t, "bf16", gelu, 1.0, 0.05, 1.0, seed=n)
    check_full(wl.mlp_inputs(cfg), t, gelu, "bf16", TOL_BF16)


@pytest.mark.parametrize("gelu", ["erf", "tanh"])
@pytest.mark.parametrize("shape", [(37, 45, 66, 3), (130, 70, 140, 2)])
def test_ragged_f32(shape, gelu):
    n, d, m, t = shape
    cfg = wl.MLPConfig("ragged", n, d, m, t, "f32", gelu, 1.0, 0.1, 1.0, seed=n)
    check_full(wl.mlp_inputs(cfg), t, gelu, "f32", TOL_F32)


def test_shard_count_does_not_change_results(gemm_variant):
    # On one GPU the shard sum is the GEMM's K-loop, in shard order for every t.
    cfg = wl.MLPConfig("t-invariance", 256, 512, 1024, 1, "bf16", "tanh", 1.0, 0.02, 1.0)
    inp = wl.mlp_inputs(cfg)
    base = run_gpu(inp, 1, "tanh", "bf16")
    for t in (2, 4, 8):
        other = run_gpu(inp, t, "tanh", "bf16")
        for k in base:
            assert torch.equal(base[k], other[k]), (t, k)


def _backward_keeping_d(X, A, B, G, Z, Y, t, gelu):
    """tpmlp_backward with a caller workspace, returning D = (G B^T) * gelu'(Z) as the
    workspace holds it ([n][m] in the operand dtype) beside dX, dA, dB."""
    n, d = X.shape
    m = A.shape[1]
    ws = torch.empty(tp.tpmlp_backward_workspace_size(n, m, X.dtype), dtype=torch.uint8, device="cuda")
    dX = torch.empty_like(X)
    dA = torch.empty((d, m), dtype=torch.float32, device="cuda")
    dB = torch.empty((m, d), dtype=torch.float32, device="cuda")
    tp.tpmlp_backward(X, A, B, G, Z, Y, dX, dA, dB, t, gelu, ws)
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    D = ws[: n * m * X.element_size()].view(X.dtype).view(n, m)
    return D, dX, dA, dB


@pytest.mark.parametrize("dtype,tol,shape,gelu", [
    ("bf16", TOL_BF16, (512, 1024, 4096, 2), "tanh"),
    ("bf16", TOL_BF16, (300, 200, 392, 7), "erf"),
    ("bf16", TOL_BF16, (129, 72, 264, 3), "tanh"),
    ("bf16", TOL_BF16, (517, 1032, 776, 8), "erf"),
    ("f32", TOL_F32, (37, 45, 66, 3), "tanh"),
    ("f32", TOL_F32, (130, 70, 140, 2), "erf"),
])
def test_dgrad1_output_d(shape, gelu, dtype, tol):
    """D = (G B^T) * gelu'(Z), the dgrad-1 GEMM's output ("024 | Megatron-LM", section 二, the D_i
    equation), compared element by element with the oracle's D (not only through dA and dX)."""
    n, d, m, t = shape
    cfg = wl.MLPConfig("d-direct", n, d, m, t, dtype, gelu, 1.0, 0.05, 1.0, seed=n + 3)
    inp = wl.mlp_inputs(cfg)
    X, A, B, G = (dev(inp[k], dtype) for k in "XABG")
    O, Z, Y = tp.forward(X, A, B, t, gelu)
    D, _, _, _ = _backward_keeping_d(X, A, B, G, Z, Y, t, gelu)
    ref = omlp.backward(inp["X"], inp["A"], inp["B"], inp["G"], gelu)["D"]
    print(assert_close("D", host(D), ref, tol))


@pytest.mark.parametrize("cfg", [wl.GPT_MLP, wl.LARGE_MLP], ids=lambda c: c.name)
def test_dgrad1_output_d_sampled(cfg):
    """D at the full GPT and large MLP sizes on sampled intermediate columns: column j of D needs
    only A[:, j] and B[j, :]."""
    inp = wl.mlp_inputs(cfg)
    X, A, B, G = (dev(inp[k], cfg.dtype) for k in "XABG")
    O, Z, Y = tp.forward(X, A, B, cfg.t, cfg.gelu)
    D, _, _, _ = _backward_keeping_d(X, A, B, G, Z, Y, cfg.t, cfg.gelu)
    J = wl.sample_indices(48, cfg.m, seed=2)
    ref = omlp.backward(inp["X"], inp["A"][:, J], inp["B"][J, :], inp["G"], cfg.gelu)["D"]
    print(cfg.name, assert_close("D[:,J]", host(D[:, torch.from_numpy(J).cuda()]), ref, TOL_BF16))


def test_empty_tokens():
    d, m = 64, 128
    X = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    A = torch.ones((d, m), dtype=torch.bfloat16, device="cuda")
    B = torch.ones((m, d), dtype=torch.bfloat16, device="cuda")
    O, Z, Y = tp.forward(X, A, B, 2, "tanh")
    assert O.shape == (0, d)
    dX, dA, dB = tp.backward(X, A, B, torch.empty_like(X), Z, Y, 2, "tanh")
    torch.cuda.synchronize()
    assert torch.count_nonzero(dA) == 0 and torch.count_nonzero(dB) == 0


def test_bad_arguments_raise():
    X = torch.zeros((8, 16), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((16, 24), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((24, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TpmlpError, match="SHAPE"):
        tp.forward(X, A, B, 5, "tanh")


def sampled_parity(cfg, n_rows=48, n_cols=48):
    """Full-size run in the benchmark's launch configuration; the oracle computes sampled
    token rows of O and dX and sampled intermediate columns of dA, dB, Z and Y."""
    inp = wl.mlp_inputs(cfg)
    got = run_gpu(inp, cfg.t, cfg.gelu, cfg.dtype)
    R = wl.sample_indices(n_rows, cfg.n, seed=1)
    J = wl.sample_indices(n_cols, cfg.m, seed=2)
    rows_f = omlp.forward(inp["X"][R], inp["A"], inp["B"], cfg.gelu)
    rows_b = omlp.backward(inp["X"][R], inp["A"], inp["B"], inp["G"][R], cfg.gelu)
    cols_b = omlp.backward(inp["X"], inp["A"][:, J], inp["B"][J, :], inp["G"], cfg.gelu)
    cols_f = omlp.forward(inp["X"], inp["A"][:, J], inp["B"][J, :], cfg.gelu)
    Rt = torch.from_numpy(R).cuda()
    Jt = torch.from_numpy(J).cuda()
    report = {}
    assert_close("O[R]", host(got["O"][Rt]), rows_f["O"], TOL_BF16, report)
    assert_close("dX[R]", host(got["dX"][Rt]), rows_b["dX"], TOL_BF16, report)
    assert_close("Z[:,J]", host(got["Z"][:, Jt]), cols_f["Z"], TOL_BF16, report)
    assert_close("Y[:,J]", host(got["Y"][:, Jt]), cols_f["Y"], TOL_BF16, report)
    assert_close("dA[:,J]", host(got["dA"][:, Jt]), cols_b["dA"], TOL_BF16, report)
    assert_close("dB[J,:]", host(got["dB"][Jt, :]), cols_b["dB"], TOL_BF16, report)
    print(cfg.name, report)


def test_gpt_mlp_sampled(gemm_variant):
    sampled_parity(wl.GPT_MLP)


def test_large_mlp_sampled():
    sampled_parity(wl.LARGE_MLP)


@pytest.mark.parametrize("dtype,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
@pytest.mark.parametrize("shape", [(512, 1024, 4096, 2), (300, 200, 392, 7), (37, 48, 72, 3)])
def test_biased_block(shape, dtype, tol, gemm_variant):
    n, d, m, t = shape
    cfg = wl.MLPConfig("biased", n, d, m, t, dtype, "tanh", 1.0, 0.05, 1.0, seed=n + 7)
    inp = wl.mlp_inputs(cfg)
    rng = np.random.default_rng(n)
    b1 = (rng.standard_normal(m) * 0.5).astype(np.float32)
    b2 = (rng.standard_normal(d) * 0.5).astype(np.float32)
    if dtype == "bf16":
        b1, b2 = wl.round_to_bf16(b1), wl.round_to_bf16(b2)
    X, A, B, G = (dev(inp[k], dtype) for k in "XABG")
    O, Z, Y = tp.forward(X, A, B, t, "tanh", bias1=dev(b1, dtype), bias2=dev(b2, dtype))
    dX, dA, dB, db1, db2 = tp.backward(X, A, B, G, Z, Y, t, "tanh", with_bias=True)
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    ref = omlp.forward(inp["X"], inp["A"], inp["B"], "tanh", b1, b2)
    ref.update(omlp.backward(inp["X"], inp["A"], inp["B"], inp["G"], "tanh", b1))
    rep = {}
    for k, got in (("Z", Z), ("O", O), ("dX", dX), ("dA", dA), ("dB", dB), ("db1", db1), ("db2", db2)):
        assert_close(k, host(got), ref[k], tol, rep)
    print(rep)


@pytest.mark.parametrize("dtype,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
def test_main_grad_accumulation_over_microbatches(dtype, tol, gemm_variant):
    """dA, dB accumulated over three micro-batches (one of them ragged) equal the oracle's
    gradients of the concatenated batch added to the buffers' starting values."""
    cfg = wl.MLPConfig("microbatches", 700, 256, 512, 4, dtype, "tanh", 1.0, 0.05, 1.0, seed=11)
    inp = wl.mlp_inputs(cfg)
    A, B = dev(inp["A"], dtype), dev(inp["B"], dtype)
    rng = np.random.default_rng(12)
    dA0 = rng.standard_normal((cfg.d, cfg.m)).astype(np.float32)
    dB0 = rng.standard_normal((cfg.m, cfg.d)).astype(np.float32)
    dA = torch.from_numpy(dA0).cuda()
    dB = torch.from_numpy(dB0).cuda()
    for lo, hi in ((0, 256), (256, 512), (512, 700)):
        X = dev(inp["X"][lo:hi], dtype)
        G = dev(inp["G"][lo:hi], dtype)
        O, Z, Y = tp.forward(X, A, B, cfg.t, "tanh")
        dX = torch.empty_like(X)
        ws = torch.empty(tp.tpmlp_backward_workspace_size(hi - lo, cfg.m, X.dtype), dtype=torch.uint8, device="cuda")
        tp.tpmlp_backward_accumulate(X, A, B, G, Z, Y, dX, dA, dB, cfg.t, "tanh", ws)
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    ref = omlp.backward(inp["X"], inp["A"], inp["B"], inp["G"], "tanh")
    assert_close("dA", host(dA) - dA0, ref["dA"], tol)
    assert_close("dB", host(dB) - dB0, ref["dB"], tol)


def test_bounded_wait_reports_timeout_and_context_survives():
    """Failure detection: a kernel waits on a barrier that nothing completes, gives up after
    50 ms and records TPMLP_ERR_TIMEOUT; the status is read on the host, cleared, and the same
    context then runs a forward pass correctly."""
    tp.tpmlp_device_status(clear=True)
    tp.tpmlp_check_wait_timeout(50_000_000)
    with pytest.raises(tp.TpmlpError, match="TIMEOUT"):
        tp.tpmlp_device_status(clear=True)
    tp.tpmlp_device_status()  # cleared
    cfg = wl.MLPConfig("after-timeout", 128, 256, 512, 2, "bf16", "tanh", 1.0, 0.05, 1.0)
    inp = wl.mlp_inputs(cfg)
    X, A, B = (dev(inp[k], "bf16") for k in "XAB")
    O, _, _ = tp.forward(X, A, B, cfg.t, "tanh")
    torch.cuda.synchronize()
    assert_close("O", host(O), omlp.forward(inp["X"], inp["A"], inp["B"], "tanh")["O"], TOL_BF16)


def test_step_replays_from_a_cuda_graph():
    """Forward + backward captured once in a CUDA graph and replayed: bit-identical to eager
    launches (no host synchronisation or allocation inside the calls; the pair GEMM's cluster
    launches and pacing-counter resets are captured like any other stream work)."""
    cfg = wl.MLPConfig("graph", 1024, 512, 2048, 4, "bf16", "tanh", 1.0, 0.05, 1.0, seed=21)
    inp = wl.mlp_inputs(cfg)
    X, A, B, G = (dev(inp[k], "bf16") for k in "XABG")
    n, d, m, t = cfg.n, cfg.d, cfg.m, cfg.t
    outs = {k: torch.empty(s, dtype=dt, device="cuda") for k, s, dt in
            (("O", (n, d), torch.bfloat16), ("Z", (n, m), torch.bfloat16), ("Y", (n, m), torch.bfloat16),
             ("dX", (n, d), torch.bfloat16), ("dA", (d, m), torch.float32), ("dB", (m, d), torch.float32))}
    ws = torch.empty(tp.tpmlp_backward_workspace_size(n, m, torch.bfloat16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step():
        tp.tpmlp_forward(X, A, B, outs["O"], outs["Z"], outs["Y"], t, "tanh", s)
        tp.tpmlp_backward(X, A, B, G, outs["Z"], outs["Y"], outs["dX"], outs["dA"], outs["dB"], t, "tanh", ws, s)

    with torch.cuda.stream(s):
        step()  # eager, also initialises the library's per-device state outside the capture
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in outs.items()}
    for v in outs.values():
        v.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    tp.tpmlp_device_status()
    for k in outs:
        assert torch.equal(outs[k], eager[k]), k
