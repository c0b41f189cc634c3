"""Pins for the float64 oracle: each test ties an oracle function to something other
than itself (closed forms, finite differences, torch autograd, brute force, the
block-matrix invariants and the ReLU counterexample of the pages)."""
import math

import numpy as np
import pytest
import torch
from scipy.integrate import quad

from oracle import collectives, mlp, rmsnorm, sp
from tensor_transformer_mlp_gb300 import workloads as wl

KINDS = ("erf", "tanh")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


# ---------------------------------------------------------------- GeLU

@pytest.mark.parametrize("kind", KINDS)
def test_gelu_closed_forms(kind):
    assert mlp.gelu(0.0, kind) == 0.0
    assert mlp.gelu_grad(0.0, kind) == 0.5
    assert abs(mlp.gelu(12.0, kind) - 12.0) < 1e-12        # phi(x) -> x as x -> +inf
    assert abs(mlp.gelu(-12.0, kind)) < 1e-12              # phi(x) -> 0 as x -> -inf
    assert abs(mlp.gelu_grad(12.0, kind) - 1.0) < 1e-12
    assert abs(mlp.gelu_grad(-12.0, kind)) < 1e-12


def test_gelu_erf_is_x_times_normal_cdf_by_quadrature():
    # Phi by numerical integration of the standard normal density: independent of erf.
    pdf = lambda u: math.exp(-0.5 * u * u) / math.sqrt(2 * math.pi)
    for x in (-3.1, -1.0, -0.25, 0.4, 1.7, 2.9):
        cdf = quad(pdf, -np.inf, x, epsabs=1e-13, epsrel=1e-13, limit=200)[0]
        assert abs(mlp.gelu(x, "erf") - x * cdf) < 1e-11


def test_gelu_tanh_tracks_erf():
    x = np.linspace(-8, 8, 20001)
    diff = np.abs(mlp.gelu(x, "tanh") - mlp.gelu(x, "erf")).max()
    assert 1e-5 < diff < 1e-3     # an approximation, and a close one


@pytest.mark.parametrize("kind", KINDS)
def test_gelu_grad_matches_finite_differences(kind):
    x = np.linspace(-6, 6, 1201)
    h = 1e-5
    fd = (mlp.gelu(x + h, kind) - mlp.gelu(x - h, kind)) / (2 * h)
    assert np.abs(fd - mlp.gelu_grad(x, kind)).max() < 1e-8


@pytest.mark.parametrize("kind", KINDS)
def test_gelu_matches_torch(kind):
    x = torch.linspace(-7, 7, 4001, dtype=torch.float64)
    ref = torch.nn.functional.gelu(x, approximate="none" if kind == "erf" else "tanh").numpy()
    assert np.abs(mlp.gelu(x.numpy(), kind) - ref).max() < 1e-14


# ---------------------------------------------------------------- MLP forward / backward

def _worked_example():
    return wl.mlp_inputs(wl.WORKED_EXAMPLE)


def test_worked_example_shapes():
    # "给两次投影标上跨卡尺寸": X 3x4, A 4x8, B 8x4; two 4x4 column blocks of A, two 4x4
    # row blocks of B, two 3x4 contributions that sum to a 3x4 output.
    inp = _worked_example()
    assert inp["X"].shape == (3, 4) and inp["A"].shape == (4, 8) and inp["B"].shape == (8, 4)
    views = mlp.shard_views(inp["A"], inp["B"], 2)
    assert [v[0].shape for v in views] == [(4, 4), (4, 4)]
    assert [v[1].shape for v in views] == [(4, 4), (4, 4)]
    contributions = [mlp.gelu(inp["X"] @ Ai, "erf") @ Bi for Ai, Bi in views]
    assert [c.shape for c in contributions] == [(3, 4), (3, 4)]


@pytest.mark.parametrize("kind", KINDS)
def test_backward_matches_finite_differences(kind):
    inp = _worked_example()
    X, A, B, G = (inp[k].astype(np.float64) for k in "XABG")
    grads = mlp.backward(X, A, B, G, kind)
    loss = lambda X_, A_, B_: float((mlp.forward(X_, A_, B_, kind)["O"] * G).sum())
    h = 1e-6
    for name, arr, key in (("X", X, "dX"), ("A", A, "dA"), ("B", B, "dB")):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args_p = {"X": X, "A": A, "B": B}
            args_m = dict(args_p)
            args_p[name], args_m[name] = plus, minus
            fd[idx] = (loss(args_p["X"], args_p["A"], args_p["B"]) - loss(args_m["X"], args_m["A"], args_m["B"])) / (2 * h)
        err = np.abs(fd - grads[key]).max() / np.abs(grads[key]).max()
        assert err < 1e-7, (name, err)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(3, 4, 8), (17, 24, 40)])
def test_forward_backward_match_torch_autograd(kind, shape):
    n, d, m = shape
    X, A, B, G = _rand((n, d), 1), _rand((d, m), 2, 0.3), _rand((m, d), 3, 0.3), _rand((n, d), 4)
    tX, tA, tB = (torch.tensor(a, requires_grad=True) for a in (X, A, B))
    Z = tX @ tA
    O = torch.nn.functional.gelu(Z, approximate="none" if kind == "erf" else "tanh") @ tB
    O.backward(torch.tensor(G))
    fwd = mlp.forward(X, A, B, kind)
    bwd = mlp.backward(X, A, B, G, kind)
    assert np.abs(fwd["O"] - O.detach().numpy()).max() < 1e-12
    assert np.abs(fwd["Z"] - Z.detach().numpy()).max() < 1e-12
    assert np.abs(bwd["dX"] - tX.grad.numpy()).max() < 1e-12
    assert np.abs(bwd["dA"] - tA.grad.numpy()).max() < 1e-12
    assert np.abs(bwd["dB"] - tB.grad.numpy()).max() < 1e-12


def test_forward_brute_force_loops():
    inp = _worked_example()
    X, A, B = (inp[k].astype(np.float64).tolist() for k in "XAB")
    n, d, m = 3, 4, 8
    O = [[0.0] * d for _ in range(n)]
    for r in range(n):
        for j in range(m):
            z = sum(X[r][k] * A[k][j] for k in range(d))
            y = 0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0)))
            for c in range(d):
                O[r][c] += y * B[j][c]
    assert np.abs(np.array(O) - mlp.forward(inp["X"], inp["A"], inp["B"], "erf")["O"]).max() < 1e-13


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_shard_sum_equals_unsharded(kind, t):
    for X, A, B, G in ((lambda i: (i["X"], i["A"], i["B"], i["G"]))(_worked_example()),
                       (_rand((16, 32), 5), _rand((32, 64), 6, 0.2), _rand((64, 32), 7, 0.2), _rand((16, 32), 8))):
        ref_f, ref_b = mlp.forward(X, A, B, kind), mlp.backward(X, A, B, G, kind)
        sh_f, sh_b = mlp.forward_sharded(X, A, B, t, kind), mlp.backward_sharded(X, A, B, G, t, kind)
        for key in ("Z", "Y", "O"):
            assert np.abs(sh_f[key] - ref_f[key]).max() < 1e-13 * max(1.0, np.abs(ref_f[key]).max())
        for key in ("D", "dA", "dB", "dX"):
            assert np.abs(sh_b[key] - ref_b[key]).max() < 1e-13 * max(1.0, np.abs(ref_b[key]).max())


def test_uneven_split_rejected():
    with pytest.raises(ValueError):
        mlp.shard_views(np.zeros((4, 8)), np.zeros((8, 4)), 3)


def test_relu_counterexample_exact():
    # "教学算例": u = 1, v = -2 gives phi(u + v) = 0 but phi(u) + phi(v) = 1.
    X = np.array([[1.0, -2.0]])
    A = np.array([[1.0], [1.0]])
    B = np.array([[1.0]])
    assert mlp.forward(X, A, B, "relu")["O"][0, 0] == 0.0
    assert mlp.forward_input_split(X, A, B, 2, "relu")[0, 0] == 1.0


@pytest.mark.parametrize("kind", KINDS)
def test_input_channel_split_is_wrong(kind):
    X, A, B = _rand((8, 16), 9), _rand((16, 32), 10, 0.5), _rand((32, 16), 11, 0.5)
    good = mlp.forward(X, A, B, kind)["O"]
    bad = mlp.forward_input_split(X, A, B, 2, kind)
    assert np.abs(good - bad).max() > 0.05 * np.abs(good).max()


# ---------------------------------------------------------------- collectives

@pytest.mark.parametrize("t", [2, 4, 8])
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_allreduce_is_allgather_of_reducescatter(t, dtype):
    parts = [np.random.default_rng(20 + i).standard_normal((8 * t, 24)).astype(dtype) for i in range(t)]
    ar = collectives.all_reduce(parts)
    ag_rs = collectives.all_gather(collectives.reduce_scatter(parts, axis=0), axis=0)
    for a, b in zip(ar, ag_rs):
        assert a.dtype == dtype and np.array_equal(a, b)
    # and the sum really is the sum (in rank order)
    assert np.allclose(ar[0], np.sum(np.stack(parts).astype(np.float64), axis=0), rtol=1e-5, atol=1e-5)


# ---------------------------------------------------------------- LayerNorm

def test_layernorm_statistics():
    x = _rand((64, 256), 12, 3.0) + 5.0
    eps = 1e-5
    y = sp.layernorm(x, np.ones(256), np.zeros(256), eps)
    var = x.var(axis=1)
    assert np.abs(y.mean(axis=1)).max() < 1e-12
    assert np.abs(y.var(axis=1) - var / (var + eps)).max() < 1e-12


def test_layernorm_matches_torch():
    x = _rand((32, 128), 13)
    g, b = _rand(128, 14), _rand(128, 15)
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (128,), torch.tensor(g), torch.tensor(b), 1e-5).numpy()
    assert np.abs(sp.layernorm(x, g, b, 1e-5) - ref).max() < 1e-12


# ---------------------------------------------------------------- dropout hash

def test_splitmix64_two_restatements_agree():
    keys = [0, 1, 2, 0xFFFFFFFFFFFFFFFF, 0x9E3779B97F4A7C15, 1 << 63, 12345678901234567] + \
           np.random.default_rng(16).integers(0, 2**63, size=4000, dtype=np.uint64).tolist()
    vec = sp.splitmix64(np.array(keys, dtype=np.uint64))
    assert [int(v) for v in vec] == [sp.splitmix64_scalar(int(k)) for k in keys]


def test_splitmix64_zero_state_closed_form():
    # The mixer maps 0 to 0, so the state that the golden-gamma step carries to 0
    # must hash to 0: this fails if the increment is dropped or has the wrong value.
    assert sp.splitmix64_scalar((1 << 64) - 0x9E3779B97F4A7C15) == 0
    assert int(sp.splitmix64(np.array([(1 << 64) - 0x9E3779B97F4A7C15], dtype=np.uint64))[0]) == 0
    assert sp.splitmix64_scalar(0) != 0


# Published SplitMix64 output streams. A generator seeded with s advances its state by the golden
# gamma and returns the mix of the new state, so its k-th output (k = 0, 1, ...) is the oracle's
# splitmix64 of s + k * gamma. The values are the ones printed for the published generator
# (Vigna's splitmix64.c seeded with 0, and the Rosetta Code "Pseudo-random numbers/Splitmix64"
# task seeded with 1234567), typed here by hand. A wrong multiplier, shift or increment in the
# oracle changes every one of them.
_SPLITMIX64_KNOWN = {
    0: [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC,
        0x1B39896A51A8749B],
    1234567: [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
              16408922859458223821],
}


@pytest.mark.parametrize("seed", sorted(_SPLITMIX64_KNOWN))
def test_splitmix64_published_output_stream(seed):
    gamma, mask = 0x9E3779B97F4A7C15, (1 << 64) - 1
    states = [(seed + k * gamma) & mask for k in range(5)]
    want = _SPLITMIX64_KNOWN[seed]
    assert [sp.splitmix64_scalar(s) for s in states] == want
    assert [int(v) for v in sp.splitmix64(np.array(states, dtype=np.uint64))] == want


def test_drop_threshold():
    assert sp.drop_threshold(0.1) == 0x1999999999999A00
    assert sp.drop_threshold(0.0) == 0
    assert sp.drop_threshold(0.5) == 1 << 63
    with pytest.raises(ValueError):
        sp.drop_threshold(1.0)


def test_dropout_kept_fraction():
    N = 2 * 4096 * 4096
    dropped = sp.drop_mask(np.arange(N, dtype=np.uint64), 0, 0.1)
    sigma = math.sqrt(0.1 * 0.9 / N)
    assert abs(dropped.mean() - 0.1) < 5 * sigma


def test_dropout_p0_is_plain_residual():
    x, y = _rand((4, 64), 17), _rand((4, 64), 18)
    out = sp.dropout_residual(x, y, 0, 0.0, np.arange(256, dtype=np.uint64).reshape(4, 64))
    assert np.array_equal(out, x + y)


@pytest.mark.parametrize("p", [0.1, 0.25, 0.5])
def test_inverted_dropout_preserves_the_mean(p):
    # Dropout scales kept elements so that the expected output equals the input ("Megatron 训练"
    # notes, Dropout section: torch.nn.Dropout semantics). With x = 0 and y = 1 the output is
    # keep / (1 - p), whose mean over N elements is 1 within 5 sigma, sigma^2 = p / ((1 - p) N);
    # dropped elements are exactly the residual and kept ones all carry one common value.
    N = 1 << 22
    flat = np.arange(N, dtype=np.uint64)
    x, y = np.zeros(N), np.ones(N)
    out = sp.dropout_residual(x, y, 5, p, flat)
    dropped = sp.drop_mask(flat, 5, p)
    assert abs(out.mean() - 1.0) < 5 * math.sqrt(p / ((1.0 - p) * N))
    assert np.array_equal(out[dropped], x[dropped])
    kept = out[~dropped]
    assert kept.min() == kept.max() > 1.0


def test_pack_mask_bits():
    m = np.random.default_rng(19).random(200) < 0.3
    words = sp.pack_mask_bits(m)
    unpacked = np.unpackbits(words.view(np.uint8), bitorder="little")[:200].astype(bool)
    assert words.dtype == np.uint32 and words.size == 7 and np.array_equal(unpacked, m)


# ---------------------------------------------------------------- SP block

@pytest.mark.parametrize("t", [2, 4, 8])
def test_sp_block_ranks_equal_unsharded(t):
    b, s, h, m = 2, 16, 32, 64
    x = _rand((b, s, h), 21)
    A, B = _rand((h, m), 22, 0.2), _rand((m, h), 23, 0.2)
    g, be = 1.0 + 0.1 * _rand(h, 24), 0.1 * _rand(h, 25)
    ref = sp.sp_block(x, g, be, 1e-5, A, B, 0.1, 7, "tanh")
    got = sp.sp_block_ranks(wl.to_shards(x, t), g, be, 1e-5, A, B, 0.1, 7, "tanh")
    assert np.abs(wl.from_shards(got) - ref["out"]).max() < 1e-12
    # the mask differs between shards (per-rank RNG domains) and is not all-or-nothing
    d = ref["dropped"]
    assert 0 < d.mean() < 0.3 and not np.array_equal(d[:, : s // t], d[:, s // t: 2 * s // t])


# ---------------------------------------------------------------- input generator

def test_bf16_rounding_matches_torch_and_ties_to_even():
    v = np.array([1 + 2**-8, 1 + 3 * 2**-8, -1 - 2**-8, 3.14159, 1e-30, 65504.0], dtype=np.float32)
    ours = wl.round_to_bf16(v)
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)
    assert ours[0] == 1.0 and ours[1] == 1 + 2**-6
    r = np.random.default_rng(26).standard_normal(100000).astype(np.float32)
    assert np.array_equal(wl.round_to_bf16(r), torch.tensor(r).to(torch.bfloat16).to(torch.float32).numpy())


def test_inputs_deterministic_and_chunk_invariant(monkeypatch):
    a = wl.mlp_inputs(wl.SINGLE_BLOCK)
    monkeypatch.setattr(wl, "_CHUNK_ELEMS", 1000)
    b = wl.mlp_inputs(wl.SINGLE_BLOCK)
    for k in "XABG":
        assert np.array_equal(a[k], b[k])
    assert abs(a["A"].std() - 0.02) < 1e-3 and abs(a["X"].std() - 1.0) < 1e-2


def test_shard_layout_roundtrip():
    x = _rand((2, 12, 5), 27)
    xs = wl.to_shards(x, 4)
    assert xs.shape == (4, 2, 3, 5)
    assert np.array_equal(xs[2, 1, 0], x[1, 6])
    assert np.array_equal(wl.from_shards(xs), x)


# ---------------------------------------------------------------- SP block backward

def _sp_small(seed=30):
    b, s, h, m = 1, 4, 8, 16
    x = _rand((b, s, h), seed) * 2.0 + 0.3
    A, B = _rand((h, m), seed + 1, 0.4), _rand((m, h), seed + 2, 0.4)
    g, be = 1.0 + 0.2 * _rand(h, seed + 3), 0.2 * _rand(h, seed + 4)
    G = _rand((b, s, h), seed + 5)
    return x, g, be, A, B, G


@pytest.mark.parametrize("kind", KINDS)
def test_sp_backward_matches_finite_differences(kind):
    x, g, be, A, B, G = _sp_small()
    p, seed, eps = 0.3, 5, 1e-5
    grads = sp.sp_block_backward(x, g, be, eps, A, B, p, seed, kind, G)
    loss = lambda x_, g_, b_, A_, B_: float((sp.sp_block(x_, g_, b_, eps, A_, B_, p, seed, kind)["out"] * G).sum())
    args = {"x": x, "g": g, "be": be, "A": A, "B": B}
    keys = {"x": "dx", "g": "dgamma", "be": "dbeta", "A": "dA", "B": "dB"}
    hstep = 1e-6
    for name, key in keys.items():
        arr = args[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            ap, am = dict(args), dict(args)
            ap[name], am[name] = arr.copy(), arr.copy()
            ap[name][idx] += hstep
            am[name][idx] -= hstep
            fd[idx] = (loss(ap["x"], ap["g"], ap["be"], ap["A"], ap["B"]) -
                       loss(am["x"], am["g"], am["be"], am["A"], am["B"])) / (2 * hstep)
        err = np.abs(fd - grads[key]).max() / np.abs(grads[key]).max()
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("kind", KINDS)
def test_sp_backward_matches_torch_autograd(kind):
    x, g, be, A, B, G = _sp_small(40)
    p, seed, eps = 0.25, 9, 1e-5
    b, s, h = x.shape
    keep = ~sp.drop_mask(np.arange(b * s * h, dtype=np.uint64).reshape(b, s, h), seed, p)
    tx, tg, tb, tA, tB = (torch.tensor(a, requires_grad=True) for a in (x, g, be, A, B))
    xn = torch.nn.functional.layer_norm(tx, (h,), tg, tb, eps)
    o = torch.nn.functional.gelu(xn @ tA, approximate="none" if kind == "erf" else "tanh") @ tB
    out = tx + torch.tensor(keep) * o / (1 - p)
    out.backward(torch.tensor(G))
    ref = sp.sp_block_backward(x, g, be, eps, A, B, p, seed, kind, G)
    for key, t in (("dx", tx), ("dgamma", tg), ("dbeta", tb), ("dA", tA), ("dB", tB)):
        assert np.abs(ref[key] - t.grad.numpy()).max() < 1e-11, key


def test_layernorm_gradient_orthogonal_to_one_and_xhat():
    # "Megatron 训练" notes, LayerNorm section: g_LN has no component along 1 or x_hat. The
    # x_hat part is exact for eps = 0; with eps > 0 it is off by the factor eps / (var + eps).
    x = _rand((16, 64), 50) * 3 + 1
    dy = _rand((16, 64), 51)
    for eps in (0.0, 1e-5):
        dx, _, _ = sp.layernorm_backward(x, np.ones(64), eps, dy)
        var = x.var(1, keepdims=True)
        xhat = (x - x.mean(1, keepdims=True)) / np.sqrt(var + eps)
        assert np.abs(dx.sum(1)).max() < 1e-12
        bound = 1e-12 + (eps / (var.min() + eps)) * np.abs(dx * xhat).sum(1).max() * 2
        assert np.abs((dx * xhat).sum(1)).max() < max(bound, 1e-11)


# ---------------------------------------------------------------- biases

@pytest.mark.parametrize("kind", KINDS)
def test_biases_match_torch_autograd(kind):
    n, d, m = 9, 12, 24
    X, A, B, G = _rand((n, d), 60), _rand((d, m), 61, 0.3), _rand((m, d), 62, 0.3), _rand((n, d), 63)
    b1, b2 = _rand(m, 64, 0.5), _rand(d, 65, 0.5)
    tX, tA, tB, tb1, tb2 = (torch.tensor(a, requires_grad=True) for a in (X, A, B, b1, b2))
    lin1 = torch.nn.functional.linear(tX, tA.T, tb1)          # torch's [out, in] weight convention
    O = torch.nn.functional.linear(torch.nn.functional.gelu(lin1, approximate="none" if kind == "erf" else "tanh"),
                                   tB.T, tb2)
    O.backward(torch.tensor(G))
    f = mlp.forward(X, A, B, kind, b1, b2)
    g = mlp.backward(X, A, B, G, kind, b1)
    assert np.abs(f["O"] - O.detach().numpy()).max() < 1e-12
    for key, t in (("dX", tX), ("dA", tA), ("dB", tB), ("db1", tb1), ("db2", tb2)):
        assert np.abs(g[key] - t.grad.numpy()).max() < 1e-11, key


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_biased_shard_sum_adds_row_bias_once(t):
    X, A, B, G = _rand((6, 16), 66), _rand((16, 32), 67, 0.3), _rand((32, 16), 68, 0.3), _rand((6, 16), 69)
    b1, b2 = _rand(32, 70), _rand(16, 71)
    ref_f, ref_b = mlp.forward(X, A, B, "tanh", b1, b2), mlp.backward(X, A, B, G, "tanh", b1)
    sh_f, sh_b = mlp.forward_sharded(X, A, B, t, "tanh", b1, b2), mlp.backward_sharded(X, A, B, G, t, "tanh", b1)
    assert np.abs(sh_f["O"] - ref_f["O"]).max() < 1e-12
    for key in ("dX", "dA", "dB", "db1", "db2"):
        assert np.abs(sh_b[key] - ref_b[key]).max() < 1e-12
    if t > 1:  # adding b2 in every shard instead of once after the sum is the mistake this rules out
        wrong = mlp.forward_sharded(X, A, B, t, "tanh", b1, None)["O"] + t * b2
        assert np.abs(wrong - ref_f["O"]).max() > 0.1


# ---------------------------------------------------------------- fp32 main_grad accumulation

@pytest.mark.parametrize("chunks", [1, 2, 3])
def test_microbatch_accumulation_equals_full_batch(chunks):
    # Weight gradients are sums over tokens, so adding the gradients of micro-batches into an
    # fp32 buffer (Megatron's main_grad with gradient_accumulation_fusion) gives the gradient of
    # the concatenated batch; the activation gradient dX stays per micro-batch.
    X, A, B, G = _rand((12, 16), 80), _rand((16, 32), 81, 0.3), _rand((32, 16), 82, 0.3), _rand((12, 16), 83)
    full = mlp.backward(X, A, B, G, "erf")
    acc_dA, acc_dB = np.zeros_like(full["dA"]), np.zeros_like(full["dB"])
    for Xc, Gc in zip(np.array_split(X, chunks), np.array_split(G, chunks)):
        g = mlp.backward(Xc, A, B, Gc, "erf")
        acc_dA += g["dA"]
        acc_dB += g["dB"]
    assert np.abs(acc_dA - full["dA"]).max() < 1e-12 and np.abs(acc_dB - full["dB"]).max() < 1e-12


# ---------------------------------------------------------------- tensor-parallel attention

from oracle import attention as oattn  # noqa: E402


def _attn_small(seed=90, b=2, s=5, h=16, heads=4):
    X = _rand((b, s, h), seed)
    Wqkv, Wo = _rand((h, 3 * h), seed + 1, 0.3), _rand((h, h), seed + 2, 0.3)
    G = _rand((b, s, h), seed + 3)
    return X, Wqkv, Wo, heads, G


def test_attention_matches_torch_autograd():
    X, Wqkv, Wo, heads, G = _attn_small()
    b, s, h = X.shape
    dh = h // heads
    tX, tW, tO = (torch.tensor(a, requires_grad=True) for a in (X, Wqkv, Wo))
    qkv = (tX @ tW).reshape(b, s, heads, 3, dh).permute(3, 0, 2, 1, 4)   # the note's reshape/permute
    q, k, v = qkv[0], qkv[1], qkv[2]
    att = torch.softmax((q @ k.transpose(-2, -1)) * dh ** -0.5, dim=-1)
    Y = (att @ v).transpose(1, 2).reshape(b, s, h) @ tO
    Y.backward(torch.tensor(G))
    f = oattn.forward(X, Wqkv, Wo, heads)
    g = oattn.backward(X, Wqkv, Wo, heads, G)
    assert np.abs(f["Y"] - Y.detach().numpy()).max() < 1e-12
    for key, t in (("dX", tX), ("dWqkv", tW), ("dWo", tO)):
        assert np.abs(g[key] - t.grad.numpy()).max() < 1e-11, key


def test_attention_matches_library_sdpa():
    X, Wqkv, Wo, heads, _ = _attn_small(95)
    b, s, h = X.shape
    dh = h // heads
    qkv = torch.tensor(X @ Wqkv).reshape(b, s, heads, 3, dh).permute(3, 0, 2, 1, 4)
    o = torch.nn.functional.scaled_dot_product_attention(qkv[0], qkv[1], qkv[2])
    ref = o.transpose(1, 2).reshape(b, s, h).numpy() @ Wo
    assert np.abs(oattn.forward(X, Wqkv, Wo, heads)["Y"] - ref).max() < 1e-12


@pytest.mark.parametrize("t", [1, 2, 4])
def test_attention_head_shards_sum_to_unsharded(t):
    X, Wqkv, Wo, heads, _ = _attn_small(100)
    assert np.abs(oattn.forward_sharded(X, Wqkv, Wo, heads, t) - oattn.forward(X, Wqkv, Wo, heads)["Y"]).max() < 1e-12


def test_attention_backward_finite_differences():
    X, Wqkv, Wo, heads, G = _attn_small(110, b=1, s=3, h=8, heads=2)
    g = oattn.backward(X, Wqkv, Wo, heads, G)
    loss = lambda X_, W_, O_: float((oattn.forward(X_, W_, O_, heads)["Y"] * G).sum())
    for name, key in (("X", "dX"), ("W", "dWqkv"), ("O", "dWo")):
        args = {"X": X, "W": Wqkv, "O": Wo}
        arr = args[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            ap, am = dict(args), dict(args)
            ap[name], am[name] = arr.copy(), arr.copy()
            ap[name][idx] += 1e-6
            am[name][idx] -= 1e-6
            fd[idx] = (loss(ap["X"], ap["W"], ap["O"]) - loss(am["X"], am["W"], am["O"])) / 2e-6
        assert np.abs(fd - g[key]).max() / np.abs(g[key]).max() < 1e-6, name


def test_softmax_rows_sum_to_one_and_shift_invariant():
    S = _rand((3, 7, 9), 120) * 5
    P = oattn.softmax(S)
    assert np.abs(P.sum(-1) - 1).max() < 1e-14
    assert np.abs(oattn.softmax(S + 100.0) - P).max() < 1e-14


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_unit_mean_square():
    # With gamma = 1 and eps = 0 every output row has mean square exactly 1; a row scaled by
    # any positive factor gives the same output (scale control), a shifted row does not.
    x = _rand((32, 96), 80) * 4 + 2
    y = rmsnorm.rmsnorm(x, np.ones(96), 0.0)
    assert np.abs((y * y).mean(axis=1) - 1.0).max() < 1e-12
    assert np.abs(rmsnorm.rmsnorm(7.5 * x, np.ones(96), 0.0) - y).max() < 1e-12
    assert np.abs(rmsnorm.rmsnorm(x + 1.0, np.ones(96), 0.0) - y).max() > 1e-3


def test_rmsnorm_matches_torch():
    x = _rand((24, 128), 81)
    g = _rand(128, 82)
    for eps in (1e-6, 1e-2):
        ref = torch.nn.functional.rms_norm(torch.tensor(x), (128,), torch.tensor(g), eps).numpy()
        assert np.abs(rmsnorm.rmsnorm(x, g, eps) - ref).max() < 1e-12


def test_rmsnorm_is_not_layernorm():
    # Dropping the mean matters: on rows with a non-zero mean the two norms differ, and they
    # agree on rows whose mean is zero (then mean(x^2) is the variance).
    x = _rand((8, 64), 83) + 3.0
    g, z = np.ones(64), np.zeros(64)
    assert np.abs(rmsnorm.rmsnorm(x, g, 1e-5) - sp.layernorm(x, g, z, 1e-5)).max() > 0.1
    xc = x - x.mean(axis=1, keepdims=True)
    assert np.abs(rmsnorm.rmsnorm(xc, g, 1e-5) - sp.layernorm(xc, g, z, 1e-5)).max() < 1e-12


def test_rmsnorm_backward_matches_torch_autograd():
    x = _rand((12, 80), 84) * 2 + 0.5
    g = _rand(80, 85)
    dy = _rand((12, 80), 86)
    tx, tg = torch.tensor(x, requires_grad=True), torch.tensor(g, requires_grad=True)
    torch.nn.functional.rms_norm(tx, (80,), tg, 1e-5).backward(torch.tensor(dy))
    dx, dg = rmsnorm.rmsnorm_backward(x, g, 1e-5, dy)
    assert np.abs(dx - tx.grad.numpy()).max() < 1e-12
    assert np.abs(dg - tg.grad.numpy()).max() < 1e-12


def test_rmsnorm_backward_finite_differences():
    x = _rand((3, 16), 87) + 0.3
    g = _rand(16, 88)
    dy = _rand((3, 16), 89)
    eps, h = 1e-3, 1e-6
    dx, dg = rmsnorm.rmsnorm_backward(x, g, eps, dy)
    f = lambda xx, gg: float((rmsnorm.rmsnorm(xx, gg, eps) * dy).sum())  # noqa: E731
    for idx in [(0, 0), (1, 7), (2, 15)]:
        e = np.zeros_like(x)
        e[idx] = h
        assert abs((f(x + e, g) - f(x - e, g)) / (2 * h) - dx[idx]) < 1e-7
    for j in (0, 9):
        e = np.zeros_like(g)
        e[j] = h
        assert abs((f(x, g + e) - f(x, g - e)) / (2 * h) - dg[j]) < 1e-7


def test_rmsnorm_gradient_orthogonal_to_x_only():
    # Scale invariance (eps = 0): the gradient has no component along x (x_hat); unlike
    # LayerNorm's it keeps its component along 1.
    x = _rand((16, 64), 90) * 3 + 1
    dy = _rand((16, 64), 91)
    dx, _ = rmsnorm.rmsnorm_backward(x, np.ones(64), 0.0, dy)
    assert np.abs((dx * x).sum(1)).max() < 1e-11
    assert np.abs(dx.sum(1)).max() > 1e-3


def test_attention_softmax_gradient_rowsum_identity():
    # The kernels take rowsum(P * dP) as rowsum(dO * O) per head and query row: with O = P V and
    # dP = dO V^T the two are the same sum, sum_j P_ij (dO_i . V_j) = dO_i . (sum_j P_ij V_j).
    # Checked on the oracle's own P, dO and V (the oracle itself uses the first form).
    X, Wqkv, Wo, heads, G = _attn_small(120)
    b, s, h = X.shape
    dh = h // heads
    f = oattn.forward(X, Wqkv, Wo, heads)
    g = oattn.backward(X, Wqkv, Wo, heads, G)
    v = np.transpose(f["QKV"].reshape(b, s, heads, 3, dh)[:, :, :, 2, :], (0, 2, 1, 3))
    dOh = np.transpose(g["dO"].reshape(b, s, heads, dh), (0, 2, 1, 3))
    Oh = np.transpose(f["O"].reshape(b, s, heads, dh), (0, 2, 1, 3))
    dP = dOh @ np.swapaxes(v, -1, -2)
    lhs = (f["P"] * dP).sum(axis=-1)
    rhs = (dOh * Oh).sum(axis=-1)
    assert np.abs(lhs - rhs).max() < 1e-12 * max(1.0, np.abs(lhs).max())
    assert np.abs(lhs).max() > 1e-3  # not a vacuous zero
