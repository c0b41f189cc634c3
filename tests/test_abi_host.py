"""Host-side checks of the C ABI that need no GPU: the library builds and loads, it
exports every entry point include/tpmlp.h declares, and bad arguments are rejected
with the documented status before anything touches the device."""
import ctypes
import os
import re
import subprocess

import pytest

from tensor_transformer_mlp_gb300 import _binding, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpmlp.h")

OK, INVALID, SHAPE, DTYPE, ALIGN, CUDA, TIMEOUT, WORKSPACE = range(8)
ERF, TANH = 0, 1
F32, BF16 = 0, 1
FAKE = 0x10000  # never dereferenced: every call below fails validation first


def declared_functions():
    text = open(HEADER).read()
    return set(re.findall(r"^\s*(?:const\s+char\s*\*|size_t|tpmlp_status)\s+(tpmlp_\w+)\s*\(", text, re.M))


@pytest.fixture(scope="module")
def lib():
    return _binding.load_library(build_if_missing=True)


def test_header_and_binding_agree():
    assert declared_functions() == set(_binding.SIGNATURES)


# C parameter and return types of include/tpmlp.h -> the ctypes type the binding must declare.
_CTYPE = {"const void*": ctypes.c_void_p, "void*": ctypes.c_void_p, "const float*": ctypes.c_void_p,
          "float*": ctypes.c_void_p, "uint32_t*": ctypes.c_void_p, "const uint32_t*": ctypes.c_void_p, "int64_t": ctypes.c_int64, "int": ctypes.c_int,
          "tpmlp_gelu": ctypes.c_int, "tpmlp_dtype": ctypes.c_int, "tpmlp_rs_mode": ctypes.c_int,
          "float": ctypes.c_float, "double": ctypes.c_double, "uint64_t": ctypes.c_uint64, "size_t": ctypes.c_size_t,
          "tpmlp_status": ctypes.c_int, "const char*": ctypes.c_char_p}


def declared_signatures():
    """{name: (return type, [parameter types])} parsed from the header's prototypes."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for ret, name, params in re.findall(r"(const\s+char\s*\*|size_t|tpmlp_status)\s+(tpmlp_\w+)\s*\(([^)]*)\)\s*;",
                                        text, re.S):
        types = []
        for p in params.split(","):
            p = " ".join(p.split())
            if p and p != "void":
                types.append(p.rsplit(" ", 1)[0].replace(" *", "*") if not p.endswith("*") else p)
        out[name] = (" ".join(ret.split()).replace(" *", "*"), types)
    return out


def test_binding_argument_types_match_header():
    # A float declared where the library takes a double (or an int where it takes int64_t)
    # passes the wrong bits without any error, so every parameter is checked.
    decl = declared_signatures()
    assert set(decl) == declared_functions()
    for name, (ret, params) in decl.items():
        restype, argtypes = _binding.SIGNATURES[name]
        assert restype is _CTYPE[ret], name
        assert [_CTYPE[p] for p in params] == list(argtypes), name


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(tpmlp_\w+)$", out, re.M))
    assert declared_functions() <= exported
    for name in declared_functions():
        assert getattr(lib, name) is not None


def fwd(lib, X=FAKE, A=FAKE, B=FAKE, O=FAKE, Z=FAKE, Y=FAKE, n=256, d=512, m=1024, t=2, g=TANH, dt=BF16):
    return lib.tpmlp_forward(X, A, B, O, Z, Y, n, d, m, t, g, dt, None)


def test_forward_validation(lib):
    assert fwd(lib, X=None) == INVALID
    assert fwd(lib, Y=None) == INVALID
    assert fwd(lib, m=1000, t=3) == SHAPE          # uneven split
    assert fwd(lib, t=0) == SHAPE
    assert fwd(lib, d=500) == SHAPE                # bf16 rows must be 16-byte multiples
    assert fwd(lib, n=-1) == SHAPE
    assert fwd(lib, A=FAKE + 8) == ALIGN
    assert fwd(lib, g=7) == INVALID
    assert fwd(lib, dt=5) == DTYPE
    assert b"divisible" in (fwd(lib, m=1000, t=3) and lib.tpmlp_last_error())
    assert fwd(lib, n=0) == OK                     # nothing to do, nothing launched


def test_biased_validation(lib):
    base = [FAKE] * 3
    assert lib.tpmlp_forward_biased(*base, None, FAKE, *([FAKE] * 3), 8, 64, 64, 2, TANH, BF16, None) == INVALID
    assert lib.tpmlp_forward_biased(*base, FAKE + 8, FAKE, *([FAKE] * 3), 8, 64, 64, 2, TANH, BF16, None) == ALIGN
    args = [FAKE] * 9
    assert lib.tpmlp_backward_biased(*args, None, FAKE, 8, 64, 64, 2, TANH, BF16, FAKE, 1 << 30, None) == INVALID
    need = lib.tpmlp_backward_biased_workspace_size(1000, 64, 128, BF16)
    assert need > lib.tpmlp_backward_workspace_size(1000, 128, BF16)
    assert lib.tpmlp_backward_biased(*args, FAKE, FAKE, 1000, 64, 128, 2, TANH, BF16, FAKE, need - 1,
                                     None) == WORKSPACE


def test_backward_validation(lib):
    args = [FAKE] * 9 + [256, 512, 1024, 2, TANH, BF16]
    assert lib.tpmlp_backward(*args, None, 0, None) == WORKSPACE
    assert lib.tpmlp_backward(*args, FAKE, 100, None) == WORKSPACE
    assert lib.tpmlp_backward(*args, FAKE + 16, 1 << 30, None) == ALIGN
    bad = list(args)
    bad[4] = None  # Z_save (n > 0)
    assert lib.tpmlp_backward(*bad, FAKE, 1 << 30, None) == INVALID
    assert lib.tpmlp_backward_workspace_size(256, 1024, BF16) == 256 * 1024 * 2
    assert lib.tpmlp_backward_workspace_size(0, 1024, BF16) == 0


def test_backward_noalloc_validation(lib):
    # The no-allocation backward keeps D in a 64 MiB static array. Everything below is rejected on
    # the host before any device work, so fake pointers are safe here; the accepted edge case
    # (exactly 64 MiB) runs on the GPU in test_zz_no_alloc.py.
    def noalloc(n, d=64, m=4096, t=8, dt=BF16, Z=FAKE):
        args = [FAKE] * 4 + [Z] + [FAKE] * 4
        return lib.tpmlp_backward_noalloc(*args, n, d, m, t, TANH, dt, None)

    assert noalloc(8193) == WORKSPACE                 # bf16: one row past 8192 x 4096 x 2 bytes
    assert b"static scratch" in lib.tpmlp_last_error()
    assert noalloc(4097, dt=F32) == WORKSPACE         # fp32 D takes twice the bytes per element
    assert noalloc(16384, d=8192, m=32768) == WORKSPACE
    # Bad arguments get tpmlp_backward's status even when D would not fit either.
    assert noalloc(1 << 20, m=4100, t=8) == SHAPE     # m % t
    assert lib.tpmlp_backward(*([FAKE] * 9), 1 << 20, 64, 4100, 8, TANH, BF16, FAKE, 1 << 40, None) == SHAPE
    assert noalloc(1 << 20, d=-1) == SHAPE
    assert noalloc(1 << 20, Z=None) == INVALID
    assert noalloc(1 << 20, Z=FAKE + 8) == ALIGN
    assert noalloc(1 << 20, dt=9) == DTYPE


def sp(lib, t=4, s=64, h=256, m=512, p=0.1, mask=FAKE, ws=FAKE, wsb=1 << 30, rs=0, eps=1e-5):
    return lib.tpmlp_sp_block(FAKE, FAKE, FAKE, eps, FAKE, FAKE, p, 0, FAKE, mask, None, None, 2, s, h, m, t, TANH,
                              BF16, rs, ws, wsb, None)


def test_sp_block_validation(lib):
    assert sp(lib, t=1) == SHAPE                   # sequence parallelism needs a TP group
    assert b"t >= 2" in lib.tpmlp_last_error()
    assert sp(lib, s=66) == SHAPE                  # s % t
    assert sp(lib, p=1.0) == INVALID
    assert sp(lib, p=-0.1) == INVALID
    assert sp(lib, eps=0.0) == INVALID
    assert sp(lib, h=264) == SHAPE                 # mask words need h % 32 == 0
    assert sp(lib, rs=9) == INVALID
    assert sp(lib, ws=None) == WORKSPACE
    need = lib.tpmlp_sp_block_workspace_size(2, 64, 256, 512, 4, BF16, 0)
    assert need > 0 and sp(lib, wsb=need - 1) == WORKSPACE
    assert lib.tpmlp_sp_block_workspace_size(2, 64, 256, 512, 4, BF16, 1) > need
    # only one of the two activation saves
    assert lib.tpmlp_sp_block(FAKE, FAKE, FAKE, 1e-5, FAKE, FAKE, 0.1, 0, FAKE, FAKE, FAKE, None, 2, 64, 256, 512, 4,
                              TANH, BF16, 0, FAKE, 1 << 30, None) == INVALID


def test_sp_block_backward_validation(lib):
    def bwd(h=256, t=4, ws=FAKE, wsb=1 << 30, p=0.1, Z=FAKE, mask=None):
        return lib.tpmlp_sp_block_backward(FAKE, FAKE, FAKE, 1e-5, FAKE, FAKE, p, 0, mask, Z, FAKE, FAKE, FAKE, FAKE,
                                           FAKE, FAKE, FAKE, 2, 64, h, 512, t, TANH, BF16, ws, wsb, None)
    assert bwd(t=1) == SHAPE
    assert bwd(h=8200) == SHAPE                    # widths up to 8192
    assert bwd(p=1.0) == INVALID
    assert bwd(Z=None) == INVALID
    assert bwd(h=264, mask=FAKE) == SHAPE           # mask words need h % 32 == 0
    assert bwd(mask=FAKE + 2) == SHAPE             # 4-byte aligned mask words
    assert bwd(ws=None) == WORKSPACE
    need = lib.tpmlp_sp_block_backward_workspace_size(2, 64, 256, 512, 4, BF16)
    assert need > 0 and bwd(wsb=need - 1) == WORKSPACE


def test_elementwise_validation(lib):
    assert lib.tpmlp_sp_gather(FAKE, FAKE, 2, 64, 256, 1, BF16, None) == SHAPE
    assert lib.tpmlp_sp_gather(FAKE, None, 2, 64, 256, 4, BF16, None) == INVALID
    assert lib.tpmlp_sp_gather(None, None, 0, 64, 256, 4, BF16, None) == OK  # no rows, nothing launched
    assert lib.tpmlp_sp_reduce_scatter(FAKE, FAKE, 2, 63, 256, 4, BF16, None) == SHAPE
    assert lib.tpmlp_sp_dropout_residual(FAKE, FAKE, FAKE, None, 1.5, 0, 2, 64, 256, 4, BF16, None) == INVALID
    assert lib.tpmlp_sp_layernorm(FAKE, FAKE, FAKE, 1e-5, FAKE, 4, 256, 9, None) == DTYPE
    assert lib.tpmlp_sp_layernorm(FAKE + 2, FAKE, FAKE, 1e-5, FAKE, 4, 256, BF16, None) == ALIGN


def test_wait_timeout_check_validation(lib):
    assert lib.tpmlp_check_wait_timeout(10, None) == INVALID
    assert lib.tpmlp_check_wait_timeout(5_000_000_000, None) == INVALID


def test_attention_validation(lib):
    P = [FAKE] * 7
    assert lib.tpmlp_attention_forward(*P, 2, 64, 256, 4, 3, BF16, FAKE, 1 << 30, None) == SHAPE   # heads % t
    assert lib.tpmlp_attention_forward(*P, 2, 64, 256, 4, 2, F32, FAKE, 1 << 30, None) == DTYPE
    assert lib.tpmlp_attention_forward(*P, 2, 60, 256, 4, 2, BF16, FAKE, 1 << 30, None) == SHAPE   # s % 8
    assert lib.tpmlp_attention_forward(*P, 2, 64, 256, 4, 2, BF16, None, 0, None) == WORKSPACE
    need = lib.tpmlp_attention_backward_workspace_size(2, 64, 256, 4, BF16)
    assert lib.tpmlp_attention_backward(*([FAKE] * 10), 2, 64, 256, 4, 2, BF16, FAKE, need - 1, None) == WORKSPACE


def test_rmsnorm_validation(lib):
    assert lib.tpmlp_rmsnorm(FAKE, FAKE, 1e-5, FAKE, 4, 256, 9, None) == DTYPE
    assert lib.tpmlp_rmsnorm(FAKE, FAKE, 1e-5, FAKE, 4, 260, BF16, None) == SHAPE      # h % 8
    assert lib.tpmlp_rmsnorm(FAKE, FAKE, 1e-5, FAKE, 4, 8200, BF16, None) == SHAPE     # h > 8192
    assert lib.tpmlp_rmsnorm(FAKE, FAKE, 1e-5, FAKE, 4, 8192, F32, None) == SHAPE      # h > 4096 (fp32)
    assert lib.tpmlp_rmsnorm(FAKE, FAKE, 0.0, FAKE, 4, 256, BF16, None) == INVALID     # eps
    assert lib.tpmlp_rmsnorm(None, FAKE, 1e-5, FAKE, 4, 256, BF16, None) == INVALID
    assert lib.tpmlp_rmsnorm(FAKE + 8, FAKE, 1e-5, FAKE, 4, 256, BF16, None) == ALIGN
    need = lib.tpmlp_rmsnorm_backward_workspace_size(4, 256)
    assert need >= 2 * 256 * 4
    P = [FAKE] * 2
    assert lib.tpmlp_rmsnorm_backward(*P, 1e-5, FAKE, FAKE, FAKE, 4, 8200, BF16, FAKE, 1 << 30, None) == SHAPE
    # the LayerNorm backward step: same width rule, workspace, null and alignment checks
    lnb = lib.tpmlp_sp_layernorm_backward
    need = lib.tpmlp_sp_layernorm_backward_workspace_size(4, 256)
    assert lnb(FAKE, FAKE, 1e-5, FAKE, None, FAKE, FAKE, FAKE, 4, 8200, BF16, FAKE, 1 << 30, None) == SHAPE
    assert lnb(FAKE, FAKE, 1e-5, FAKE, None, FAKE, FAKE, None, 4, 256, BF16, FAKE, need, None) == INVALID
    assert lnb(FAKE, FAKE, 1e-5, FAKE, FAKE + 8, FAKE, FAKE, FAKE, 4, 256, BF16, FAKE, need, None) == ALIGN
    assert lnb(FAKE, FAKE, 1e-5, FAKE, None, FAKE, FAKE, FAKE, 4, 256, BF16, FAKE, need - 1, None) == WORKSPACE
    assert lnb(FAKE, FAKE, 0.0, FAKE, None, FAKE, FAKE, FAKE, 4, 256, BF16, FAKE, need, None) == INVALID
    dgg = lib.tpmlp_sp_dropout_grad_gather
    assert dgg(FAKE, FAKE, None, 1.0, 0, 2, 64, 256, 4, BF16, None) == INVALID       # p outside [0, 1)
    assert dgg(FAKE, FAKE, None, 0.1, 0, 2, 66, 256, 4, BF16, None) == SHAPE         # s % t
    assert dgg(FAKE, None, None, 0.1, 0, 2, 64, 256, 4, BF16, None) == INVALID
    assert dgg(FAKE, FAKE, FAKE, 0.1, 0, 2, 64, 264, 4, BF16, None) == SHAPE         # mask needs h % 32 == 0
    assert lib.tpmlp_rmsnorm_backward(*P, 1e-5, FAKE, FAKE, None, 4, 256, BF16, FAKE, need, None) == INVALID
    assert lib.tpmlp_rmsnorm_backward(*P, 1e-5, FAKE, FAKE, FAKE, 4, 256, BF16, FAKE, need - 1, None) == WORKSPACE
    assert lib.tpmlp_rmsnorm_backward(*P, 1e-5, FAKE, FAKE, FAKE, 4, 256, 7, FAKE, need, None) == DTYPE


def test_last_error_never_null(lib):
    assert isinstance(lib.tpmlp_last_error(), bytes)


def test_gemm_variant_validation(lib):
    # Only this call selects the GEMM kernel (no environment variable does); it touches no device.
    assert lib.tpmlp_set_gemm_variant(4, 1, 0) == INVALID
    assert lib.tpmlp_set_gemm_variant(1, -1, 0) == INVALID
    assert lib.tpmlp_set_gemm_variant(1, 1, 5000) == INVALID
    assert lib.tpmlp_set_gemm_variant(0, 0, -4) == OK
    assert lib.tpmlp_set_gemm_variant(1, 1, 0) == OK  # back to the defaults


def test_library_reads_no_environment_switch():
    # The shipped library's behaviour must not depend on the caller's environment.
    srcdir = os.path.join(ROOT, "tensor_transformer_mlp_gb300", "csrc")
    for name in os.listdir(srcdir):
        text = open(os.path.join(srcdir, name)).read()
        assert "getenv" not in text, name
