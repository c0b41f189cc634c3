"""Thin ctypes binding over libtpmlp.so (argument marshalling only).

Each function takes torch CUDA tensors, checks that their shapes and dtypes agree
with one another, and passes raw device pointers, sizes and the current CUDA
stream to the C entry point of the same name. Every step of the computation runs
in the library's kernels; if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

GELU = {"erf": 0, "tanh": 1}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
RS_MODE = {"fused": 0, "splitk": 1}
STATUS = {0: "TPMLP_OK", 1: "TPMLP_ERR_INVALID", 2: "TPMLP_ERR_SHAPE", 3: "TPMLP_ERR_DTYPE", 4: "TPMLP_ERR_ALIGN",
          5: "TPMLP_ERR_CUDA", 6: "TPMLP_ERR_TIMEOUT", 7: "TPMLP_ERR_WORKSPACE"}

# Every entry point declared in include/tpmlp.h, with its ctypes signature.
_P, _I64, _I, _F, _U64, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
_D = ctypes.c_double
SIGNATURES = {
    "tpmlp_forward": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P]),
    "tpmlp_forward_biased": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P]),
    "tpmlp_backward_workspace_size": (_SZ, [_I64, _I64, _I]),
    "tpmlp_backward_accumulate": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _SZ, _P]),
    "tpmlp_backward_biased_workspace_size": (_SZ, [_I64, _I64, _I64, _I]),
    "tpmlp_backward_biased": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _SZ,
                                   _P]),
    "tpmlp_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _SZ, _P]),
    "tpmlp_backward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P]),
    "tpmlp_sp_block_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I, _I, _I]),
    "tpmlp_sp_block": (_I, [_P, _P, _P, _F, _P, _P, _D, _U64, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I, _I, _I, _I,
                            _P, _SZ, _P]),
    "tpmlp_sp_block_backward_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I, _I]),
    "tpmlp_sp_block_backward": (_I, [_P, _P, _P, _F, _P, _P, _D, _U64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                     _I64, _I64, _I, _I, _I, _P, _SZ, _P]),
    "tpmlp_sp_layernorm": (_I, [_P, _P, _P, _F, _P, _I64, _I64, _I, _P]),
    "tpmlp_rmsnorm": (_I, [_P, _P, _F, _P, _I64, _I64, _I, _P]),
    "tpmlp_rmsnorm_backward_workspace_size": (_SZ, [_I64, _I64]),
    "tpmlp_rmsnorm_backward": (_I, [_P, _P, _F, _P, _P, _P, _I64, _I64, _I, _P, _SZ, _P]),
    "tpmlp_sp_layernorm_backward_workspace_size": (_SZ, [_I64, _I64]),
    "tpmlp_sp_layernorm_backward": (_I, [_P, _P, _F, _P, _P, _P, _P, _P, _I64, _I64, _I, _P, _SZ, _P]),
    "tpmlp_sp_dropout_grad_gather": (_I, [_P, _P, _P, _D, _U64, _I64, _I64, _I64, _I, _I, _P]),
    "tpmlp_sp_gather": (_I, [_P, _P, _I64, _I64, _I64, _I, _I, _P]),
    "tpmlp_sp_reduce_scatter": (_I, [_P, _P, _I64, _I64, _I64, _I, _I, _P]),
    "tpmlp_sp_dropout_residual": (_I, [_P, _P, _P, _P, _D, _U64, _I64, _I64, _I64, _I, _I, _P]),
    "tpmlp_attention_forward_workspace_size": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "tpmlp_attention_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _SZ, _P]),
    "tpmlp_attention_backward_workspace_size": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "tpmlp_attention_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _SZ,
                                      _P]),
    "tpmlp_last_error": (ctypes.c_char_p, []),
    "tpmlp_device_status": (_I, [_P, _I]),
    "tpmlp_check_wait_timeout": (_I, [_U64, _P]),
    "tpmlp_set_gemm_variant": (_I, [_I, _I, _I]),
}

_lib = None
_lock = threading.Lock()


class TpmlpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if it is missing or stale) libtpmlp.so and declare its signatures."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing and _build.is_stale():
                _build.build()
            if not os.path.exists(_build.LIB_PATH):
                raise RuntimeError(f"libtpmlp.so is missing at {_build.LIB_PATH}; run the build first")
            lib = ctypes.CDLL(_build.LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != 0:
        msg = load_library().tpmlp_last_error().decode(errors="replace")
        raise TpmlpError(status, msg)


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _cuda(*ts: torch.Tensor | None) -> None:
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in DTYPE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return DTYPE[t.dtype]


# ----------------------------------------------------------------------- C-ABI mirrors

def tpmlp_forward(X, A, B, O, Z_save, Y_save, t: int, gelu: str = "tanh", stream=None) -> None:
    n, d = X.shape
    m = A.shape[1]
    assert A.shape == (d, m) and B.shape == (m, d) and O.shape == (n, d) and Y_save.shape == (n, m)
    assert Z_save is None or Z_save.shape == (n, m)
    _cuda(X, A, B, O, Z_save, Y_save)
    _check(load_library().tpmlp_forward(_ptr(X), _ptr(A), _ptr(B), _ptr(O), _ptr(Z_save), _ptr(Y_save), n, d, m, t,
                                        GELU[gelu], _dt(X), _stream(stream)))


def tpmlp_forward_biased(X, A, B, bias1, bias2, O, Z_save, Y_save, t: int, gelu: str = "tanh", stream=None) -> None:
    n, d = X.shape
    m = A.shape[1]
    assert A.shape == (d, m) and B.shape == (m, d) and O.shape == (n, d) and Y_save.shape == (n, m)
    assert bias1.shape == (m,) and bias2.shape == (d,) and bias1.dtype == X.dtype and bias2.dtype == X.dtype
    assert Z_save is None or Z_save.shape == (n, m)
    _cuda(X, A, B, bias1, bias2, O, Z_save, Y_save)
    _check(load_library().tpmlp_forward_biased(_ptr(X), _ptr(A), _ptr(B), _ptr(bias1), _ptr(bias2), _ptr(O),
                                               _ptr(Z_save), _ptr(Y_save), n, d, m, t, GELU[gelu], _dt(X),
                                               _stream(stream)))


def tpmlp_backward_accumulate(X, A, B, G, Z_save, Y_save, dX, dA, dB, t: int, gelu: str = "tanh", workspace=None,
                              stream=None) -> None:
    """tpmlp_backward, but dA += X^T D and dB += Y^T G into the given fp32 buffers."""
    n, d = X.shape
    m = A.shape[1]
    assert G.shape == (n, d) and Z_save.shape == (n, m) and Y_save.shape == (n, m) and dX.shape == (n, d)
    assert dA.shape == (d, m) and dB.shape == (m, d) and dA.dtype == torch.float32 and dB.dtype == torch.float32
    _cuda(X, A, B, G, Z_save, Y_save, dX, dA, dB, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().tpmlp_backward_accumulate(_ptr(X), _ptr(A), _ptr(B), _ptr(G), _ptr(Z_save), _ptr(Y_save),
                                                    _ptr(dX), _ptr(dA), _ptr(dB), n, d, m, t, GELU[gelu], _dt(X),
                                                    _ptr(workspace), ws_bytes, _stream(stream)))


def tpmlp_backward_biased_workspace_size(n: int, d: int, m: int, dtype: torch.dtype) -> int:
    return load_library().tpmlp_backward_biased_workspace_size(n, d, m, DTYPE[dtype])


def tpmlp_backward_biased(X, A, B, G, Z_save, Y_save, dX, dA, dB, dbias1, dbias2, t: int, gelu: str = "tanh",
                          workspace=None, stream=None) -> None:
    n, d = X.shape
    m = A.shape[1]
    assert G.shape == (n, d) and Z_save.shape == (n, m) and Y_save.shape == (n, m) and dX.shape == (n, d)
    assert dA.shape == (d, m) and dB.shape == (m, d) and dbias1.shape == (m,) and dbias2.shape == (d,)
    for g_ in (dA, dB, dbias1, dbias2):
        assert g_.dtype == torch.float32
    _cuda(X, A, B, G, Z_save, Y_save, dX, dA, dB, dbias1, dbias2, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().tpmlp_backward_biased(_ptr(X), _ptr(A), _ptr(B), _ptr(G), _ptr(Z_save), _ptr(Y_save),
                                                _ptr(dX), _ptr(dA), _ptr(dB), _ptr(dbias1), _ptr(dbias2), n, d, m, t,
                                                GELU[gelu], _dt(X), _ptr(workspace), ws_bytes, _stream(stream)))


def tpmlp_backward_workspace_size(n: int, m: int, dtype: torch.dtype) -> int:
    return load_library().tpmlp_backward_workspace_size(n, m, DTYPE[dtype])


def tpmlp_backward(X, A, B, G, Z_save, Y_save, dX, dA, dB, t: int, gelu: str = "tanh", workspace=None,
                   stream=None) -> None:
    n, d = X.shape
    m = A.shape[1]
    assert G.shape == (n, d) and Z_save.shape == (n, m) and Y_save.shape == (n, m) and dX.shape == (n, d)
    assert dA.shape == (d, m) and dB.shape == (m, d) and dA.dtype == torch.float32 and dB.dtype == torch.float32
    _cuda(X, A, B, G, Z_save, Y_save, dX, dA, dB, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().tpmlp_backward(_ptr(X), _ptr(A), _ptr(B), _ptr(G), _ptr(Z_save), _ptr(Y_save), _ptr(dX),
                                         _ptr(dA), _ptr(dB), n, d, m, t, GELU[gelu], _dt(X), _ptr(workspace),
                                         ws_bytes, _stream(stream)))


def tpmlp_sp_block_workspace_size(b, s, h, m, t, dtype: torch.dtype, rs: str = "fused") -> int:
    return load_library().tpmlp_sp_block_workspace_size(b, s, h, m, t, DTYPE[dtype], RS_MODE[rs])


def tpmlp_sp_block(x_shards, gamma, beta, eps, A, B, p_drop, seed, out_shards, mask_bits, t: int, gelu="tanh",
                   rs="fused", workspace=None, stream=None, Z_save=None, Y_save=None) -> None:
    tt, b, sl, h = x_shards.shape
    assert tt == t and out_shards.shape == x_shards.shape
    m = A.shape[1]
    assert A.shape == (h, m) and B.shape == (m, h) and gamma.shape == (h,) and beta.shape == (h,)
    assert gamma.dtype == torch.float32 and beta.dtype == torch.float32
    if mask_bits is not None:
        assert mask_bits.dtype in (torch.int32, torch.uint32) and mask_bits.numel() >= (b * sl * t * h + 31) // 32
    for sv in (Z_save, Y_save):
        assert sv is None or sv.shape == (b * sl * t, m)
    _cuda(x_shards, gamma, beta, A, B, out_shards, mask_bits, workspace, Z_save, Y_save)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().tpmlp_sp_block(_ptr(x_shards), _ptr(gamma), _ptr(beta), eps, _ptr(A), _ptr(B), p_drop,
                                         seed, _ptr(out_shards), _ptr(mask_bits), _ptr(Z_save), _ptr(Y_save), b,
                                         sl * t, h, m, t, GELU[gelu], _dt(x_shards), RS_MODE[rs], _ptr(workspace),
                                         ws_bytes, _stream(stream)))


def tpmlp_sp_block_backward_workspace_size(b, s, h, m, t, dtype: torch.dtype) -> int:
    return load_library().tpmlp_sp_block_backward_workspace_size(b, s, h, m, t, DTYPE[dtype])


def tpmlp_sp_block_backward(x_shards, gamma, beta, eps, A, B, p_drop, seed, Z_save, Y_save, dout_shards, dx_shards,
                            dgamma, dbeta, dA, dB, t: int, gelu="tanh", workspace=None, stream=None,
                            mask_bits=None) -> None:
    tt, b, sl, h = x_shards.shape
    m = A.shape[1]
    assert tt == t and dout_shards.shape == x_shards.shape and dx_shards.shape == x_shards.shape
    assert Z_save.shape == (b * sl * t, m) and Y_save.shape == (b * sl * t, m)
    assert dgamma.shape == (h,) and dbeta.shape == (h,) and dA.shape == (h, m) and dB.shape == (m, h)
    assert mask_bits is None or mask_bits.numel() * 32 >= x_shards.numel()
    _cuda(x_shards, gamma, beta, A, B, Z_save, Y_save, dout_shards, dx_shards, dgamma, dbeta, dA, dB, workspace,
          mask_bits)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().tpmlp_sp_block_backward(
        _ptr(x_shards), _ptr(gamma), _ptr(beta), eps, _ptr(A), _ptr(B), p_drop, seed, _ptr(mask_bits), _ptr(Z_save),
        _ptr(Y_save),
        _ptr(dout_shards), _ptr(dx_shards), _ptr(dgamma), _ptr(dbeta), _ptr(dA), _ptr(dB), b, sl * t, h, m, t,
        GELU[gelu], _dt(x_shards), _ptr(workspace), ws_bytes, _stream(stream)))


def tpmlp_sp_layernorm(x, gamma, beta, eps, y, stream=None) -> None:
    h = x.shape[-1]
    rows = x.numel() // h
    assert y.shape == x.shape and gamma.shape == (h,) and beta.shape == (h,)
    _cuda(x, gamma, beta, y)
    _check(load_library().tpmlp_sp_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), eps, _ptr(y), rows, h, _dt(x),
                                             _stream(stream)))


def tpmlp_rmsnorm(x, gamma, eps, y, stream=None) -> None:
    h = x.shape[-1]
    rows = x.numel() // h
    assert y.shape == x.shape and gamma.shape == (h,) and gamma.dtype == torch.float32
    _cuda(x, gamma, y)
    _check(load_library().tpmlp_rmsnorm(_ptr(x), _ptr(gamma), eps, _ptr(y), rows, h, _dt(x), _stream(stream)))


def tpmlp_rmsnorm_backward_workspace_size(rows: int, h: int) -> int:
    return load_library().tpmlp_rmsnorm_backward_workspace_size(rows, h)


def tpmlp_rmsnorm_backward(x, gamma, eps, dy, dx, dgamma, workspace, stream=None) -> None:
    h = x.shape[-1]
    rows = x.numel() // h
    assert dy.shape == x.shape and dx.shape == x.shape and gamma.shape == (h,) and dgamma.shape == (h,)
    assert dgamma.dtype == torch.float32 and workspace.dtype == torch.uint8
    _cuda(x, gamma, dy, dx, dgamma, workspace)
    _check(load_library().tpmlp_rmsnorm_backward(_ptr(x), _ptr(gamma), eps, _ptr(dy), _ptr(dx), _ptr(dgamma), rows, h,
                                                 _dt(x), _ptr(workspace), workspace.numel(), _stream(stream)))


def tpmlp_sp_layernorm_backward_workspace_size(rows: int, h: int) -> int:
    return load_library().tpmlp_sp_layernorm_backward_workspace_size(rows, h)


def tpmlp_sp_layernorm_backward(x, gamma, eps, dy, dres, dx, dgamma, dbeta, workspace, stream=None) -> None:
    h = x.shape[-1]
    rows = x.numel() // h
    assert dy.shape == x.shape and dx.shape == x.shape and gamma.shape == (h,)
    assert dres is None or (dres.shape == x.shape and dres.dtype == x.dtype)
    assert dgamma.shape == (h,) and dbeta.shape == (h,) and dgamma.dtype == dbeta.dtype == torch.float32
    assert workspace.dtype == torch.uint8
    _cuda(x, gamma, dy, dres, dx, dgamma, dbeta, workspace)
    _check(load_library().tpmlp_sp_layernorm_backward(_ptr(x), _ptr(gamma), eps, _ptr(dy), _ptr(dres), _ptr(dx),
                                                      _ptr(dgamma), _ptr(dbeta), rows, h, _dt(x), _ptr(workspace),
                                                      workspace.numel(), _stream(stream)))


def tpmlp_sp_dropout_grad_gather(dout_shards, dtok, p_drop: float, seed: int, stream=None, mask_bits=None) -> None:
    t, b, sl, h = dout_shards.shape
    assert dtok.shape == (b, sl * t, h) and dtok.dtype == dout_shards.dtype
    assert mask_bits is None or mask_bits.numel() * 32 >= dout_shards.numel()
    _cuda(dout_shards, dtok, mask_bits)
    _check(load_library().tpmlp_sp_dropout_grad_gather(_ptr(dout_shards), _ptr(dtok), _ptr(mask_bits), float(p_drop),
                                                       seed, b, sl * t, h, t, _dt(dout_shards), _stream(stream)))


def tpmlp_sp_gather(x_shards, x_full, stream=None) -> None:
    t, b, sl, h = x_shards.shape
    assert x_full.shape == (b, sl * t, h) and x_full.dtype == x_shards.dtype
    _cuda(x_shards, x_full)
    _check(load_library().tpmlp_sp_gather(_ptr(x_shards), _ptr(x_full), b, sl * t, h, t, _dt(x_shards),
                                          _stream(stream)))


def tpmlp_sp_reduce_scatter(partials, out_shards, stream=None) -> None:
    t, b, sl, h = out_shards.shape
    assert partials.shape == (t, b * sl * t, h) and partials.dtype == torch.float32
    _cuda(partials, out_shards)
    _check(load_library().tpmlp_sp_reduce_scatter(_ptr(partials), _ptr(out_shards), b, sl * t, h, t,
                                                  _dt(out_shards), _stream(stream)))


def tpmlp_sp_dropout_residual(x_shards, y_shards, out_shards, mask_bits, p_drop, seed, stream=None) -> None:
    t, b, sl, h = x_shards.shape
    assert y_shards.shape == x_shards.shape and out_shards.shape == x_shards.shape
    _cuda(x_shards, y_shards, out_shards, mask_bits)
    _check(load_library().tpmlp_sp_dropout_residual(_ptr(x_shards), _ptr(y_shards), _ptr(out_shards),
                                                    _ptr(mask_bits), p_drop, seed, b, sl * t, h, t, _dt(x_shards),
                                                    _stream(stream)))


def tpmlp_check_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load_library().tpmlp_check_wait_timeout(limit_ns, _stream(stream)))


def tpmlp_device_status(stream=None, clear: bool = True) -> None:
    _check(load_library().tpmlp_device_status(_stream(stream), 1 if clear else 0))


def tpmlp_set_gemm_variant(pair_kernel: int = 1, pair_pacing: int = 1, pair_group: int = 0) -> None:
    _check(load_library().tpmlp_set_gemm_variant(pair_kernel, pair_pacing, pair_group))


# ----------------------------------------------------------------------- conveniences

def forward(X, A, B, t: int, gelu: str = "tanh", save_z: bool = True, stream=None, bias1=None, bias2=None):
    """Allocate O, Z, Y with torch and run tpmlp_forward (tpmlp_forward_biased when biases are
    given). Returns (O, Z, Y)."""
    n, m = X.shape[0], A.shape[1]
    O = torch.empty_like(X)
    Z = torch.empty((n, m), dtype=X.dtype, device=X.device) if save_z else None
    Y = torch.empty((n, m), dtype=X.dtype, device=X.device)
    if bias1 is not None or bias2 is not None:
        tpmlp_forward_biased(X, A, B, bias1, bias2, O, Z, Y, t, gelu, stream)
    else:
        tpmlp_forward(X, A, B, O, Z, Y, t, gelu, stream)
    return O, Z, Y


def backward(X, A, B, G, Z, Y, t: int, gelu: str = "tanh", stream=None, with_bias: bool = False):
    """Allocate gradients and the workspace with torch and run tpmlp_backward (or, with_bias,
    tpmlp_backward_biased). Returns (dX, dA, dB) or (dX, dA, dB, dbias1, dbias2)."""
    n, d = X.shape
    m = A.shape[1]
    dX = torch.empty_like(X)
    dA = torch.empty((d, m), dtype=torch.float32, device=X.device)
    dB = torch.empty((m, d), dtype=torch.float32, device=X.device)
    if with_bias:
        db1 = torch.empty(m, dtype=torch.float32, device=X.device)
        db2 = torch.empty(d, dtype=torch.float32, device=X.device)
        ws = torch.empty(max(1, tpmlp_backward_biased_workspace_size(n, d, m, X.dtype)), dtype=torch.uint8,
                         device=X.device)
        tpmlp_backward_biased(X, A, B, G, Z, Y, dX, dA, dB, db1, db2, t, gelu, ws, stream)
        return dX, dA, dB, db1, db2
    ws = torch.empty(max(1, tpmlp_backward_workspace_size(n, m, X.dtype)), dtype=torch.uint8, device=X.device)
    tpmlp_backward(X, A, B, G, Z, Y, dX, dA, dB, t, gelu, ws, stream)
    return dX, dA, dB


def sp_block(x_shards, gamma, beta, eps, A, B, p_drop, seed, t: int, gelu="tanh", rs="fused", with_mask=True,
             save_for_backward=False, stream=None):
    """Allocate outputs and workspace and run tpmlp_sp_block.
    Returns (out_shards, mask_bits or None, (Z, Y) or None)."""
    tt, b, sl, h = x_shards.shape
    n, m = b * sl * t, A.shape[1]
    out = torch.empty_like(x_shards)
    mask = torch.empty(((n * h + 31) // 32,), dtype=torch.int32, device=x_shards.device) if with_mask else None
    saves = None
    if save_for_backward:
        saves = tuple(torch.empty((n, m), dtype=x_shards.dtype, device=x_shards.device) for _ in range(2))
    ws = torch.empty(max(1, tpmlp_sp_block_workspace_size(b, sl * t, h, m, t, x_shards.dtype, rs)),
                     dtype=torch.uint8, device=x_shards.device)
    tpmlp_sp_block(x_shards, gamma, beta, eps, A, B, p_drop, seed, out, mask, t, gelu, rs, ws, stream,
                   *(saves if saves else (None, None)))
    return out, mask, saves


def sp_block_backward(x_shards, gamma, beta, eps, A, B, p_drop, seed, Z, Y, dout_shards, t: int, gelu="tanh",
                      stream=None, mask_bits=None):
    """Allocate gradients and workspace and run tpmlp_sp_block_backward.
    Returns (dx_shards, dgamma, dbeta, dA, dB)."""
    tt, b, sl, h = x_shards.shape
    m = A.shape[1]
    dev = x_shards.device
    dx = torch.empty_like(x_shards)
    dgamma = torch.empty(h, dtype=torch.float32, device=dev)
    dbeta = torch.empty(h, dtype=torch.float32, device=dev)
    dA = torch.empty((h, m), dtype=torch.float32, device=dev)
    dB = torch.empty((m, h), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, tpmlp_sp_block_backward_workspace_size(b, sl * t, h, m, t, x_shards.dtype)),
                     dtype=torch.uint8, device=dev)
    tpmlp_sp_block_backward(x_shards, gamma, beta, eps, A, B, p_drop, seed, Z, Y, dout_shards, dx, dgamma, dbeta, dA,
                            dB, t, gelu, ws, stream, mask_bits)
    return dx, dgamma, dbeta, dA, dB


# ----------------------------------------------------------------------- attention block

def rmsnorm(x, gamma, eps: float = 1e-5, stream=None):
    """Allocates y and runs tpmlp_rmsnorm."""
    y = torch.empty_like(x)
    tpmlp_rmsnorm(x, gamma, eps, y, stream)
    return y


def rmsnorm_backward(x, gamma, dy, eps: float = 1e-5, stream=None):
    """Allocates dx, dgamma and the workspace and runs tpmlp_rmsnorm_backward; returns (dx, dgamma)."""
    h = x.shape[-1]
    dx = torch.empty_like(x)
    dgamma = torch.empty(h, dtype=torch.float32, device=x.device)
    ws = torch.empty(tpmlp_rmsnorm_backward_workspace_size(x.numel() // h, h), dtype=torch.uint8, device=x.device)
    tpmlp_rmsnorm_backward(x, gamma, eps, dy, dx, dgamma, ws, stream)
    return dx, dgamma


def attention_forward(X, Wqkv, Wo, heads: int, t: int, stream=None):
    """X [b, s, h] bf16; allocates Y, the saves and the workspace and runs tpmlp_attention_forward.
    Returns (Y [b, s, h], (QKV, P, O))."""
    b, s, h = X.shape
    _cuda(X, Wqkv, Wo)
    assert Wqkv.shape == (h, 3 * h) and Wo.shape == (h, h)
    dev = X.device
    Y = torch.empty_like(X)
    QKV = torch.empty((b * s, 3 * h), dtype=X.dtype, device=dev)
    P = torch.empty((b, heads, s, s), dtype=X.dtype, device=dev)
    O = torch.empty((b * s, h), dtype=X.dtype, device=dev)
    lib = load_library()
    ws = torch.empty(max(1, lib.tpmlp_attention_forward_workspace_size(b, s, h, heads, _dt(X))), dtype=torch.uint8,
                     device=dev)
    _check(lib.tpmlp_attention_forward(_ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(Y), _ptr(QKV), _ptr(P), _ptr(O), b, s, h,
                                       heads, t, _dt(X), _ptr(ws), ws.numel(), _stream(stream)))
    return Y, (QKV, P, O)


def attention_backward(X, Wqkv, Wo, G, saves, heads: int, t: int, stream=None):
    """Runs tpmlp_attention_backward; returns (dX [b, s, h], dWqkv [h, 3h] fp32, dWo [h, h] fp32)."""
    b, s, h = X.shape
    QKV, P, O = saves
    _cuda(X, Wqkv, Wo, G, QKV, P, O)
    dev = X.device
    dX = torch.empty_like(X)
    dWqkv = torch.empty((h, 3 * h), dtype=torch.float32, device=dev)
    dWo = torch.empty((h, h), dtype=torch.float32, device=dev)
    lib = load_library()
    ws = torch.empty(max(1, lib.tpmlp_attention_backward_workspace_size(b, s, h, heads, _dt(X))), dtype=torch.uint8,
                     device=dev)
    _check(lib.tpmlp_attention_backward(_ptr(X), _ptr(Wqkv), _ptr(Wo), _ptr(G), _ptr(QKV), _ptr(P), _ptr(O), _ptr(dX),
                                        _ptr(dWqkv), _ptr(dWo), b, s, h, heads, t, _dt(X), _ptr(ws), ws.numel(),
                                        _stream(stream)))
    return dX, dWqkv, dWo
