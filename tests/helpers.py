"""Shared test utilities: moving seeded inputs to the GPU and measuring parity."""
import numpy as np
import torch

# Tolerances on max|gpu - ref| / max|ref| per output tensor: bf16 inputs with fp32
# accumulation, and the fp32 path.
TOL_BF16 = 2e-2
TOL_F32 = 1e-5

TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def dev(a: np.ndarray, dtype: str | torch.dtype, device="cuda") -> torch.Tensor:
    """Upload float32 arrays whose values are already exact in `dtype`."""
    td = TORCH_DTYPE.get(dtype, dtype)
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
    out = t.to(td)
    return out.contiguous()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


def assert_close(name, got, ref, tol, report=None):
    e = rel_err(got, ref)
    if report is not None:
        report[name] = e
    assert np.all(np.isfinite(np.asarray(got, np.float64))), f"{name}: non-finite values"
    assert e <= tol, f"{name}: max|err|/max|ref| = {e:.3e} > {tol:.1e}"
    return e
