"""Helpers shared by the GPU parity tests (host <-> device copies and the
element-wise tolerance check). No method arithmetic lives here."""
import numpy as np
import torch

import oracle as oracle_mod


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> CUDA tensor, bit for bit (uint32 travels as int32)."""
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f16(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.detach().cpu().numpy().astype(np.float16)


def assert_within(y_gpu, y_ref, S, what="", bound=None):
    """|y - y_ref| <= 2^-10 |y_ref| + 1e-4 S element-wise (or an explicit bound).
    Returns the worst error/bound ratio."""
    y = np.asarray(y_gpu, dtype=np.float64)
    tol = oracle_mod.tolerance(y_ref, S) if bound is None else bound
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at "
                             f"{i}: gpu={y[i]!r} ref={y_ref[i]!r} tol={tol[i]!r}")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / tol, 0.0)
    return float(ratio.max()) if ratio.size else 0.0
