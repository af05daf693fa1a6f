"""Shared helpers of the GPU parity tests (comparison rules only)."""
import numpy as np
import torch

import oracle as O


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a float32 / bfloat16 tensor."""
    return t.detach().float().cpu().double().numpy()


def rounder(dtype):
    return O.round_to_bf16 if dtype == torch.bfloat16 else O.round_to_f32


def assert_rounded_within(got: torch.Tensor, exact: np.ndarray, tol, what=""):
    """got (stored in its dtype) must be a rounding of some value within `tol`
    of `exact`: rounding is monotone, so got lies in [rn(exact - tol),
    rn(exact + tol)].  `tol` may be a scalar or an array."""
    rn = rounder(got.dtype)
    g = f64(got)
    lo, hi = rn(exact - tol), rn(exact + tol)
    bad = ~((g >= lo) & (g <= hi))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        err = np.abs(g - exact)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {g.size} values outside the tolerance band; "
            f"max |err| = {err.max():.3e} vs tol {np.max(tol):.3e}; first at {idx.tolist()}")


def rms(x: np.ndarray) -> float:
    return float(np.sqrt(np.mean(np.square(x))))


def cuda(t):
    return t.to("cuda")


def padded(rows, cols, dtype, pad_to=8, fill=float("nan")):
    """A [rows, cols] view with a row pitch rounded up to `pad_to` columns
    (exercises ld > cols); the padding holds `fill`."""
    ld = (cols + pad_to - 1) // pad_to * pad_to
    base = torch.full((rows, ld), fill, dtype=dtype, device="cuda")
    return base[:, :cols]
