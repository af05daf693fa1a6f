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


def update_then_clip_band(w_exact, tol, row_factor, rn, gamma_rel=1e-6):
    """Band of the stored weight after the Muon update (stored, i.e. rounded,
    in the weight dtype) and then the clip (multiply by row_factor > 0,
    rounded again).  w_exact: exact updated weights; tol: update tolerance;
    row_factor: per-row factor gamma^e (1 for untouched rows); gamma_rel:
    relative uncertainty of the device's gamma (its S_max is an fp32 sum)."""
    lo, hi = rn(w_exact - tol), rn(w_exact + tol)
    f = np.asarray(row_factor, np.float64).reshape(-1, 1)
    lo, hi = lo * f, hi * f
    clipped = f != 1.0
    lo = np.where(clipped, lo - gamma_rel * np.abs(lo), lo)
    hi = np.where(clipped, hi + gamma_rel * np.abs(hi), hi)
    return rn(lo), rn(hi)


def check_argmax(arg_gpu, q, k, ks, heads, ref_s, ref_arg, scale=None):
    """The device argmax of each head in `heads` (flat index (b S + i) S + j)
    must be the oracle's pair, or, where another pair ties within the fp32
    accumulation error, a causal pair whose exact logit is within 2e-6 of the
    maximum.  ref_s / ref_arg: the oracle's S_max and (b, i, j) for those
    heads, in the same order."""
    import math
    S = q.shape[1]
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale
    got = arg_gpu.cpu().numpy()
    exact = 0
    for n, h in enumerate(heads):
        b, i, j = (int(x) for x in ref_arg[n])
        flat = (b * S + i) * S + j
        if int(got[h]) == flat:
            exact += 1
            continue
        gb, rem = divmod(int(got[h]), S * S)
        gi, gj = divmod(rem, S)
        assert gj <= gi, (h, "non-causal pair", gi, gj)
        kv = f64(k[gb, gj, h])
        if ks is not None:
            kv = np.concatenate([kv, f64(ks[gb, gj])])
        other = float(f64(q[gb, gi, h]) @ kv) * scale
        assert abs(other - ref_s[n]) <= 2e-6 * abs(ref_s[n]) + 1e-6, (h, int(got[h]), flat)
    return exact
