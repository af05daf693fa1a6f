"""Float emulation of the split Newton-Schulz plan's roundings (test
infrastructure, no GPU): the evidence behind the library's product plan.

Newton-Schulz as [K2-internals] "Algorithm 1" orthogonalises with the quintic
X <- a X + (b A + c A^2) X, A = X X^T.  The library stores every operand as a
16-bit (hi, lo) pair (bf16 in the first iteration, fp16 after it), takes one,
two or three products per k-step (hi*hi; hi*hi + hi*lo of the right operand;
hi*hi + hi*lo + lo*hi) and folds a I into the polynomial of three-term
iterations.  This module restates those roundings with torch fp32 matmuls
(the tensor cores accumulate in fp32) so that a plan's error against exact
float64 arithmetic can be measured on the CPU.
"""
import torch

A_NS, B_NS, C_NS = 3.4445, -4.7750, 2.0315


def _r(x, fmt):
    return x.to(torch.bfloat16 if fmt == "b" else torch.float16).to(torch.float32)


def _split(x, fmt):
    hi = _r(x, fmt)
    return hi, _r(x - hi, fmt)


def _pair(x, fmt):
    hi, lo = _split(x, fmt)
    return hi + lo


def _mm(x, y, products, fmt):
    """x @ y with `products` per k-step: 1 (hi*hi), 2 (hi*hi + hi*lo of y,
    the library's), "2x" (hi*hi + lo of x * hi, the other choice of two),
    3 (hi*hi + hi*lo + lo*hi)."""
    if products == 1:
        return _r(x, fmt) @ _r(y, fmt)
    xh, xl = _split(x, fmt)
    yh, yl = _split(y, fmt)
    if products == 2:
        return xh @ yh + xh @ yl
    if products == "2x":
        return xh @ yh + xl @ yh
    return xh @ yh + (xh @ yl + xl @ yh)


def emulate(M, fast=3, last_update=2, trailing_updates=2, fold_fast=False, steps=5):
    """The library's plan on M (float64, rows <= cols): `fast` leading
    one-product iterations (the update adds a X from X's pair, or with
    fold_fast takes B + a I rounded to one plane), then iterations whose Gram
    takes one product and whose polynomial (a I folded in) takes three, the
    update `trailing_updates` products except the last one's `last_update`."""
    X = _pair((M / torch.linalg.norm(M)).float(), "b")
    eye = torch.eye(M.shape[0])
    for it in range(steps):
        fmt = "b" if it == 0 else "h"
        A = _pair(_mm(X, X.T, 1, fmt), fmt)
        if it < fast:
            if fold_fast:
                Bp = _r(A_NS * eye + B_NS * A + C_NS * _mm(A, A, 1, fmt), fmt)
                X = _pair(_mm(Bp, X, 1, fmt), "h")
            else:
                Bp = _r(B_NS * A + C_NS * _mm(A, A, 1, fmt), fmt)
                X = _pair(A_NS * X + _mm(Bp, X, 1, fmt), "h")
        else:
            Bp = _pair(A_NS * eye + B_NS * A + C_NS * _mm(A, A, 3, "h"), "h")
            prods = last_update if it == steps - 1 else trailing_updates
            X = _pair(_mm(Bp, X, prods, "h"), "h")
    return X


def exact(M, steps=5):
    X = M / torch.linalg.norm(M)
    for _ in range(steps):
        A = X @ X.T
        X = A_NS * X + (B_NS * A + C_NS * (A @ A)) @ X
    return X


def max_error(O, M):
    """max |O - O_exact| / RMS(O_exact)."""
    O64 = exact(M)
    return float((O.double() - O64).abs().max()) / float(torch.sqrt(torch.mean(O64 ** 2)))


def gaussian(m, n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(m, n, generator=g, dtype=torch.float64)


def adversarial(m, n, k, floor, seed):
    """k unit singular values over a rest at `floor`."""
    g = torch.Generator().manual_seed(seed)
    U, _ = torch.linalg.qr(torch.randn(m, m, generator=g, dtype=torch.float64))
    V, _ = torch.linalg.qr(torch.randn(n, m, generator=g, dtype=torch.float64))
    s = torch.full((m,), floor, dtype=torch.float64)
    s[:k] = 1.0
    return (U * s) @ V.T
