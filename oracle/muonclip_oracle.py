"""Plain fp64 CPU oracle for the MuonClip optimizer step (Muon + per-head QK-Clip).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may call it.  It shares no code with the CUDA library (no kernels, headers,
helpers or constants); both sides only consume the same seeded inputs.

Every function restates one step of the method in float64 with numpy, in the
order and notation of the pages it cites.  Library primitives used as steps:
``numpy.matmul`` (a dense product) and ``numpy.linalg.norm`` (Frobenius norm).
Nothing is blocked, fused or reordered beyond what the cited definition states.

Sources (web pages on Kimi K2 / MuonClip; cited by title and section):
  [K2-notes]     "Kimi K2: Open Agentic Intelligence" (paper-notes-site),
                 section 3.2 "MuonClip" and its pseudocode block.
  [K2-internals] "Kimi K2 内部机制" (LLM-101-CN deep dive): "核心数学"
                 (S_max, gamma), "MLA 的特殊处理" (scaling table),
                 "Algorithm 1 MuonClip Optimizer".
  [K2-explained] "Kimi K2, explained" (vibeengines): "Pretraining with
                 MuonClip" and its symbol list (Newton-Schulz, sqrt(max)*0.2,
                 tau, gamma_h).
  [K2-zhihu]     zhihu Q&A page on K2: the MuonClip formula written with
                 msign, and the "Muon's Infra Scalability" answer.

Readings of points the pages leave open (each is a parameter, default shown):
  * Newton-Schulz polynomial p(x) = a x + b x^3 + c x^5, applied to matrices as
    X <- a X + (b A + c A^2) X with A = X X^T.  The pages name the iteration
    ("an odd matrix polynomial that pushes singular values toward 1") but give
    no coefficients; default (a,b,c) = (3.4445, -4.7750, 2.0315), the quintic
    of the published Muon method the pages cite; 5 steps.
  * Normalisation X0 = M / (||M||_F + eps), eps = 1e-7.
  * Orientation: the iteration runs on whichever of M, M^T has rows <= cols.
    For an odd matrix polynomial p(M^T) = p(M)^T exactly, so this choice only
    changes cost, never the result.
  * Softmax scale 1/sqrt(d), d = the q.k length (MLA: d_nope + d_rope).
  * Causal attention: the max runs over key positions j <= i.
  * S_max^h == tau and S_max^h <= 0 do not clip; NaN S does not clip.
  * Argmax ties go to the smallest (b, i, j) in lexicographic order.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

# Default hyper-parameters.  mu=0.95 is the pseudocode default in [K2-notes]
# section 3.2; lr=2e-4, weight_decay=0.1 and tau=100 are the K2 training recipe
# ([K2-notes] section 3.5, [K2-explained] "Pretraining with MuonClip");
# rms_scale=0.2 is Algorithm 1's "Match Adam RMS" factor ([K2-internals]).
DEFAULT_NS_COEFFS = (3.4445, -4.7750, 2.0315)


@dataclass
class Hparams:
    mu: float = 0.95
    lr: float = 2e-4
    weight_decay: float = 0.1
    rms_scale: float = 0.2
    ns_steps: int = 5
    ns_coeffs: tuple = DEFAULT_NS_COEFFS
    ns_eps: float = 1e-7
    tau: float = 100.0
    alpha: float = 0.5
    scale_mode: str = "rms"        # "rms": 0.2 sqrt(max(n, m)); "spectral": sqrt(max(1, out/in))


# ---------------------------------------------------------------------------
# Muon
# ---------------------------------------------------------------------------

def momentum(M_prev: np.ndarray, G: np.ndarray, mu: float) -> np.ndarray:
    """M_t = mu * M_{t-1} + G_t, with M_0 = 0 (plain heavy-ball momentum).

    [K2-internals] Algorithm 1, momentum step; [K2-zhihu] MuonClip formula
    (first row); [K2-notes] section 3.2 pseudocode (M.mul_(momentum).add_(G)).
    """
    return mu * np.asarray(M_prev, np.float64) + np.asarray(G, np.float64)


def ns_iterate(X: np.ndarray, steps: int, coeffs=DEFAULT_NS_COEFFS) -> np.ndarray:
    """Apply the odd matrix polynomial `steps` times to an already scaled X.

    Each step: A = X X^T;  B = b A + c A A;  X <- a X + B X.
    [K2-explained] symbol list: Newton-Schulz is "a few iterations of an odd
    matrix polynomial" pushing singular values toward 1.
    """
    a, b, c = coeffs
    X = np.asarray(X, np.float64)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X


def newton_schulz(M: np.ndarray, steps: int = 5, coeffs=DEFAULT_NS_COEFFS,
                  eps: float = 1e-7) -> np.ndarray:
    """NewtonSchulz(M) ~ msign(M) = U V^T for M = U S V^T.

    [K2-explained] symbol list ("approximating the orthogonal factor U V^T");
    [K2-zhihu] MuonClip formula (msign(M_t)).  Frobenius normalisation first,
    then `steps` polynomial iterations on the orientation with rows <= cols.
    """
    M = np.asarray(M, np.float64)
    transpose = M.shape[0] > M.shape[1]
    X = M.T if transpose else M
    X = X / (np.linalg.norm(X) + eps)
    X = ns_iterate(X, steps, coeffs)
    return X.T if transpose else X


def update_scale(rows: int, cols: int, hp: Hparams) -> float:
    """Factor on NewtonSchulz(M) for a weight stored [out=rows, in=cols].

    "rms": sqrt(max(n, m)) * 0.2, matching AdamW's update RMS ([K2-internals]
    Algorithm 1, "Match Adam RMS"; [K2-zhihu] MuonClip formula).
    "spectral": sqrt(max(1, d_out / d_in)), the MuP-style scale the zhihu
    answer's section 3.2 describes for later Muon versions."""
    if hp.scale_mode == "spectral":
        return math.sqrt(max(1.0, rows / cols))
    return math.sqrt(max(rows, cols)) * hp.rms_scale


def muon_direction(M: np.ndarray, hp: Hparams) -> np.ndarray:
    """O_t = NewtonSchulz(M_t) * update_scale (default sqrt(max(n, m)) * 0.2).

    [K2-internals] Algorithm 1, orthogonalisation step ("Match Adam RMS");
    [K2-zhihu] MuonClip formula (second row).
    """
    r, c = M.shape
    return newton_schulz(M, hp.ns_steps, hp.ns_coeffs, hp.ns_eps) * update_scale(r, c, hp)


def muon_apply(W_prev: np.ndarray, O: np.ndarray, lr: float, weight_decay: float) -> np.ndarray:
    """W_t = W_{t-1} - lr * (O_t + weight_decay * W_{t-1}) (decoupled decay).

    [K2-internals] Algorithm 1, weight update step; [K2-zhihu] MuonClip formula
    (third row); [K2-notes] section 3.2 pseudocode (W.add_(O + wd*W, -lr)).
    """
    W_prev = np.asarray(W_prev, np.float64)
    return W_prev - lr * (np.asarray(O, np.float64) + weight_decay * W_prev)


def muon_step(W: np.ndarray, G: np.ndarray, M_prev: np.ndarray, hp: Hparams):
    """One Muon step for one matrix; returns (W_t exact in fp64, M_t, O_t)."""
    M = momentum(M_prev, G, hp.mu)
    O = muon_direction(M, hp)
    return muon_apply(W, O, hp.lr, hp.weight_decay), M, O


# ---------------------------------------------------------------------------
# QK-Clip
# ---------------------------------------------------------------------------

def head_keys(K: np.ndarray, K_shared, b: int, h: int) -> np.ndarray:
    """Key vectors k_j of head h in batch b: [k^C_j (head h) || k^R_j (shared)].

    MHA: K_shared is None and k_j = K[b, j, h, :].
    MLA: the head-specific part is concatenated with the rotary key shared by
    every head ([K2-internals] "MLA 的特殊处理").
    """
    k = np.asarray(K[b, :, h, :], np.float64)
    if K_shared is not None:
        k = np.concatenate([k, np.asarray(K_shared[b], np.float64)], axis=1)
    return k


def max_logit(Q: np.ndarray, K: np.ndarray, K_shared=None, causal: bool = True,
              scale=None, row_chunk: int = 2048):
    """Per-head max attention logit over the batch.

    S_max^h = (1/sqrt(d)) * max_{X in B} max_{i,j} Q_i^h . K_j^h
    ([K2-internals] "核心数学"; the notes page writes 1/d, a garbled 1/sqrt(d)).
    The max over j is restricted to j <= i when `causal`.

    Q: [B, S, H, dq];  K: [B, S, H, dk];  K_shared: [B, S, dr] or None,
    dq = dk + dr.  Returns (S [H] float64, argmax [H, 3] int64 of (b, i, j)).
    The max over i is taken `row_chunk` query rows at a time (a nested max,
    equal to the flat one) so that long sequences fit in memory.
    """
    Bsz, S, H, dq = Q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(dq)
    smax = np.full(H, -np.inf)
    arg = np.zeros((H, 3), np.int64)
    jj = np.arange(S)
    for h in range(H):
        best, best_at = -np.inf, (0, 0, 0)
        for b in range(Bsz):
            k = head_keys(K, K_shared, b, h)
            q_all = np.asarray(Q[b, :, h, :], np.float64)
            for i0 in range(0, S, row_chunk):
                q = q_all[i0:i0 + row_chunk]
                L = q @ k.T
                if causal:
                    ii = np.arange(i0, i0 + q.shape[0])
                    L = np.where(jj[None, :] <= ii[:, None], L, -np.inf)
                flat = int(np.argmax(L))          # first occurrence: smallest (i, j)
                v = L.flat[flat]
                if v > best:                      # strict: earlier (b, i) wins ties
                    best = v
                    best_at = (b, i0 + flat // S, flat % S)
        smax[h] = best * scale
        arg[h] = best_at
    return smax, arg


def attention_forward(Q: np.ndarray, K: np.ndarray, V: np.ndarray, K_shared=None,
                      causal: bool = True, scale=None, row_chunk: int = 1024):
    """Attention output with the per-head max logit taken along the way.

    O^h = softmax(scale * Q^h K^h^T) V^h with scale = 1/sqrt(d)
    ([K2-internals] "核心数学"), the softmax over j <= i when `causal`; the
    max logit S_max^h is the max_logit definition above, i.e. the largest
    entry of the same scaled logit matrix before the softmax.

    Q: [B, S, H, dq]; K: [B, S, H, dk]; K_shared: [B, S, dr] or None (dq = dk + dr);
    V: [B, S, H, dv].  Returns (O [B, S, H, dv], lse [B, H, S], smax [H]) in
    float64, lse being the natural log of each row's softmax denominator.
    """
    Bsz, S, H, dq = Q.shape
    dv = V.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(dq)
    O = np.zeros((Bsz, S, H, dv))
    lse = np.zeros((Bsz, H, S))
    smax = np.full(H, -np.inf)
    jj = np.arange(S)
    for b in range(Bsz):
        for h in range(H):
            k = head_keys(K, K_shared, b, h)
            v = np.asarray(V[b, :, h, :], np.float64)
            q_all = np.asarray(Q[b, :, h, :], np.float64)
            for i0 in range(0, S, row_chunk):
                q = q_all[i0:i0 + row_chunk]
                L = scale * (q @ k.T)
                if causal:
                    ii = np.arange(i0, i0 + q.shape[0])
                    L = np.where(jj[None, :] <= ii[:, None], L, -np.inf)
                smax[h] = max(smax[h], float(np.max(L)))
                m = np.max(L, axis=1, keepdims=True)
                E = np.exp(L - m)
                den = np.sum(E, axis=1, keepdims=True)
                O[b, i0:i0 + q.shape[0], h, :] = (E / den) @ v
                lse[b, h, i0:i0 + q.shape[0]] = (m + np.log(den))[:, 0]
    return O, lse, smax


def clip_factors(smax: np.ndarray, tau: float):
    """gamma_h = min(1, tau / S_max^h); a head clips only when S_max^h > tau.

    [K2-internals] "核心数学" (per-head gamma) and Algorithm 1 QK-Clip branch;
    [K2-notes] section 3.2 pseudocode ("if s_max <= tau: continue").
    """
    smax = np.asarray(smax, np.float64)
    mask = smax > tau                     # NaN compares False: no clip
    gamma = np.ones_like(smax)
    gamma[mask] = tau / smax[mask]
    return gamma, mask


@dataclass
class ClipSegment:
    """Rows of one weight matrix that belong to every head, and their exponent.

    Head h owns rows [offset + h*stride, offset + h*stride + rows) of W (weights
    stored [out, in], so a head's query/key features are a row block).  The
    head's rows are multiplied by gamma_h ** exponent.
      MHA ([K2-internals] "核心数学"):  W_q -> alpha, W_k -> 1 - alpha.
      MLA ([K2-internals] "MLA 的特殊处理"): q^C -> 1/2, k^C -> 1/2, q^R -> 1;
      the shared rotary key k^R has no segment (left untouched).
    """
    name: str
    offset: int
    stride: int
    rows: int
    exponent: float


def qk_clip(weights: dict, segments, smax: np.ndarray, tau: float):
    """Rescale the offending heads' weight rows; returns (new weights, gamma, mask).

    [K2-internals] Algorithm 1 QK-Clip branch (W_qc, W_kc by sqrt(gamma),
    W_qr by gamma); [K2-zhihu] MuonClip formula (QK-Clip rows).
    """
    gamma, mask = clip_factors(smax, tau)
    out = {k: np.array(v, np.float64) for k, v in weights.items()}
    for seg in segments:
        W = out[seg.name]
        for h in np.nonzero(mask)[0]:
            r0 = seg.offset + h * seg.stride
            W[r0:r0 + seg.rows] *= gamma[h] ** seg.exponent
    return out, gamma, mask


def total_clip_factor(smax: np.ndarray, tau: float) -> float:
    """The naive all-head variant: one gamma = min(1, tau / max_h S_max^h).

    [K2-internals] "核心数学" (朴素实现); [K2-zhihu] (Total Clip before Per-Head).
    A NaN among the S_max values means no clip.
    """
    s = float(np.max(smax))
    return tau / s if s > tau else 1.0


def qk_clip_total(weights: dict, segments, smax: np.ndarray, tau: float):
    """Total QK-Clip: every head's segment rows scale by gamma^exponent with the
    one gamma of total_clip_factor.  Returns (new weights, gamma)."""
    g = total_clip_factor(smax, tau)
    out = {k: np.array(v, np.float64) for k, v in weights.items()}
    if g < 1.0:
        H = len(smax)
        for seg in segments:
            W = out[seg.name]
            for h in range(H):
                r0 = seg.offset + h * seg.stride
                W[r0:r0 + seg.rows] *= g ** seg.exponent
    return out, g


def mha_segments(H: int, d: int, alpha: float = 0.5):
    return [ClipSegment("Wq", 0, d, d, alpha), ClipSegment("Wk", 0, d, d, 1.0 - alpha)]


def mla_segments(H: int, d_nope: int = 128, d_rope: int = 64, d_v: int = 128):
    """W_UQ rows per head = [q^C (d_nope) || q^R (d_rope)];
    W_UKV rows per head = [k^C (d_nope) || v (d_v)]; W_KR (shared) untouched."""
    dq = d_nope + d_rope
    dkv = d_nope + d_v
    return [ClipSegment("W_UQ", 0, dq, d_nope, 0.5),
            ClipSegment("W_UQ", d_nope, dq, d_rope, 1.0),
            ClipSegment("W_UKV", 0, dkv, d_nope, 0.5)]


def muonclip_step(weights: dict, grads: dict, moms: dict, hp: Hparams,
                  layers=()):
    """One MuonClip step: Muon on every matrix, then per-head QK-Clip.

    [K2-internals] Algorithm 1: (1) for each weight, momentum -> Newton-Schulz
    -> RMS match -> decoupled decay; (2) for every head of every attention layer,
    with S_max^h from this step's forward, clip if S_max^h > tau.
    `layers` is a sequence of (smax [H], segments).  Returns (W, M, gammas).
    """
    W_new, M_new = {}, {}
    for name in weights:
        W_new[name], M_new[name], _ = muon_step(weights[name], grads[name],
                                                 moms[name], hp)
    gammas = []
    for smax, segs in layers:
        W_new, gamma, _ = qk_clip(W_new, segs, smax, hp.tau)
        gammas.append(gamma)
    return W_new, M_new, gammas


# ---------------------------------------------------------------------------
# Forward-side helpers the tests use to produce Q/K from weights (the
# projections Q^h = X W_q^h, K^h = X W_k^h of [K2-internals] "核心数学").
# ---------------------------------------------------------------------------

def project_mha(X: np.ndarray, Wq: np.ndarray, Wk: np.ndarray, H: int):
    """Q = X Wq^T, K = X Wk^T split into H heads: X [B,S,D] -> [B,S,H,d]."""
    X = np.asarray(X, np.float64)
    Bsz, S, _ = X.shape
    Q = X @ np.asarray(Wq, np.float64).T
    K = X @ np.asarray(Wk, np.float64).T
    return Q.reshape(Bsz, S, H, -1), K.reshape(Bsz, S, H, -1)


def rms_norm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Weightless RMSNorm over the last axis (the MLA latent norms)."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope(x: np.ndarray, theta: float = 10000.0) -> np.ndarray:
    """Rotary embedding on interleaved pairs (x[2k], x[2k+1]) at positions
    0..S-1 along axis 1; x is [B, S, ..., d] with d even."""
    x = np.asarray(x, np.float64)
    S, d = x.shape[1], x.shape[-1]
    inv = theta ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    ang = np.arange(S, dtype=np.float64)[:, None] * inv[None, :]
    shape = [1, S] + [1] * (x.ndim - 3) + [d // 2]
    cos, sin = np.cos(ang).reshape(shape), np.sin(ang).reshape(shape)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * cos - x1 * sin
    out[..., 1::2] = x0 * sin + x1 * cos
    return out


def project_mla(X, W_DQ, W_UQ, W_DKV, W_UKV, W_KR, H: int, d_nope: int = 128,
                d_rope: int = 64, d_v: int = 128):
    """MLA query/key features: returns (Q [B,S,H,d_nope+d_rope] = [q^C||q^R],
    K^C [B,S,H,d_nope], K^R [B,S,d_rope] shared by all heads)."""
    X = np.asarray(X, np.float64)
    Bsz, S, _ = X.shape
    cq = rms_norm(X @ np.asarray(W_DQ, np.float64).T)
    q = (cq @ np.asarray(W_UQ, np.float64).T).reshape(Bsz, S, H, d_nope + d_rope)
    q = np.concatenate([q[..., :d_nope], rope(q[..., d_nope:])], axis=-1)
    ckv = rms_norm(X @ np.asarray(W_DKV, np.float64).T)
    kv = (ckv @ np.asarray(W_UKV, np.float64).T).reshape(Bsz, S, H, d_nope + d_v)
    kc = kv[..., :d_nope]
    kr = rope(X @ np.asarray(W_KR, np.float64).T)
    return q, kc, kr


# ---------------------------------------------------------------------------
# Number formats (inputs are decoded from, and results compared in, the
# storage formats the device path uses).
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16) to float64 exactly."""
    u = np.asarray(u16, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significand bits), ties
    to even, returned as float64.  Exact: frexp splits v = m * 2**e with
    0.5 <= |m| < 1, m * 256 is exact in float64, and numpy's round() is
    round-half-to-even.  Normal range only (no bf16 subnormals in the tests)."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    r = np.round(m * 256.0)
    out = np.ldexp(r, e - 8)
    return np.where(np.isfinite(x), out, x)


def round_to_f32(x: np.ndarray) -> np.ndarray:
    """Round float64 to the nearest float32 (IEEE, ties to even) as float64."""
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
