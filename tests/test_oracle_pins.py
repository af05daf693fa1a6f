"""Pins for the CPU oracle: each test fixes the oracle against something other
than itself (closed forms, brute force, stated invariants, hand-worked values).

A plausible mistake in the oracle (a dropped polynomial term, a wrong sign, a
transposed operand, an off-by-one causal mask, sqrt(min) for sqrt(max), gamma
instead of sqrt(gamma) on q^C/k^C) fails at least one of these.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "hand_examples.json")))
QUINTIC = (3.4445, -4.7750, 2.0315)
CUBIC = (1.5, -0.5, 0.0)


def scalar_poly(x, coeffs, steps):
    """Scalar recursion x <- a x + b x^3 + c x^5 (the odd polynomial on one
    singular value), written out independently of the oracle's matrix form."""
    a, b, c = coeffs
    x = np.asarray(x, np.float64).copy()
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def random_orthogonal(n, rng):
    q, r = np.linalg.qr(rng.standard_normal((n, n)))
    return q * np.sign(np.diag(r))


def svd_built(r, c, s, rng):
    """M = U diag(s) V^T with random orthogonal U, V; returns (M, U_k, V_k)."""
    k = min(r, c)
    U = random_orthogonal(r, rng)[:, :k]
    V = random_orthogonal(c, rng)[:, :k]
    return (U * s) @ V.T, U, V


# --------------------------------------------------------------------------
# Hand-worked values
# --------------------------------------------------------------------------

def test_golden_momentum():
    g = GOLD["momentum"]
    M = np.zeros(())
    for want in g["M"]:
        M = O.momentum(M, np.array(g["G"]), g["mu"])
        assert float(M) == pytest.approx(want, abs=1e-15)


def test_golden_apply():
    g = GOLD["apply"]
    w = O.muon_apply(np.array(g["W"]), np.array(g["O"]), g["lr"], g["weight_decay"])
    assert float(w) == pytest.approx(g["W_new"], abs=1e-15)


def test_golden_newton_schulz_one_step():
    g = GOLD["newton_schulz_one_step"]
    X = O.newton_schulz(np.array(g["M"]), g["steps"], tuple(g["coeffs"]), g["eps"])
    np.testing.assert_allclose(X, np.array(g["X1"]), atol=1e-12)


def test_golden_max_logit():
    g = GOLD["max_logit"]
    Q = np.array(g["Q"], np.float64)[None, :, None, :]
    K = np.array(g["K"], np.float64)[None, :, None, :]
    for causal, key in ((True, "causal"), (False, "non_causal")):
        s, arg = O.max_logit(Q, K, causal=causal)
        assert s[0] == pytest.approx(g[key]["S"], abs=1e-15)
        assert list(arg[0]) == g[key]["argmax_bij"]


def test_golden_clip_mha():
    g = GOLD["clip_mha"]
    W = {"Wq": np.ones((4, 3)), "Wk": np.full((4, 3), 2.0)}
    out, gamma, mask = O.qk_clip(W, O.mha_segments(1, 4), np.array([g["S"]]), g["tau"])
    assert gamma[0] == pytest.approx(g["gamma"], abs=1e-15)
    np.testing.assert_allclose(out["Wq"], g["row_factor"], atol=1e-15)
    np.testing.assert_allclose(out["Wk"], 2.0 * g["row_factor"], atol=1e-15)


def test_golden_clip_mla():
    g = GOLD["clip_mla"]
    dn, dr, dv = 4, 2, 3
    W = {"W_UQ": np.ones((dn + dr, 5)), "W_UKV": np.ones((dn + dv, 5))}
    out, gamma, _ = O.qk_clip(W, O.mla_segments(1, dn, dr, dv), np.array([g["S"]]), g["tau"])
    f = g["factors"]
    assert gamma[0] == g["gamma"]
    np.testing.assert_array_equal(out["W_UQ"][:dn], f["q_C"])
    np.testing.assert_array_equal(out["W_UQ"][dn:], f["q_R"])
    np.testing.assert_array_equal(out["W_UKV"][:dn], f["k_C"])
    np.testing.assert_array_equal(out["W_UKV"][dn:], 1.0)       # v rows untouched


# --------------------------------------------------------------------------
# Momentum
# --------------------------------------------------------------------------

def test_momentum_closed_form():
    rng = np.random.default_rng(0)
    G = rng.standard_normal((7, 5))
    mu = 0.95
    M = np.zeros_like(G)
    for t in range(1, 31):
        M = O.momentum(M, G, mu)
        np.testing.assert_allclose(M, G * (1 - mu ** t) / (1 - mu), rtol=1e-13)


def test_momentum_zero_mu_is_gradient():
    rng = np.random.default_rng(1)
    G, M = rng.standard_normal((3, 4)), rng.standard_normal((3, 4))
    np.testing.assert_array_equal(O.momentum(M, G, 0.0), G)


# --------------------------------------------------------------------------
# Newton-Schulz
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(24, 40), (40, 24), (16, 16)])
@pytest.mark.parametrize("coeffs", [QUINTIC, CUBIC])
@pytest.mark.parametrize("steps", [1, 5])
def test_ns_svd_closed_form(shape, coeffs, steps):
    """NS(U diag(s) V^T) = U diag(p^steps(s / ||s||)) V^T (exact arithmetic)."""
    rng = np.random.default_rng(hash((shape, coeffs, steps)) % 2**32)
    k = min(shape)
    s = np.exp(rng.uniform(np.log(1e-2), 0.0, k))
    M, U, V = svd_built(*shape, s, rng)
    x = s / np.linalg.norm(s)
    want = (U * scalar_poly(x, coeffs, steps)) @ V.T
    got = O.newton_schulz(M, steps, coeffs, eps=0.0)
    np.testing.assert_allclose(got, want, atol=1e-10)


def test_ns_diagonal_is_scalar_recursion():
    d = np.array([3.0, -1.0, 0.5, 2.0])
    M = np.zeros((4, 6))
    M[np.arange(4), np.arange(4)] = d
    got = O.newton_schulz(M, 5, QUINTIC, eps=0.0)
    x = d / np.linalg.norm(d)
    np.testing.assert_allclose(np.diag(got[:, :4]), scalar_poly(x, QUINTIC, 5), atol=1e-12)
    assert np.count_nonzero(got[:, 4:]) == 0


def test_ns_rank_one_cubic_fixed_point():
    """Normalised rank-1 M has its one singular value at 1, where the cubic
    1.5x - 0.5x^3 is fixed: NS(sigma u v^T) = u v^T."""
    rng = np.random.default_rng(3)
    u = rng.standard_normal(9); u /= np.linalg.norm(u)
    v = rng.standard_normal(13); v /= np.linalg.norm(v)
    got = O.newton_schulz(7.5 * np.outer(u, v), 5, CUBIC, eps=0.0)
    np.testing.assert_allclose(got, np.outer(u, v), atol=1e-14)


def test_ns_singular_values_in_band():
    """Exact NS maps each normalised singular value x through p^5, so the output
    spectrum lies in [min p^5, max p^5] over the input range."""
    rng = np.random.default_rng(4)
    M = rng.standard_normal((48, 96))
    sv_in = np.linalg.svd(M, compute_uv=False)
    x = sv_in / np.linalg.norm(sv_in)
    grid = np.linspace(x.min(), x.max(), 20001)
    band = scalar_poly(grid, QUINTIC, 5)
    sv_out = np.linalg.svd(O.newton_schulz(M, 5, QUINTIC, eps=0.0), compute_uv=False)
    assert sv_out.min() >= band.min() - 1e-9 and sv_out.max() <= band.max() + 1e-9
    np.testing.assert_allclose(np.sort(sv_out), np.sort(scalar_poly(x, QUINTIC, 5)), atol=1e-10)


def test_ns_zero_matrix_gives_zero():
    got = O.newton_schulz(np.zeros((5, 8)), 5, QUINTIC, eps=1e-7)
    assert np.all(got == 0.0)


@pytest.mark.parametrize("shape", [(20, 50), (50, 20)])
def test_rms_match_is_point_two(shape):
    """With msign exact (60 cubic steps converge every singular value to 1),
    O = msign(M) * sqrt(max(n, m)) * 0.2 has RMS exactly 0.2 (Algorithm 1's
    "Match Adam RMS")."""
    rng = np.random.default_rng(5)
    s = rng.uniform(0.3, 1.0, min(shape))
    M, _, _ = svd_built(*shape, s, rng)
    hp = O.Hparams(ns_steps=60, ns_coeffs=CUBIC, ns_eps=0.0)
    Od = O.muon_direction(M, hp)
    assert math.sqrt(np.mean(Od ** 2)) == pytest.approx(0.2, abs=1e-12)


def test_update_decay_only():
    rng = np.random.default_rng(6)
    W = rng.standard_normal((6, 10))
    hp = O.Hparams()
    Wn, M, Od = O.muon_step(W, np.zeros_like(W), np.zeros_like(W), hp)
    np.testing.assert_array_equal(Od, 0.0)
    np.testing.assert_allclose(Wn, (1 - hp.lr * hp.weight_decay) * W, rtol=1e-15)


def test_update_descends():
    """The step moves W against the momentum direction: <W_new - W, M> < 0."""
    rng = np.random.default_rng(7)
    W = rng.standard_normal((16, 24)) * 0.02
    G = rng.standard_normal((16, 24))
    hp = O.Hparams(weight_decay=0.0)
    Wn, M, Od = O.muon_step(W, G, np.zeros_like(W), hp)
    assert np.sum((Wn - W) * M) < 0


# --------------------------------------------------------------------------
# Max logit
# --------------------------------------------------------------------------

def brute_max_logit(Q, K, Ks, causal):
    """Explicit loops over (b, i, j) and the feature index; no matrix products."""
    B, S, H, dq = Q.shape
    out, arg = [], []
    for h in range(H):
        best, at = -math.inf, None
        for b in range(B):
            for i in range(S):
                for j in range(S):
                    if causal and j > i:
                        continue
                    kv = list(K[b, j, h]) + (list(Ks[b, j]) if Ks is not None else [])
                    dot = 0.0
                    for t in range(dq):
                        dot += float(Q[b, i, h, t]) * float(kv[t])
                    if dot > best:
                        best, at = dot, (b, i, j)
        out.append(best / math.sqrt(dq))
        arg.append(at)
    return np.array(out), np.array(arg)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("mla", [False, True])
def test_max_logit_brute_force(causal, mla):
    rng = np.random.default_rng(10 + causal + 2 * mla)
    B, S, H = 2, 6, 3
    if mla:
        Q = rng.standard_normal((B, S, H, 5))
        K = rng.standard_normal((B, S, H, 3))
        Ks = rng.standard_normal((B, S, 2))
    else:
        Q = rng.standard_normal((B, S, H, 4))
        K = rng.standard_normal((B, S, H, 4))
        Ks = None
    s, arg = O.max_logit(Q, K, Ks, causal=causal)
    sb, ab = brute_max_logit(Q, K, Ks, causal)
    np.testing.assert_allclose(s, sb, rtol=1e-13)
    np.testing.assert_array_equal(arg, ab)


def test_max_logit_row_chunking_is_exact():
    rng = np.random.default_rng(11)
    Q = rng.standard_normal((1, 37, 2, 8)); K = rng.standard_normal((1, 37, 2, 8))
    a, aa = O.max_logit(Q, K)
    b, bb = O.max_logit(Q, K, row_chunk=5)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(aa, bb)


def test_max_logit_single_token():
    rng = np.random.default_rng(12)
    Q = rng.standard_normal((1, 1, 2, 16)); K = rng.standard_normal((1, 1, 2, 16))
    s, _ = O.max_logit(Q, K)
    np.testing.assert_allclose(s, np.einsum("hd,hd->h", Q[0, 0], K[0, 0]) / 4.0, rtol=1e-14)


def test_max_logit_homogeneous_per_head():
    rng = np.random.default_rng(13)
    Q = rng.standard_normal((2, 9, 3, 8)); K = rng.standard_normal((2, 9, 3, 8))
    # make every head's max positive so positive scaling commutes with max
    Q[0, 4, :, :] = 10 * K[0, 2, :, :]
    s0, _ = O.max_logit(Q, K)
    Q2 = Q.copy(); Q2[:, :, 1, :] *= 3.0
    s1, _ = O.max_logit(Q2, K)
    assert s1[1] == pytest.approx(3.0 * s0[1], rel=1e-14)
    assert s1[0] == s0[0] and s1[2] == s0[2]


# --------------------------------------------------------------------------
# QK-Clip
# --------------------------------------------------------------------------

def test_clip_factors_edges():
    g, m = O.clip_factors(np.array([50.0, 100.0, 150.0, 0.0, -5.0, np.nan, 400.0]), 100.0)
    np.testing.assert_array_equal(m, [False, False, True, False, False, False, True])
    np.testing.assert_allclose(g, [1, 1, 100 / 150, 1, 1, 1, 0.25])


def test_clip_below_tau_is_bit_identical():
    rng = np.random.default_rng(20)
    W = {"Wq": rng.standard_normal((8, 5)), "Wk": rng.standard_normal((8, 5))}
    out, g, m = O.qk_clip(W, O.mha_segments(2, 4), np.array([99.0, 100.0]), 100.0)
    assert not m.any()
    for k in W:
        np.testing.assert_array_equal(out[k], W[k])


def mha_layer(rng, D=32, H=4, d=8, scale_heads=(1, 3), r=25.0):
    Wq = rng.standard_normal((H * d, D)) * 0.3
    Wk = rng.standard_normal((H * d, D)) * 0.3
    for h in scale_heads:
        Wq[h * d:(h + 1) * d] *= r
        Wk[h * d:(h + 1) * d] *= r
    X = rng.standard_normal((2, 12, D))
    return X, Wq, Wk


def test_clip_mha_remeasured_is_min_s_tau():
    """After the clip, the re-measured max logit is min(S, tau) per head, and
    only the offending heads' rows changed ([K2-explained]: the factor
    "brings that maximum back to tau"; heads under tau untouched)."""
    rng = np.random.default_rng(21)
    H, d, tau = 4, 8, 100.0
    X, Wq, Wk = mha_layer(rng, H=H, d=d)
    S0, _ = O.max_logit(*O.project_mha(X, Wq, Wk, H))
    assert (S0 > tau).sum() == 2 and (S0 < tau).sum() == 2
    out, g, m = O.qk_clip({"Wq": Wq, "Wk": Wk}, O.mha_segments(H, d), S0, tau)
    S1, _ = O.max_logit(*O.project_mha(X, out["Wq"], out["Wk"], H))
    np.testing.assert_allclose(S1, np.minimum(S0, tau), rtol=1e-12)
    for h in range(H):
        rows = slice(h * d, (h + 1) * d)
        same = np.array_equal(out["Wq"][rows], Wq[rows]) and np.array_equal(out["Wk"][rows], Wk[rows])
        assert same == (not m[h])


@pytest.mark.parametrize("alpha", [0.5, 0.25])
def test_clip_mha_alpha_split(alpha):
    rng = np.random.default_rng(22)
    Wq, Wk = rng.standard_normal((4, 3)), rng.standard_normal((4, 3))
    out, g, _ = O.qk_clip({"Wq": Wq, "Wk": Wk}, O.mha_segments(1, 4, alpha), np.array([400.0]), 100.0)
    np.testing.assert_allclose(out["Wq"], Wq * 0.25 ** alpha, rtol=1e-15)
    np.testing.assert_allclose(out["Wk"], Wk * 0.25 ** (1 - alpha), rtol=1e-15)


def test_clip_mla_remeasured_and_shared_key_untouched():
    """MLA: q^C, k^C by sqrt(gamma), q^R by gamma, k^R (shared) and v untouched;
    every head's logits then scale by exactly gamma_h ([K2-explained])."""
    rng = np.random.default_rng(23)
    H, dn, dr, dv, D, ql, kl = 4, 8, 4, 8, 40, 24, 12
    W = {
        "W_DQ": rng.standard_normal((ql, D)) * 0.2,
        "W_UQ": rng.standard_normal((H * (dn + dr), ql)) * 0.4,
        "W_DKV": rng.standard_normal((kl, D)) * 0.2,
        "W_UKV": rng.standard_normal((H * (dn + dv), kl)) * 0.4,
        "W_KR": rng.standard_normal((dr, D)) * 0.4,
    }
    for h in (0, 2):
        W["W_UQ"][h * (dn + dr):(h + 1) * (dn + dr)] *= 12.0
        W["W_UKV"][h * (dn + dv):h * (dn + dv) + dn] *= 12.0
    X = rng.standard_normal((1, 10, D))
    args = lambda w: (X, w["W_DQ"], w["W_UQ"], w["W_DKV"], w["W_UKV"], w["W_KR"], H, dn, dr, dv)
    S0, _ = O.max_logit(*O.project_mla(*args(W)))
    tau = float(np.sort(S0)[1] + np.sort(S0)[2]) / 2      # two heads above, two below
    out, g, m = O.qk_clip(W, O.mla_segments(H, dn, dr, dv), S0, tau)
    assert m.sum() == 2
    S1, _ = O.max_logit(*O.project_mla(*args(out)))
    np.testing.assert_allclose(S1, np.minimum(S0, tau), rtol=1e-12)
    np.testing.assert_array_equal(out["W_KR"], W["W_KR"])
    for h in range(H):
        vrows = slice(h * (dn + dv) + dn, (h + 1) * (dn + dv))
        np.testing.assert_array_equal(out["W_UKV"][vrows], W["W_UKV"][vrows])
    # whole-logit scaling by gamma: every (i, j) logit of a clipped head
    q0, kc0, kr0 = O.project_mla(*args(W))
    q1, kc1, kr1 = O.project_mla(*args(out))
    for h in range(H):
        L0 = q0[0, :, h] @ np.concatenate([kc0[0, :, h], kr0[0]], 1).T
        L1 = q1[0, :, h] @ np.concatenate([kc1[0, :, h], kr1[0]], 1).T
        np.testing.assert_allclose(L1, g[h] * L0, rtol=1e-11, atol=1e-12)


def test_total_clip_variant():
    assert O.total_clip_factor(np.array([10.0, 250.0, 50.0]), 100.0) == pytest.approx(0.4)
    assert O.total_clip_factor(np.array([10.0, 50.0]), 100.0) == 1.0
    assert O.total_clip_factor(np.array([100.0, 50.0]), 100.0) == 1.0
    assert O.total_clip_factor(np.array([np.nan, 500.0]), 100.0) == 1.0


def test_total_clip_scales_every_head_and_caps_the_max():
    """Total clip ([K2-internals] 核心数学, naive form): all heads share one
    gamma, so the largest re-measured max logit becomes exactly tau and the
    others shrink by the same factor."""
    rng = np.random.default_rng(25)
    H, d, tau = 4, 8, 100.0
    X, Wq, Wk = mha_layer(rng, H=H, d=d)
    S0, _ = O.max_logit(*O.project_mha(X, Wq, Wk, H))
    out, g = O.qk_clip_total({"Wq": Wq, "Wk": Wk}, O.mha_segments(H, d), S0, tau)
    S1, _ = O.max_logit(*O.project_mha(X, out["Wq"], out["Wk"], H))
    assert g == pytest.approx(tau / S0.max())
    np.testing.assert_allclose(S1, S0 * g, rtol=1e-12)
    assert S1.max() == pytest.approx(tau, rel=1e-12)


@pytest.mark.parametrize("shape", [(20, 50), (50, 20)])
def test_spectral_scale_gives_unit_or_aspect_norm(shape):
    """MuP-style scale sqrt(max(1, out/in)): with converged msign every singular
    value of O equals the scale (zhihu answer, section 3.2)."""
    rng = np.random.default_rng(26)
    s = rng.uniform(0.3, 1.0, min(shape))
    M, _, _ = svd_built(*shape, s, rng)
    hp = O.Hparams(ns_steps=60, ns_coeffs=CUBIC, ns_eps=0.0, scale_mode="spectral")
    sv = np.linalg.svd(O.muon_direction(M, hp), compute_uv=False)
    want = math.sqrt(max(1.0, shape[0] / shape[1]))
    np.testing.assert_allclose(sv, want, rtol=1e-12)


def test_muonclip_step_order_muon_then_clip():
    """Algorithm 1: Muon updates every matrix, then the clip rescales the
    updated weights with S from this step's forward."""
    rng = np.random.default_rng(24)
    H, d = 2, 4
    W = {"Wq": rng.standard_normal((8, 6)) * 0.1, "Wk": rng.standard_normal((8, 6)) * 0.1}
    G = {k: rng.standard_normal(v.shape) for k, v in W.items()}
    M = {k: np.zeros_like(v) for k, v in W.items()}
    hp = O.Hparams()
    smax = np.array([300.0, 20.0])
    Wn, Mn, gam = O.muonclip_step(W, G, M, hp, [(smax, O.mha_segments(H, d))])
    for k in W:
        Wm, _, _ = O.muon_step(W[k], G[k], M[k], hp)
        want = Wm.copy(); want[:d] *= math.sqrt(100.0 / 300.0)
        np.testing.assert_allclose(Wn[k], want, rtol=1e-15)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def test_round_to_bf16_ties_and_exact_values():
    one = 1.0
    ulp = 2.0 ** -7
    vals = np.array([one, one + ulp / 2, one + 3 * ulp / 2, one + ulp / 2 + 1e-12, -2.75, 0.0])
    want = np.array([one, one, one + 2 * ulp, one + ulp, -2.75, 0.0])
    np.testing.assert_array_equal(O.round_to_bf16(vals), want)


def test_bf16_decode():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000], np.uint16)
    np.testing.assert_array_equal(O.bf16_bits_to_f64(bits), [1.0, -2.0, 1.0 + 2 ** -7, 0.0])


# ------------------------------------------------------------------ attention forward (S_max fused)
def _attn_inputs(B, S, H, dq, dv, seed, dr=0):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, S, H, dq))
    K = rng.standard_normal((B, S, H, dq - dr))
    Ks = rng.standard_normal((B, S, dr)) if dr else None
    V = rng.standard_normal((B, S, H, dv))
    return Q, K, Ks, V


def test_attention_zero_queries_average_the_prefix():
    """Q = 0: every logit is 0, so row i averages V_0..V_i and lse_i = log(i + 1)."""
    _, K, _, V = _attn_inputs(2, 9, 3, 8, 5, 40)
    Q = np.zeros((2, 9, 3, 8))
    Out, lse, smax = O.attention_forward(Q, K, V)
    prefix_mean = np.cumsum(V, axis=1) / np.arange(1, 10)[None, :, None, None]
    np.testing.assert_allclose(Out, prefix_mean, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, 10)), (2, 3, 9)), atol=1e-14)
    np.testing.assert_array_equal(smax, np.zeros(3))
    Out_nc, lse_nc, _ = O.attention_forward(Q, K, V, causal=False)
    np.testing.assert_allclose(Out_nc, np.broadcast_to(V.mean(axis=1, keepdims=True), V.shape), atol=1e-14)
    np.testing.assert_allclose(lse_nc, np.log(9.0), atol=1e-14)


def test_attention_one_hot_key_closed_form():
    """One key j* with q.k = c, every other logit 0: row i >= j* gets
    (e^{c s} V_j* + sum_{j != j*, j <= i} V_j) / (e^{c s} + i), s the scale."""
    S, d, dv, js, c = 7, 4, 3, 2, 3.0
    Q = np.zeros((1, S, 1, d)); Q[0, :, 0, 0] = 1.0
    K = np.zeros((1, S, 1, d)); K[0, js, 0, 0] = c
    V = np.random.default_rng(41).standard_normal((1, S, 1, dv))
    Out, lse, smax = O.attention_forward(Q, K, V)
    s = 1.0 / math.sqrt(d)
    for i in range(S):
        others = [V[0, j, 0] for j in range(i + 1) if j != js]
        if i >= js:
            w = math.exp(c * s)
            want = (w * V[0, js, 0] + sum(others, np.zeros(dv))) / (w + i)
            np.testing.assert_allclose(lse[0, 0, i], math.log(w + i), atol=1e-14)
        else:
            want = sum(others, np.zeros(dv)) / (i + 1)
        np.testing.assert_allclose(Out[0, i, 0], want, atol=1e-14)
    assert smax[0] == pytest.approx(c * s, abs=1e-15)


def test_attention_constant_values_pass_through():
    Q, K, Ks, _ = _attn_inputs(1, 12, 2, 10, 4, 42, dr=3)
    V = np.broadcast_to(np.array([1.5, -2.0, 0.25, 7.0]), (1, 12, 2, 4)).copy()
    Out, _, _ = O.attention_forward(Q, K, V, Ks)
    np.testing.assert_allclose(Out, V, rtol=1e-13)


def test_attention_row_shift_changes_only_lse():
    """Adding u to every key adds scale * q_i . u to row i's logits: O is
    unchanged (softmax shift invariance) and lse moves by exactly that."""
    Q, K, _, V = _attn_inputs(1, 10, 2, 6, 3, 43)
    u = np.random.default_rng(44).standard_normal(6)
    O1, l1, _ = O.attention_forward(Q, K, V)
    O2, l2, _ = O.attention_forward(Q, K + u, V)
    np.testing.assert_allclose(O2, O1, atol=1e-12)
    shift = np.einsum("bshd,d->bhs", Q, u) / math.sqrt(6)
    np.testing.assert_allclose(l2 - l1, shift, atol=1e-12)


def test_attention_key_permutation_invariance_without_mask():
    Q, K, Ks, V = _attn_inputs(2, 11, 2, 8, 4, 45, dr=2)
    perm = np.random.default_rng(46).permutation(11)
    O1, l1, s1 = O.attention_forward(Q, K, V, Ks, causal=False)
    O2, l2, s2 = O.attention_forward(Q, K[:, perm], V[:, perm], Ks[:, perm], causal=False)
    np.testing.assert_allclose(O2, O1, atol=1e-13)
    np.testing.assert_allclose(l2, l1, atol=1e-13)
    np.testing.assert_array_equal(s2, s1)


@pytest.mark.parametrize("mla", [False, True])
def test_attention_smax_is_the_max_logit(mla):
    Q, K, Ks, V = _attn_inputs(2, 13, 3, 12, 5, 47, dr=4 if mla else 0)
    _, _, smax = O.attention_forward(Q, K, V, Ks, row_chunk=5)
    ref, _ = O.max_logit(Q, K, Ks)
    np.testing.assert_allclose(smax, ref, rtol=1e-15)


# ------------------------------------------------------------------ setup projection: RoPE, RMSNorm
# The MLA feature projection (the untimed setup forward) uses a rotary
# embedding on interleaved pairs and a weightless RMSNorm.  Both are pinned
# by properties that fix them up to nothing: the rotation of each pair by a
# position-proportional angle, its frequencies, its direction and the norm.

def test_rope_hand_worked_angles():
    """d = 2: the one pair turns by p radians at position p (frequency
    theta^0 = 1).  d = 4, theta = 100: the second pair's frequency is
    100^(-2/4) = 0.1, so at position 3 it turns by 0.3 rad.  The direction is
    counter-clockwise: (1, 0) -> (cos a, sin a), (0, 1) -> (-sin a, cos a)."""
    x = np.zeros((1, 3, 2))
    x[0, 1] = (1.0, 0.0)
    x[0, 2] = (0.0, 1.0)
    y = O.rope(x, theta=10000.0)
    np.testing.assert_allclose(y[0, 1], [math.cos(1.0), math.sin(1.0)], atol=1e-15)
    np.testing.assert_allclose(y[0, 2], [-math.sin(2.0), math.cos(2.0)], atol=1e-15)
    x4 = np.zeros((1, 4, 4))
    x4[0, 3] = (0.0, 0.0, 2.0, -1.0)
    y4 = O.rope(x4, theta=100.0)
    a = 0.3
    want = (0.0, 0.0, 2.0 * math.cos(a) + math.sin(a), 2.0 * math.sin(a) - math.cos(a))
    np.testing.assert_allclose(y4[0, 3], want, atol=1e-15)


def test_rope_position_zero_is_identity_and_pairs_keep_their_norm():
    rng = np.random.default_rng(40)
    x = rng.standard_normal((2, 37, 3, 64))
    y = O.rope(x)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])
    n_in = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_out = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)
    # a pair stays in its own two coordinates
    e = np.zeros((1, 9, 8))
    e[0, :, 4] = 1.0
    z = O.rope(e)
    assert np.all(z[0, :, [0, 1, 2, 3, 6, 7]] == 0.0)


def test_rope_logits_depend_only_on_relative_position():
    """With the same query vector q at every position and the same key vector
    k, rope(q)_i . rope(k)_j is a function of i - j alone (the property that
    makes the embedding relative)."""
    rng = np.random.default_rng(41)
    d, S = 64, 50
    q = np.broadcast_to(rng.standard_normal(d), (1, S, d)).copy()
    k = np.broadcast_to(rng.standard_normal(d), (1, S, d)).copy()
    rq, rk = O.rope(q)[0], O.rope(k)[0]
    for delta in (0, 1, 7, 30):
        vals = [rq[i] @ rk[i - delta] for i in range(delta, S)]
        np.testing.assert_allclose(vals, vals[0], rtol=1e-10, atol=1e-10)
    assert abs(rq[10] @ rk[3] - rq[3] @ rk[10]) > 1e-6      # and on its sign


def test_rms_norm_unit_rms_scale_invariance_and_hand_value():
    rng = np.random.default_rng(42)
    x = rng.standard_normal((5, 7, 512)) * rng.uniform(0.1, 10.0, size=(5, 7, 1))
    y = O.rms_norm(x, eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y ** 2, axis=-1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(O.rms_norm(3.5 * x, eps=0.0), y, rtol=1e-12)
    assert np.all(np.sign(y) == np.sign(x))
    # [3, 4]: mean square 12.5, so y = [3, 4] / sqrt(12.5)
    np.testing.assert_allclose(O.rms_norm(np.array([3.0, 4.0]), eps=0.0),
                               [3.0 / math.sqrt(12.5), 4.0 / math.sqrt(12.5)], rtol=1e-15)
    # eps enters under the root: [1e-3, 1e-3] with eps 1e-6 -> 1e-3 / sqrt(2e-6)
    np.testing.assert_allclose(O.rms_norm(np.array([1e-3, 1e-3]), eps=1e-6),
                               1e-3 / math.sqrt(2e-6), rtol=1e-12)
