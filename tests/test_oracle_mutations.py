"""Each plausible oracle mistake, planted on the CPU through monkeypatch, must
make at least one pin in test_oracle_pins fail.  This shows that the pins
constrain the oracle rather than restate it."""
import numpy as np
import pytest

import oracle as O
import oracle.muonclip_oracle as OM
from tests import test_oracle_pins as P


def _ns_dropped_quintic(X, steps, coeffs=O.DEFAULT_NS_COEFFS):
    a, b, c = coeffs
    for _ in range(steps):
        A = X @ X.T
        X = a * X + (b * A) @ X                      # c A^2 term dropped
    return X


def _newton_schulz_no_unorient(M, steps=5, coeffs=O.DEFAULT_NS_COEFFS, eps=1e-7):
    M = np.asarray(M, np.float64)
    X = M.T if M.shape[0] > M.shape[1] else M
    X = X / (np.linalg.norm(X) + eps)
    return OM.ns_iterate(X, steps, coeffs)                 # forgot to transpose back


def _ns_wrong_sign(X, steps, coeffs=O.DEFAULT_NS_COEFFS):
    a, b, c = coeffs
    for _ in range(steps):
        A = X @ X.T
        X = a * X - (b * A + c * (A @ A)) @ X
    return X


def _apply_wrong_sign(W_prev, Od, lr, wd):
    return W_prev - lr * (Od - wd * W_prev)


def _direction_sqrt_min(M, hp):
    r, c = M.shape
    return O.newton_schulz(M, hp.ns_steps, hp.ns_coeffs, hp.ns_eps) * (min(r, c) ** 0.5 * hp.rms_scale)


def _mla_segments_gamma_on_qc(H, d_nope=128, d_rope=64, d_v=128):
    dq, dkv = d_nope + d_rope, d_nope + d_v
    return [O.ClipSegment("W_UQ", 0, dq, d_nope, 1.0),          # gamma instead of sqrt(gamma)
            O.ClipSegment("W_UQ", d_nope, dq, d_rope, 1.0),
            O.ClipSegment("W_UKV", 0, dkv, d_nope, 0.5)]


def _max_logit_strict_causal(Q, K, K_shared=None, causal=True, scale=None, row_chunk=2048):
    # off by one: excludes the diagonal j == i
    import math
    B, S, H, dq = Q.shape
    scale = 1 / math.sqrt(dq) if scale is None else scale
    out = np.full(H, -np.inf); arg = np.zeros((H, 3), np.int64)
    for h in range(H):
        for b in range(B):
            k = O.head_keys(K, K_shared, b, h)
            L = np.asarray(Q[b, :, h, :], np.float64) @ k.T
            if causal:
                L = np.where(np.arange(S)[None, :] < np.arange(S)[:, None], L, -np.inf)
            if S == 1:
                L = np.full((1, 1), -np.inf)
            v = L.max()
            if v * scale > out[h]:
                out[h] = v * scale
    return out, arg


def _momentum_nesterov(M_prev, G, mu):
    return mu * (mu * M_prev + G) + G


def _attention_unmasked(Q, K, V, K_shared=None, causal=True, scale=None, row_chunk=1024):
    return _attn_real(Q, K, V, K_shared, False, scale, row_chunk)         # causal mask dropped


def _attention_scale_one_over_d(Q, K, V, K_shared=None, causal=True, scale=None, row_chunk=1024):
    return _attn_real(Q, K, V, K_shared, causal, 1.0 / Q.shape[3], row_chunk)


def _attention_values_of_query(Q, K, V, K_shared=None, causal=True, scale=None, row_chunk=1024):
    Out, lse, smax = _attn_real(Q, K, V, K_shared, causal, scale, row_chunk)
    return Out[:, ::-1], lse, smax                                        # rows reversed


def _attention_unnormalised(Q, K, V, K_shared=None, causal=True, scale=None, row_chunk=1024):
    Out, lse, smax = _attn_real(Q, K, V, K_shared, causal, scale, row_chunk)
    den = np.exp(lse).transpose(0, 2, 1)[..., None]
    return Out * den, lse, smax                                           # no division by the sum


_attn_real = OM.attention_forward
_rope_real = OM.rope
_rms_real = OM.rms_norm


def _rope_clockwise(x, theta=10000.0):
    # the rotation by -angle: apply the real one to the conjugate pair and conjugate back
    xc = x.copy()
    xc[..., 1::2] *= -1.0
    yc = _rope_real(xc, theta)
    yc[..., 1::2] *= -1.0
    return yc


def _rope_positions_from_one(x, theta=10000.0):
    S = x.shape[1]
    pad = np.concatenate([np.zeros_like(x[:, :1]), x], axis=1)
    return _rope_real(pad, theta)[:, 1:S + 1]                            # angle (p + 1) at p


def _rope_frequency_over_d_half(x, theta=10000.0):
    return _rope_real(x, theta ** 0.5)                                   # theta^(-t/d) for pair t


def _rms_norm_mean_abs(x, eps=1e-6):
    x = np.asarray(x, np.float64)
    return x / (np.mean(np.abs(x), axis=-1, keepdims=True) + eps)         # mean |x| for the RMS


def _rms_norm_eps_outside(x, eps=1e-6):
    x = np.asarray(x, np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps)

def _mla_segments_sqrt_gamma_on_qr(H, d_nope=128, d_rope=64, d_v=128):
    dq, dkv = d_nope + d_rope, d_nope + d_v
    return [O.ClipSegment("W_UQ", 0, dq, d_nope, 0.5), O.ClipSegment("W_UQ", d_nope, dq, d_rope, 0.5),
            O.ClipSegment("W_UKV", 0, dkv, d_nope, 0.5)]


def _clip_factors_at_tau(smax, tau):
    # S = tau clips (the pseudocode skips S <= tau)
    smax = np.asarray(smax, np.float64)
    mask = smax >= tau
    gamma = np.ones_like(smax)
    gamma[mask] = tau / smax[mask]
    return gamma, mask


def _clip_factors_inverted(smax, tau):
    smax = np.asarray(smax, np.float64)
    mask = smax > tau
    gamma = np.ones_like(smax)
    gamma[mask] = smax[mask] / tau
    return gamma, mask


def _qk_clip_head_rows_by_height(weights, segments, smax, tau):
    # head h's block found at h * rows instead of h * stride
    gamma, mask = O.clip_factors(smax, tau)
    out = {k: np.array(v, np.float64) for k, v in weights.items()}
    for seg in segments:
        W = out[seg.name]
        for h in np.nonzero(mask)[0]:
            r0 = seg.offset + h * seg.rows
            W[r0:r0 + seg.rows] *= gamma[h] ** seg.exponent
    return out, gamma, mask


def _total_clip_smallest_head(smax, tau):
    s = float(np.min(smax))
    return tau / s if s > tau else 1.0


def _update_scale_spectral_inverted(rows, cols, hp):
    if hp.scale_mode == "spectral":
        return np.sqrt(max(1.0, cols / rows))
    return np.sqrt(max(rows, cols)) * hp.rms_scale


def _mha_segments_alpha_swapped(H, d, alpha=0.5):
    return [O.ClipSegment("Wq", 0, d, d, 1.0 - alpha), O.ClipSegment("Wk", 0, d, d, alpha)]


def _newton_schulz_max_abs_normalised(M, steps=5, coeffs=O.DEFAULT_NS_COEFFS, eps=1e-7):
    M = np.asarray(M, np.float64)
    t = M.shape[0] > M.shape[1]
    X = M.T if t else M
    X = O.ns_iterate(X / (np.abs(X).max() + eps), steps, coeffs)
    return X.T if t else X


def _head_keys_shared_first(K, K_shared, b, h):
    k = np.asarray(K[b, :, h, :], np.float64)
    if K_shared is not None:
        k = np.concatenate([np.asarray(K_shared[b], np.float64), k], axis=1)
    return k


def _muonclip_step_clip_first(weights, grads, moms, hp, layers=()):
    W = {k: np.array(v, np.float64) for k, v in weights.items()}
    gammas = []
    for smax, segs in layers:
        W, gamma, _ = O.qk_clip(W, segs, smax, hp.tau)
        gammas.append(gamma)
    W_new, M_new = {}, {}
    for name in W:
        W_new[name], M_new[name], _ = O.muon_step(W[name], grads[name], moms[name], hp)
    return W_new, M_new, gammas


def _momentum_dampened(M_prev, G, mu):
    return mu * np.asarray(M_prev, np.float64) + (1.0 - mu) * np.asarray(G, np.float64)


_max_logit = O.max_logit


def _max_logit_scale_one_over_d(Q, K, K_shared=None, causal=True, scale=None, row_chunk=2048):
    return _max_logit(Q, K, K_shared, causal, 1.0 / Q.shape[-1] if scale is None else scale, row_chunk)


MUTATIONS = [
    ("ns_iterate", _ns_dropped_quintic, [P.test_golden_newton_schulz_one_step]),
    ("ns_iterate", _ns_wrong_sign, [P.test_golden_newton_schulz_one_step]),
    ("muon_apply", _apply_wrong_sign, [P.test_golden_apply]),
    ("muon_direction", _direction_sqrt_min, [lambda: P.test_rms_match_is_point_two((20, 50))]),
    ("mla_segments", _mla_segments_gamma_on_qc, [P.test_golden_clip_mla]),
    ("max_logit", _max_logit_strict_causal, [P.test_max_logit_single_token]),
    ("momentum", _momentum_nesterov, [P.test_golden_momentum]),
    ("attention_forward", _attention_unmasked, [P.test_attention_zero_queries_average_the_prefix]),
    ("attention_forward", _attention_scale_one_over_d, [P.test_attention_one_hot_key_closed_form]),
    ("attention_forward", _attention_values_of_query, [P.test_attention_one_hot_key_closed_form]),
    ("attention_forward", _attention_unnormalised, [P.test_attention_constant_values_pass_through]),
    ("rope", _rope_clockwise, [P.test_rope_hand_worked_angles]),
    ("rope", _rope_positions_from_one, [P.test_rope_position_zero_is_identity_and_pairs_keep_their_norm]),
    ("rope", _rope_frequency_over_d_half, [P.test_rope_hand_worked_angles]),
    ("rms_norm", _rms_norm_mean_abs, [P.test_rms_norm_unit_rms_scale_invariance_and_hand_value]),
    ("rms_norm", _rms_norm_eps_outside, [P.test_rms_norm_unit_rms_scale_invariance_and_hand_value]),
    ("mla_segments", _mla_segments_sqrt_gamma_on_qr, [P.test_clip_mla_remeasured_and_shared_key_untouched]),
    ("clip_factors", _clip_factors_at_tau, [P.test_clip_factors_edges]),
    ("clip_factors", _clip_factors_inverted, [P.test_clip_factors_edges]),
    ("qk_clip", _qk_clip_head_rows_by_height, [P.test_clip_mla_remeasured_and_shared_key_untouched]),
    ("total_clip_factor", _total_clip_smallest_head, [P.test_total_clip_variant]),
    ("update_scale", _update_scale_spectral_inverted,
     [lambda: P.test_spectral_scale_gives_unit_or_aspect_norm((50, 20))]),
    ("mha_segments", _mha_segments_alpha_swapped, [lambda: P.test_clip_mha_alpha_split(0.25)]),
    ("newton_schulz", _newton_schulz_max_abs_normalised,
     [lambda: P.test_ns_svd_closed_form((24, 40), P.QUINTIC, 1)]),
    ("head_keys", _head_keys_shared_first, [lambda: P.test_max_logit_brute_force(True, True)]),
    ("muonclip_step", _muonclip_step_clip_first, [P.test_muonclip_step_order_muon_then_clip]),
    ("momentum", _momentum_dampened, [P.test_momentum_closed_form]),
    ("max_logit", _max_logit_scale_one_over_d, [P.test_max_logit_single_token]),
]


@pytest.mark.parametrize("name,bad,pins", MUTATIONS, ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bad, pins):
    monkeypatch.setattr(OM, name, bad)
    monkeypatch.setattr(O, name, bad)
    caught = False
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            caught = True
    assert caught, f"planted mistake in {name} went unnoticed"


def test_missing_unorient_is_caught(monkeypatch):
    monkeypatch.setattr(OM, "newton_schulz", _newton_schulz_no_unorient)
    monkeypatch.setattr(O, "newton_schulz", _newton_schulz_no_unorient)
    with pytest.raises((AssertionError, ValueError)):
        P.test_ns_svd_closed_form((40, 24), P.QUINTIC, 1)
