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
