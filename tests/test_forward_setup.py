"""The setup forward that builds Q/K for qk_max_logit (row a8: untimed, not part
of the MuonClip step) against the oracle's projections, whose RoPE and RMSNorm
are pinned in test_oracle_pins.  Both take the same inputs; the setup runs in
fp32 (CPU), the oracle in fp64, so they agree to fp32 rounding."""
import numpy as np
import torch

import oracle as O
from muon_qk_clip_gb300 import forward, synth


def test_project_mha_matches_oracle():
    B, S, D, H = 2, 16, 48, 4
    X = synth.normal((B, S, D), 1.0, "fx", 1)
    Wq = synth.normal((D, D), 0.1, "fq", 1)
    Wk = synth.normal((D, D), 0.1, "fk", 1)
    q, k = forward.project_mha(X, Wq, Wk, H)
    qo, ko = O.project_mha(X.double().numpy(), Wq.double().numpy(), Wk.double().numpy(), H)
    np.testing.assert_allclose(q.double().numpy(), qo, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(k.double().numpy(), ko, rtol=1e-5, atol=1e-5)


def test_project_mla_matches_oracle():
    """MLA features (R8 layout): q = [q^C || RoPE(q^R)] from the RMS-normed
    query latent, k^C from the RMS-normed key latent, and the shared rotary
    key RoPE(X W_KR^T)."""
    B, S, D, H, ql, kl, dn, dr, dv = 1, 24, 64, 3, 32, 16, 16, 8, 16
    W = {"W_DQ": synth.normal((ql, D), 0.1, "dq", 2), "W_UQ": synth.normal((H * (dn + dr), ql), 0.2, "uq", 2),
         "W_DKV": synth.normal((kl, D), 0.1, "dkv", 2), "W_UKV": synth.normal((H * (dn + dv), kl), 0.2, "ukv", 2),
         "W_KR": synth.normal((dr, D), 0.1, "kr", 2)}
    X = synth.normal((B, S, D), 1.0, "mx", 2)
    q, kc, kr, v = forward.project_mla(X, W, H, dn, dr, dv, with_v=True)
    Wd = {n: w.double().numpy() for n, w in W.items()}
    qo, kco, kro = O.project_mla(X.double().numpy(), Wd["W_DQ"], Wd["W_UQ"], Wd["W_DKV"], Wd["W_UKV"],
                                 Wd["W_KR"], H, dn, dr, dv)
    np.testing.assert_allclose(q.double().numpy(), qo, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(kc.double().numpy(), kco, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(kr.double().numpy(), kro, rtol=1e-4, atol=1e-5)
    # the values are the other half of the key/value projection, per head
    ckv = O.rms_norm(X.double().numpy() @ Wd["W_DKV"].T)
    vo = (ckv @ Wd["W_UKV"].T).reshape(B, S, H, dn + dv)[..., dn:]
    np.testing.assert_allclose(v.double().numpy(), vo, rtol=1e-4, atol=1e-5)
