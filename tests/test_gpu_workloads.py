"""Full-size GPU parity on the workloads of the pages' model, against the CPU
oracle on seeded samples (the oracle cannot run every full-size matrix or head
in seconds):

  dense_block   every matrix exactly; S_max and argmax of 4 of the 16 heads,
                the clip mask of all 16 (named heads clear tau by a wide margin)
  k2_mla_layer  all 6 MLA matrices exactly (W_O, 7168 x 8192, takes the fp64
                oracle ~30 s); S_max of 4 of the 64 heads (MLA keys: per-head
                k^C + shared k^R)
  moe_experts   the whole 128-matrix expert batch in one step, in the
                benchmark's launch configuration; 4 matrices exactly, among
                them the last of each 64-matrix shape
  long_mla      at 32768 tokens: S_max and argmax of 4 of the 64 heads, the
                clip mask of all 64, and the step with the clip on the layer's
                MLA matrices (W_UQ, W_UKV, W_DKV, W_KR exactly)

Tolerances are those of test_gpu_parity.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from muon_qk_clip_gb300 import build
from muon_qk_clip_gb300 import binding as mc
from muon_qk_clip_gb300 import forward, synth
from tests.gpu_helpers import assert_rounded_within, check_argmax, f64, rms, update_then_clip_band

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available()


def fp32(x):
    return float(np.float32(x))


def oracle_hp(hp):
    return O.Hparams(mu=fp32(hp.mu), lr=fp32(hp.lr), weight_decay=fp32(hp.weight_decay),
                     rms_scale=fp32(hp.rms_scale), ns_steps=hp.ns_steps,
                     ns_coeffs=tuple(fp32(c) for c in hp.ns_coeffs), ns_eps=fp32(hp.ns_eps))


def check_heads(smax, q, k, ks, heads, argmax=None):
    qh, kh = f64(q[:, :, heads]), f64(k[:, :, heads])
    ref, arg = O.max_logit(qh, kh, None if ks is None else f64(ks))
    np.testing.assert_allclose(f64(smax)[heads], ref, rtol=1e-3)
    if argmax is not None:
        check_argmax(argmax, q, k, ks, heads, ref, arg)
    return ref


def run_step(wl, seed, names=None):
    W, G, M = synth.muon_inputs(wl, seed=seed, device="cuda")
    names = names or [m.name for m in wl.matrices]
    W0 = {n: W[n].clone() for n in names}
    return W, G, M, W0, names


def test_dense_block_full_size():
    wl = synth.workload("dense_block")
    att = wl.attention
    W, G, M, W0, names = run_step(wl, seed=31)
    G0 = {n: G[n].cpu() for n in names}
    X = synth.normal((att.B, att.S, att.d_model), 1.0, "X", 31, torch.bfloat16, "cuda")
    q, k = forward.project_mha(X, W["Wq"], W["Wk"], att.H)
    q, k = q.contiguous(), k.contiguous()
    hp = mc.Hparams()
    arg = torch.empty(att.H, dtype=torch.int64, device="cuda")
    smax, _ = mc.qk_max_logit(q, k, argmax=arg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer = mc.ClipLayer(smax, mc.mha_segments(W["Wq"], W["Wk"], att.H))
    mc.muonclip_step([W[n] for n in names], [G[n] for n in names], [M[n] for n in names], hp,
                     layers=[layer], status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    heads = [0, 2, 7, 13]
    ref = check_heads(smax, q, k, None, heads, argmax=arg)
    s_all = f64(smax)
    named = sorted(att.scaled_heads)
    assert sorted(np.nonzero(s_all > 100.0)[0].tolist()) == named
    assert np.all(np.abs(s_all - 100.0) > 20.0)          # the mask has a wide margin
    gamma_all = np.where(s_all > 100.0, 100.0 / s_all, 1.0)
    s_rel = float(np.max(np.abs(s_all[heads] / ref - 1.0))) + 1e-7
    ohp = oracle_hp(hp)
    for n in names:
        Wn, _, Od = O.muon_step(f64(W0[n]), f64(G0[n]), np.zeros(W0[n].shape), ohp)
        tol = 2e-2 * rms(ohp.lr * Od)
        if n in ("Wq", "Wk"):
            factor = np.repeat(np.sqrt(gamma_all), att.d_head)
            lo, hi = update_then_clip_band(Wn, tol, factor, O.round_to_bf16, gamma_rel=s_rel)
            got = f64(W[n])
            assert np.all((got >= lo) & (got <= hi)), n
        else:
            assert_rounded_within(W[n], Wn, tol, n)


def test_k2_mla_layer_full_size():
    wl = synth.workload("k2_mla_layer")
    att = wl.attention
    W, G, M, W0, names = run_step(wl, seed=32)
    G0 = {n: G[n].cpu() for n in names}
    X, Wa = synth.attention_inputs(wl, seed=32, device="cuda")
    q, kc, kr = forward.project_mla(X, Wa, att.H)
    del X
    hp = mc.Hparams()
    smax, _ = mc.qk_max_logit(q, kc, kr)
    layer = mc.ClipLayer(smax, mc.mla_segments(W["W_UQ"], W["W_UKV"], att.H))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.muonclip_step([W[n] for n in names], [G[n] for n in names], [M[n] for n in names], hp,
                     layers=[layer], status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    heads = [0, 5, 17, 40]
    ref = check_heads(smax, q, kc, kr, heads)
    s_all = f64(smax)
    assert sorted(np.nonzero(s_all > 100.0)[0].tolist()) == sorted(att.scaled_heads)
    gamma_all = np.where(s_all > 100.0, 100.0 / s_all, 1.0)
    s_rel = float(np.max(np.abs(s_all[heads] / ref - 1.0))) + 1e-7
    ohp = oracle_hp(hp)
    dq, dkv = att.d_nope + att.d_rope, att.d_nope + att.d_v
    for n in names:
        Wn, _, Od = O.muon_step(f64(W0[n]), f64(G0[n]), np.zeros(W0[n].shape), ohp)
        tol = 2e-2 * rms(ohp.lr * Od)
        if n in ("W_UQ", "W_UKV"):
            f = np.ones(W0[n].shape[0])
            for h in range(att.H):
                if n == "W_UQ":
                    f[h * dq:h * dq + att.d_nope] = math.sqrt(gamma_all[h])
                    f[h * dq + att.d_nope:(h + 1) * dq] = gamma_all[h]
                else:
                    f[h * dkv:h * dkv + att.d_nope] = math.sqrt(gamma_all[h])
            lo, hi = update_then_clip_band(Wn, tol, f, O.round_to_bf16, gamma_rel=s_rel)
            got = f64(W[n])
            assert np.all((got >= lo) & (got <= hi)), n
        else:
            assert_rounded_within(W[n], Wn, tol, n)


def test_moe_expert_batch_full():
    """One muonclip_step over all 128 expert matrices (one shape group of 128
    after orientation, 19 GB of workspace), as the benchmark runs it."""
    wl = synth.workload("moe_experts")
    W, G, M = synth.muon_inputs(wl, seed=33, device="cuda")
    names = [m.name for m in wl.matrices]
    check = ("E0_up", "E63_up", "E17_down", "E63_down")
    W0 = {n: W[n].cpu() for n in check}
    G0 = {n: G[n].cpu() for n in check}
    hp = mc.Hparams()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.muonclip_step([W[n] for n in names], [G[n] for n in names], [M[n] for n in names], hp, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    del G
    ohp = oracle_hp(hp)
    for n in check:
        Wn, Mn, Od = O.muon_step(f64(W0[n]), f64(G0[n]), np.zeros(W0[n].shape), ohp)
        assert_rounded_within(M[n], Mn, 0.0, n + " momentum")
        assert_rounded_within(W[n], Wn, 2e-2 * rms(ohp.lr * Od), n)


def test_long_mla_full_step():
    """The 32768-token MLA layer: S_max (and argmax) from qk_max_logit, then
    one muonclip_step over the layer's six matrices with the clip of the
    heads over tau; the oracle checks 4 heads' S_max and argmax, the mask of
    all 64 heads, and W_UQ, W_UKV (clipped rows), W_DKV and W_KR."""
    wl = synth.workload("long_mla")
    att = wl.attention
    W, G, M, W0, names = run_step(wl, seed=34)
    check = ("W_UQ", "W_UKV", "W_DKV", "W_KR")
    W0 = {n: W0[n].cpu() for n in check}
    G0 = {n: G[n].cpu() for n in check}
    X, Wa = synth.attention_inputs(wl, seed=34, device="cuda")
    q, kc, kr = forward.project_mla(X, Wa, att.H)
    del X, Wa
    arg = torch.empty(att.H, dtype=torch.int64, device="cuda")
    smax, _ = mc.qk_max_logit(q, kc, kr, argmax=arg)
    hp = mc.Hparams()
    ncl = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer = mc.ClipLayer(smax, mc.mla_segments(W["W_UQ"], W["W_UKV"], att.H), nclipped=ncl)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.muonclip_step([W[n] for n in names], [G[n] for n in names], [M[n] for n in names], hp,
                     layers=[layer], status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    del G, M
    s_all = f64(smax)
    named = sorted(att.scaled_heads)
    assert sorted(np.nonzero(s_all > 100.0)[0].tolist()) == named and ncl.item() == len(named)
    assert np.all(np.abs(s_all - 100.0) > 20.0)          # the mask has a wide margin
    heads = [0, 3, 11, 40]                                # 3 and 11 are over tau
    ref = check_heads(smax, q, kc, kr, heads, argmax=arg)
    del q, kc, kr
    gamma_all = np.where(s_all > 100.0, 100.0 / s_all, 1.0)
    s_rel = float(np.max(np.abs(s_all[heads] / ref - 1.0))) + 1e-7
    ohp = oracle_hp(hp)
    dq, dkv = att.d_nope + att.d_rope, att.d_nope + att.d_v
    for n in check:
        Wn, _, Od = O.muon_step(f64(W0[n]), f64(G0[n]), np.zeros(W0[n].shape), ohp)
        tol = 2e-2 * rms(ohp.lr * Od)
        if n in ("W_UQ", "W_UKV"):
            f = np.ones(W0[n].shape[0])
            for h in range(att.H):
                if n == "W_UQ":
                    f[h * dq:h * dq + att.d_nope] = math.sqrt(gamma_all[h])
                    f[h * dq + att.d_nope:(h + 1) * dq] = gamma_all[h]
                else:
                    f[h * dkv:h * dkv + att.d_nope] = math.sqrt(gamma_all[h])
            lo, hi = update_then_clip_band(Wn, tol, f, O.round_to_bf16, gamma_rel=s_rel)
            got = f64(W[n])
            assert np.all((got >= lo) & (got <= hi)), n
        else:
            assert_rounded_within(W[n], Wn, tol, n)
