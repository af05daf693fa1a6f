"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Tolerances (floating point; each derived from the arithmetic of its path):
  * momentum:                 within 1 fp32 rounding of the exact mu*M + G
  * Newton-Schulz, split bf16: |O - O_exact| <= 2e-2 * RMS(O_exact) before the
                               output rounding (the bound stated for the
                               bf16 tensor-core path)
  * Newton-Schulz, fp32:      1e-5 * RMS(O_exact)
  * Newton-Schulz, bf16:      2.5e-1 * RMS max, 2.5e-2 * RMS root-mean-square
  * updated weights:          |W - W_exact| <= tol * RMS(lr O) before the final
                               rounding to the weight dtype
  * S_max:                    relative 1e-3 (bf16 features), 1e-5 (fp32)
  * clip mask / argmax:       exact (argmax where the oracle's top-2 gap is
                               clear of the fp32 accumulation error)
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from muon_qk_clip_gb300 import abi, build
from muon_qk_clip_gb300 import binding as mc
from muon_qk_clip_gb300 import forward, synth
from tests.gpu_helpers import assert_rounded_within, f64, padded, rms, update_then_clip_band

pytestmark = pytest.mark.gpu

F32, BF16 = torch.float32, torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    abi.load()


def fp32(x):
    return float(np.float32(x))


def new_status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------------ momentum
@pytest.mark.parametrize("shapes", [[(64, 64)], [(100, 77), (3, 5)], [(300, 1000), (1000, 300)]])
@pytest.mark.parametrize("gdtype", [F32, BF16])
def test_momentum_parity(shapes, gdtype):
    mu = 0.95
    Ms, Gs, ref = [], [], []
    for i, (r, c) in enumerate(shapes):
        M0 = synth.normal((r, c), 1.0, f"m{i}", 1)
        G0 = synth.normal((r, c), 0.5, f"g{i}", 1).to(gdtype)
        M = padded(r, c, F32); M.copy_(M0)
        G = padded(r, c, gdtype); G.copy_(G0)
        Ms.append(M); Gs.append(G)
        ref.append(O.momentum(f64(M0), f64(G0), fp32(mu)))
    st = new_status()
    mc.muon_momentum(Ms, Gs, mu, status=st)
    torch.cuda.synchronize()
    for M, want in zip(Ms, ref):
        assert_rounded_within(M, want, 0.0, "momentum")
    assert st.item() == 0


def test_momentum_flags_nonfinite():
    M = torch.zeros(64, 64, device="cuda")
    G = torch.zeros(64, 64, device="cuda")
    G[3, 5] = float("nan")
    st = new_status()
    mc.muon_momentum([M], [G], 0.9, status=st)
    torch.cuda.synchronize()
    assert st.item() & abi.MC_STATUS_NONFINITE_UPDATE


# ------------------------------------------------------------------ Newton-Schulz
NS_CASES = {
    "single": [(256, 512)],
    "transposed": [(384, 256)],
    "ragged_groups": [(200, 328), (328, 200), (64, 1000)],
    "batched": [(512, 512), (512, 512), (512, 512), (256, 768)],
    "tall_thin": [(1000, 64)],
    "large": [(1024, 1536)],
}


def run_ns(shapes, precision, out_dtype, steps=5, seed=0, fast_steps=3):
    Ms, Os, ref = [], [], []
    hp = mc.Hparams(ns_precision=precision, ns_steps=steps, ns_fast_steps=fast_steps)
    ohp = O.Hparams(ns_steps=steps, ns_coeffs=tuple(fp32(c) for c in hp.ns_coeffs),
                    ns_eps=fp32(hp.ns_eps), rms_scale=fp32(hp.rms_scale))
    for i, (r, c) in enumerate(shapes):
        M0 = synth.ns_test_matrix(r, c, seed, f"ns{i}")
        M = M0.cuda()
        Ms.append(M)
        Os.append(torch.full((r, c), float("nan"), dtype=out_dtype, device="cuda"))
        ref.append(O.muon_direction(f64(M0), ohp))
    st = new_status()
    mc.muon_newton_schulz(Ms, Os, hp, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return Os, ref


@pytest.mark.parametrize("case", list(NS_CASES))
@pytest.mark.parametrize("out_dtype", [F32, BF16])
def test_ns_split_bf16_parity(case, out_dtype):
    Os, ref = run_ns(NS_CASES[case], abi.MC_NS_SPLIT_BF16, out_dtype)
    for o, want in zip(Os, ref):
        assert_rounded_within(o, want, 2e-2 * rms(want), f"NS split {case}")


@pytest.mark.parametrize("fast_steps", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("case", ["batched", "ragged_groups", "large"])
def test_ns_split_fast_steps(case, fast_steps):
    """Leading iterations with one product (hi operands) per k-step: every
    setting stays in tolerance.  Every matrix of smaller side 256 or more
    takes up to three (4 acts as 3); the ragged groups' matrices (smaller side
    under 256) keep three products throughout."""
    Os, ref = run_ns(NS_CASES[case], abi.MC_NS_SPLIT_BF16, F32, fast_steps=fast_steps)
    for o, want in zip(Os, ref):
        assert_rounded_within(o, want, 2e-2 * rms(want), f"NS fast={fast_steps} {case}")


@pytest.mark.parametrize("case", ["single", "transposed", "ragged_groups"])
def test_ns_fp32_parity(case):
    Os, ref = run_ns(NS_CASES[case], abi.MC_NS_FP32, F32)
    for o, want in zip(Os, ref):
        assert_rounded_within(o, want, 1e-5 * rms(want), f"NS fp32 {case}")


@pytest.mark.parametrize("case", ["single", "ragged_groups"])
def test_ns_bf16_parity(case):
    Os, ref = run_ns(NS_CASES[case], abi.MC_NS_BF16, F32)
    for o, want in zip(Os, ref):
        err = f64(o) - want
        assert np.abs(err).max() <= 0.25 * rms(want)
        assert rms(err) <= 2.5e-2 * rms(want)


@pytest.mark.parametrize("steps", [0, 1, 2])
def test_ns_few_steps(steps):
    Os, ref = run_ns([(128, 320), (320, 128)], abi.MC_NS_SPLIT_BF16, F32, steps=steps)
    for o, want in zip(Os, ref):
        assert_rounded_within(o, want, 2e-2 * rms(want), f"NS {steps} steps")


def test_ns_zero_matrix():
    M = torch.zeros(128, 256, device="cuda")
    Ot = torch.full((128, 256), float("nan"), device="cuda")
    mc.muon_newton_schulz([M], [Ot])
    torch.cuda.synchronize()
    assert torch.count_nonzero(Ot).item() == 0


# ------------------------------------------------------------------ full Muon step
def oracle_muon(W, G, M, hp):
    ohp = O.Hparams(mu=fp32(hp.mu), lr=fp32(hp.lr), weight_decay=fp32(hp.weight_decay),
                    rms_scale=fp32(hp.rms_scale), ns_steps=hp.ns_steps,
                    ns_coeffs=tuple(fp32(c) for c in hp.ns_coeffs), ns_eps=fp32(hp.ns_eps),
                    scale_mode="spectral" if hp.scale_mode == abi.MC_SCALE_SPECTRAL else "rms")
    return O.muon_step(f64(W), f64(G), f64(M), ohp), ohp


@pytest.mark.parametrize("wdtype,precision,tol", [(F32, abi.MC_NS_FP32, 1e-5),
                                                  (BF16, abi.MC_NS_SPLIT_BF16, 2e-2)])
@pytest.mark.parametrize("warm", [False, True])
def test_muon_step_parity(wdtype, precision, tol, warm):
    shapes = [(256, 512), (384, 128), (96, 96)]
    hp = mc.Hparams(ns_precision=precision)
    W, G, M, want = [], [], [], []
    for i, (r, c) in enumerate(shapes):
        w = synth.normal((r, c), 0.02, f"w{i}", 3).to(wdtype)
        g = synth.normal((r, c), 1.0, f"g{i}", 3)
        m = synth.normal((r, c), 3.0, f"m{i}", 3) if warm else torch.zeros(r, c)
        (Wn, Mn, Od), _ = oracle_muon(w, g, m, hp)
        want.append((Wn, Mn, Od))
        W.append(w.cuda()); G.append(g.cuda()); M.append(m.cuda())
    st = new_status()
    mc.muonclip_step(W, G, M, hp, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for (Wn, Mn, Od), w, m in zip(want, W, M):
        assert_rounded_within(m, Mn, 0.0, "momentum state")
        assert_rounded_within(w, Wn, tol * rms(fp32(hp.lr) * Od), "updated W")


@pytest.mark.parametrize("wdtype,precision,tol", [(F32, abi.MC_NS_FP32, 1e-5),
                                                  (BF16, abi.MC_NS_SPLIT_BF16, 2e-2)])
def test_muon_step_spectral_scale(wdtype, precision, tol):
    """The MuP-style update scale sqrt(max(1, out/in)): tall, wide and square
    weights in one call (factor 3, 1 and 1)."""
    shapes = [(576, 64), (128, 320), (96, 96)]
    hp = mc.Hparams(ns_precision=precision, scale_mode=abi.MC_SCALE_SPECTRAL)
    W, G, M, want = [], [], [], []
    for i, (r, c) in enumerate(shapes):
        w = synth.normal((r, c), 0.02, f"sw{i}", 13).to(wdtype)
        g = synth.normal((r, c), 1.0, f"sg{i}", 13)
        m = synth.normal((r, c), 2.0, f"sm{i}", 13)
        (Wn, Mn, Od), ohp = oracle_muon(w, g, m, hp)
        assert ohp.scale_mode == "spectral"
        want.append((Wn, Od))
        W.append(w.cuda()); G.append(g.cuda()); M.append(m.cuda())
    st = new_status()
    mc.muonclip_step(W, G, M, hp, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for (Wn, Od), w in zip(want, W):
        assert_rounded_within(w, Wn, tol * rms(fp32(hp.lr) * Od), "updated W")


def test_step_is_deterministic_and_resumable():
    """Two runs from the same state are bit-identical; a step taken after
    saving and reloading (M, W) equals the uninterrupted second step."""
    hp = mc.Hparams()
    shapes = [(256, 384), (384, 256)]
    base = [(synth.normal(s, 0.02, f"w{i}", 4).to(BF16), synth.normal(s, 1.0, f"g{i}", 4))
            for i, s in enumerate(shapes)]
    G2 = [synth.normal(s, 1.0, f"h{i}", 4).cuda() for i, s in enumerate(shapes)]

    def run(two_steps, reload=False):
        W = [w.cuda() for w, _ in base]
        G = [g.cuda() for _, g in base]
        M = [torch.zeros(s, device="cuda") for s in shapes]
        mc.muonclip_step(W, G, M, hp)
        if reload:
            W = [w.cpu().cuda() for w in W]
            M = [m.cpu().cuda() for m in M]
        if two_steps:
            mc.muonclip_step(W, G2, M, hp)
        torch.cuda.synchronize()
        return W, M

    a, b = run(True), run(True)
    c = run(True, reload=True)
    for x, y, z in zip(a[0] + a[1], b[0] + b[1], c[0] + c[1]):
        assert torch.equal(x, y) and torch.equal(x, z)


# ------------------------------------------------------------------ max logit
ML_CASES = {
    "tiny_fp32": dict(B=2, S=128, H=4, dk=64, dr=0, dtype=F32, causal=True),
    "ragged_bf16": dict(B=1, S=200, H=3, dk=128, dr=0, dtype=BF16, causal=True),
    "mla_bf16": dict(B=2, S=129, H=2, dk=128, dr=64, dtype=BF16, causal=True),
    "noncausal": dict(B=1, S=96, H=2, dk=64, dr=0, dtype=BF16, causal=False),
    "single_token": dict(B=3, S=1, H=2, dk=64, dr=0, dtype=BF16, causal=True),
    "fp32_mla": dict(B=1, S=70, H=2, dk=32, dr=16, dtype=F32, causal=True),
}


def check_smax(s_gpu, arg_gpu, q, k, ks, causal, dtype):
    ref, arg = O.max_logit(f64(q), f64(k), None if ks is None else f64(ks), causal=causal)
    S = q.shape[1]
    rel = 1e-5 if dtype == F32 else 1e-3
    np.testing.assert_allclose(f64(s_gpu), ref, rtol=rel, atol=0)
    if arg_gpu is not None:
        # compare the argmax where the oracle's best beats every other pair by
        # more than the fp32 accumulation error
        got = arg_gpu.cpu().numpy()
        for h in range(q.shape[2]):
            b, i, j = arg[h]
            flat = (b * S + i) * S + j
            if got[h] != flat:
                gb, rem = divmod(int(got[h]), S * S)
                gi, gj = divmod(rem, S)
                kv = np.concatenate([f64(k)[gb, gj, h]] + ([f64(ks)[gb, gj]] if ks is not None else []))
                other = float(f64(q)[gb, gi, h] @ kv) / math.sqrt(q.shape[-1])
                assert abs(other - ref[h]) <= 2e-6 * abs(ref[h]) + 1e-6, (h, got[h], flat)


@pytest.mark.parametrize("case", list(ML_CASES))
@pytest.mark.parametrize("with_argmax", [False, True])
def test_max_logit_parity(case, with_argmax):
    c = ML_CASES[case]
    q, k, ks = synth.attention_features(c["B"], c["S"], c["H"], c["dk"] + c["dr"], c["dk"],
                                        c["dr"], c["dtype"], seed=5, key=case)
    qd, kd = q.cuda(), k.cuda()
    ksd = None if ks is None else ks.cuda()
    arg = torch.empty(c["H"], dtype=torch.int64, device="cuda") if with_argmax else None
    st = new_status()
    s, a = mc.qk_max_logit(qd, kd, ksd, causal=c["causal"], argmax=arg, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_smax(s, a, q, k, ks, c["causal"], c["dtype"])


def test_max_logit_strided_mla_views():
    """K^C as a strided view into the [k^C || v] projection, shared K^R."""
    wl = synth.scaled(synth.workload("k2_mla_layer"), S=80)
    X, W = synth.attention_inputs(wl, seed=2, device="cuda")
    q, kc, kr = forward.project_mla(X, W, wl.attention.H)
    q, kc = q[:, :, :6], kc[:, :, :6]
    # device K^C keeps the projection's layout: a view with head stride 256
    kv_d = torch.zeros(kc.shape[:3] + (256,), dtype=kc.dtype, device="cuda")
    kc_d = kv_d[..., :128]
    kc_d.copy_(kc)
    assert kc_d.stride(2) == 256
    s, a = mc.qk_max_logit(q.cuda(), kc_d, kr.cuda(),
                           argmax=torch.empty(6, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    check_smax(s, a, q, kc, kr, True, BF16)


def test_max_logit_accumulate_over_microbatches():
    q, k, _ = synth.attention_features(4, 64, 3, 64, 64, 0, BF16, seed=6)
    qd, kd = q.cuda(), k.cuda()
    full, _ = mc.qk_max_logit(qd, kd)
    part, _ = mc.qk_max_logit(qd[:2], kd[:2])
    mc.qk_max_logit(qd[2:], kd[2:], smax=part, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(full, part)


def test_max_logit_negative_and_mixed_sign_accumulate():
    """S_max is max-combined in place as a float: a micro-batch whose logits
    are all negative (every q feature positive, every k feature negative),
    then one whose heads 0 and 1 turn positive while heads 2 and 3 stay
    negative.  Each result equals the oracle's maximum over the batches seen,
    on the tensor-core path and through the attention forward."""
    B, S, H, d = 2, 160, 4, 64
    qa, ka, _ = synth.attention_features(B, S, H, d, d, 0, BF16, seed=23)
    qb, kb, _ = synth.attention_features(B, S, H, d, d, 0, BF16, seed=24)
    qa, ka = qa.abs(), -ka.abs()
    qb, kb = qb.abs(), kb.abs()
    kb[:, :, 2:] = -kb[:, :, 2:]
    ra, _ = O.max_logit(f64(qa), f64(ka))
    rb, _ = O.max_logit(f64(qb), f64(kb))
    assert np.all(ra < 0) and np.all(rb[:2] > 0) and np.all(rb[2:] < 0)
    v = torch.zeros(B, S, H, d, dtype=BF16, device="cuda")
    for run in ("max_logit", "attention"):
        if run == "max_logit":
            s, _ = mc.qk_max_logit(qa.cuda(), ka.cuda())
        else:
            _, _, s = mc.qk_attention_forward(qa.cuda(), ka.cuda(), v)
        torch.cuda.synchronize()
        np.testing.assert_allclose(f64(s), ra, rtol=1e-3)
        if run == "max_logit":
            mc.qk_max_logit(qb.cuda(), kb.cuda(), smax=s, accumulate=True)
        else:
            mc.qk_attention_forward(qb.cuda(), kb.cuda(), v, smax=s, accumulate=True)
        torch.cuda.synchronize()
        np.testing.assert_allclose(f64(s), np.maximum(ra, rb), rtol=1e-3)


def test_max_logit_flags_nonfinite():
    q, k, _ = synth.attention_features(1, 32, 2, 64, 64, 0, BF16, seed=7)
    q[0, 5, 1, 3] = float("inf")
    st = new_status()
    mc.qk_max_logit(q.cuda(), k.cuda(), status=st)
    torch.cuda.synchronize()
    assert st.item() & abi.MC_STATUS_NONFINITE_LOGIT


@pytest.mark.parametrize("kind", ["+inf", "-inf", "nan"])
def test_max_logit_flags_each_nonfinite_kind(kind):
    """One query row whose logits are all +inf, all -inf or all NaN (one
    feature of q is non-finite, that feature of k is positive, the rest of the
    row is zero); every other logit is finite.  Each kind must set the flag on
    its own, on the tensor-core path (bf16, d 64) and with argmax."""
    B, S, H, d = 2, 300, 3, 64
    q, k, _ = synth.attention_features(B, S, H, d, d, 0, BF16, seed=17)
    k[:, :, 1, 7] = k[:, :, 1, 7].abs() + 0.5
    q[1, 211, 1, :] = 0
    q[1, 211, 1, 7] = {"+inf": float("inf"), "-inf": float("-inf"), "nan": float("nan")}[kind]
    for argmax in (None, torch.empty(H, dtype=torch.int64, device="cuda")):
        st = new_status()
        mc.qk_max_logit(q.cuda(), k.cuda(), status=st, argmax=argmax)
        torch.cuda.synchronize()
        assert st.item() & abi.MC_STATUS_NONFINITE_LOGIT, (kind, argmax is not None)
    st = new_status()
    q[1, 211, 1, 7] = 1.0
    mc.qk_max_logit(q.cuda(), k.cuda(), status=st)
    torch.cuda.synchronize()
    assert st.item() == 0


# ------------------------------------------------------------------ QK-Clip
def test_clip_mha_parity_and_untouched_heads():
    H, d, D, tau = 8, 16, 40, 100.0
    Wq = synth.normal((H * d, D), 1.0, "cq", 8).to(BF16)
    Wk = synth.normal((H * d, D), 1.0, "ck", 8).to(BF16)
    smax = torch.tensor([50.0, 100.0, 150.0, 400.0, 0.0, -3.0, 101.0, 1e4])
    Wq_d, Wk_d, s_d = Wq.cuda(), Wk.cuda(), smax.cuda()
    gamma = torch.empty(H, device="cuda")
    ncl = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.qk_clip_apply(s_d, tau, mc.mha_segments(Wq_d, Wk_d, H, 0.5), gamma_out=gamma, nclipped=ncl)
    torch.cuda.synchronize()
    out, g, mask = O.qk_clip({"Wq": f64(Wq), "Wk": f64(Wk)}, O.mha_segments(H, d, 0.5),
                             f64(smax), tau)
    assert ncl.item() == int(mask.sum()) == 4
    np.testing.assert_allclose(f64(gamma), g, rtol=1e-6)
    for name, dev, src in (("Wq", Wq_d, Wq), ("Wk", Wk_d, Wk)):
        for h in range(H):
            rows = slice(h * d, (h + 1) * d)
            if not mask[h]:
                assert torch.equal(dev[rows].cpu(), src[rows]), f"{name} head {h} changed"
        assert_rounded_within(dev, out[name], 1e-6 * np.abs(out[name]), f"clip {name}")


def test_clip_mla_parity_shared_key_untouched():
    H, dn, dr, dv, ql, kl, tau = 4, 16, 8, 16, 24, 16, 100.0
    W_UQ = synth.normal((H * (dn + dr), ql), 1.0, "uq", 9).to(BF16)
    W_UKV = synth.normal((H * (dn + dv), kl), 1.0, "ukv", 9).to(BF16)
    W_KR = synth.normal((dr, 40), 1.0, "kr", 9).to(BF16)
    smax = torch.tensor([300.0, 20.0, 100.5, 99.0])
    d_uq, d_ukv, d_kr = W_UQ.cuda(), W_UKV.cuda(), W_KR.cuda()
    mc.qk_clip_apply(smax.cuda(), tau, mc.mla_segments(d_uq, d_ukv, H, dn, dr, dv))
    torch.cuda.synchronize()
    out, g, mask = O.qk_clip({"W_UQ": f64(W_UQ), "W_UKV": f64(W_UKV)},
                             O.mla_segments(H, dn, dr, dv), f64(smax), tau)
    assert_rounded_within(d_uq, out["W_UQ"], 1e-6 * np.abs(out["W_UQ"]), "W_UQ")
    assert_rounded_within(d_ukv, out["W_UKV"], 1e-6 * np.abs(out["W_UKV"]), "W_UKV")
    assert torch.equal(d_kr.cpu(), W_KR)
    for h in range(H):
        v = slice(h * (dn + dv) + dn, (h + 1) * (dn + dv))
        assert torch.equal(d_ukv[v].cpu(), W_UKV[v])


def test_clip_fp32_alpha_split():
    H, d, D = 4, 8, 12
    Wq = synth.normal((H * d, D), 1.0, "fq", 10)
    Wk = synth.normal((H * d, D), 1.0, "fk", 10)
    smax = torch.tensor([1000.0, 10.0, 250.0, 90.0])
    dq, dk = Wq.cuda(), Wk.cuda()
    mc.qk_clip_apply(smax.cuda(), 100.0, mc.mha_segments(dq, dk, H, 0.25))
    torch.cuda.synchronize()
    out, _, _ = O.qk_clip({"Wq": f64(Wq), "Wk": f64(Wk)}, O.mha_segments(H, d, 0.25),
                          f64(smax), 100.0)
    assert_rounded_within(dq, out["Wq"], 1e-6 * np.abs(out["Wq"]), "Wq")
    assert_rounded_within(dk, out["Wk"], 1e-6 * np.abs(out["Wk"]), "Wk")


def test_clip_nan_smax_flags_and_leaves_weights():
    H, d = 2, 8
    Wq = synth.normal((H * d, 16), 1.0, "nq", 11).to(BF16).cuda()
    Wk = synth.normal((H * d, 16), 1.0, "nk", 11).to(BF16).cuda()
    before = (Wq.clone(), Wk.clone())
    st = new_status()
    mc.qk_clip_apply(torch.tensor([float("nan"), 5.0], device="cuda"), 100.0,
                     mc.mha_segments(Wq, Wk, H), status=st)
    torch.cuda.synchronize()
    assert st.item() & abi.MC_STATUS_NONFINITE_SMAX
    assert torch.equal(Wq, before[0]) and torch.equal(Wk, before[1])


@pytest.mark.parametrize("smax_vals,clipped", [([50.0, 100.0, 150.0, 400.0], True),
                                               ([50.0, 99.0, 100.0, -1.0], False)])
def test_clip_total_mode_parity(smax_vals, clipped):
    """Total clip: one gamma = tau / max_h S_max^h on every head's rows."""
    H, d, D, tau = 4, 16, 40, 100.0
    Wq = synth.normal((H * d, D), 1.0, "tq", 14).to(BF16)
    Wk = synth.normal((H * d, D), 1.0, "tk", 14).to(BF16)
    smax = torch.tensor(smax_vals)
    dq, dk = Wq.cuda(), Wk.cuda()
    gamma = torch.empty(H, device="cuda")
    ncl = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.qk_clip_apply(smax.cuda(), tau, mc.mha_segments(dq, dk, H, 0.5), gamma_out=gamma,
                     nclipped=ncl, mode=abi.MC_CLIP_TOTAL)
    torch.cuda.synchronize()
    out, g = O.qk_clip_total({"Wq": f64(Wq), "Wk": f64(Wk)}, O.mha_segments(H, d, 0.5),
                             f64(smax), tau)
    assert (g < 1.0) == clipped
    assert ncl.item() == (H if clipped else 0)
    np.testing.assert_allclose(f64(gamma), np.full(H, g), rtol=1e-6)
    if clipped:
        assert_rounded_within(dq, out["Wq"], 1e-6 * np.abs(out["Wq"]), "Wq")
        assert_rounded_within(dk, out["Wk"], 1e-6 * np.abs(out["Wk"]), "Wk")
    else:
        assert torch.equal(dq.cpu(), Wq) and torch.equal(dk.cpu(), Wk)


def test_clip_total_mode_mla_in_step():
    """Total clip of an MLA layer inside muonclip_step (beside one unrelated
    Muon matrix): q^C and k^C by sqrt(gamma), q^R by gamma, v rows untouched."""
    H, dn, dr, dv, ql, kl, tau = 4, 16, 8, 16, 24, 16, 100.0
    W_UQ = synth.normal((H * (dn + dr), ql), 1.0, "tuq", 15).to(BF16)
    W_UKV = synth.normal((H * (dn + dv), kl), 1.0, "tukv", 15).to(BF16)
    smax = torch.tensor([30.0, 250.0, 99.0, 120.0])
    d_uq, d_ukv = W_UQ.cuda(), W_UKV.cuda()
    layer = mc.ClipLayer(smax.cuda(), mc.mla_segments(d_uq, d_ukv, H, dn, dr, dv),
                         mode=abi.MC_CLIP_TOTAL)
    w = synth.normal((64, 96), 0.02, "tw", 15).to(BF16).cuda()
    mc.muonclip_step([w], [torch.ones(64, 96, device="cuda")], [torch.zeros(64, 96, device="cuda")],
                     mc.Hparams(), layers=[layer])
    torch.cuda.synchronize()
    out, g = O.qk_clip_total({"W_UQ": f64(W_UQ), "W_UKV": f64(W_UKV)},
                             O.mla_segments(H, dn, dr, dv), f64(smax), tau)
    assert g == pytest.approx(0.4)
    assert_rounded_within(d_uq, out["W_UQ"], 1e-6 * np.abs(out["W_UQ"]), "W_UQ")
    assert_rounded_within(d_ukv, out["W_UKV"], 1e-6 * np.abs(out["W_UKV"]), "W_UKV")
    for h in range(H):
        v = slice(h * (dn + dv) + dn, (h + 1) * (dn + dv))
        assert torch.equal(d_ukv[v].cpu(), W_UKV[v])


def test_clip_total_mode_nan_clips_nothing():
    H, d = 3, 8
    Wq = synth.normal((H * d, 16), 1.0, "tnq", 16).to(BF16).cuda()
    Wk = synth.normal((H * d, 16), 1.0, "tnk", 16).to(BF16).cuda()
    before = (Wq.clone(), Wk.clone())
    st = new_status()
    gamma = torch.empty(H, device="cuda")
    mc.qk_clip_apply(torch.tensor([500.0, float("nan"), 5.0], device="cuda"), 100.0,
                     mc.mha_segments(Wq, Wk, H), gamma_out=gamma, status=st,
                     mode=abi.MC_CLIP_TOTAL)
    torch.cuda.synchronize()
    assert st.item() & abi.MC_STATUS_NONFINITE_SMAX
    assert torch.equal(Wq, before[0]) and torch.equal(Wk, before[1])
    assert torch.equal(gamma.cpu(), torch.ones(H))


@pytest.mark.parametrize("kind", ["mha", "mla"])
def test_clip_tau30(kind):
    """The threshold of the pages' small-model ablation, tau = 30: heads
    between 30 and 100 clip (at tau = 100 they would not), a head at exactly
    30 does not, and the factor is gamma = 30 / S_max."""
    tau = 30.0
    if kind == "mha":
        H, d, D = 8, 16, 40
        Wq = synth.normal((H * d, D), 1.0, "t30q", 17).to(BF16)
        Wk = synth.normal((H * d, D), 1.0, "t30k", 17).to(BF16)
        smax = torch.tensor([10.0, 30.0, 31.0, 45.0, 99.0, 150.0, 29.9, 1000.0])
        w = {"Wq": Wq, "Wk": Wk}
        dev = {n: t.cuda() for n, t in w.items()}
        segs, osegs = mc.mha_segments(dev["Wq"], dev["Wk"], H, 0.5), O.mha_segments(H, d, 0.5)
        want = [False, False, True, True, True, True, False, True]
    else:
        H, dn, dr, dv, ql, kl = 4, 16, 8, 16, 24, 16
        W_UQ = synth.normal((H * (dn + dr), ql), 1.0, "t30uq", 17).to(BF16)
        W_UKV = synth.normal((H * (dn + dv), kl), 1.0, "t30ukv", 17).to(BF16)
        smax = torch.tensor([30.5, 29.0, 80.0, 300.0])
        w = {"W_UQ": W_UQ, "W_UKV": W_UKV}
        dev = {n: t.cuda() for n, t in w.items()}
        segs, osegs = mc.mla_segments(dev["W_UQ"], dev["W_UKV"], H, dn, dr, dv), O.mla_segments(H, dn, dr, dv)
        want = [True, False, True, True]
    gamma = torch.empty(H, device="cuda")
    ncl = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.qk_clip_apply(smax.cuda(), tau, segs, gamma_out=gamma, nclipped=ncl)
    torch.cuda.synchronize()
    out, g, mask = O.qk_clip({n: f64(t) for n, t in w.items()}, osegs, f64(smax), tau)
    assert mask.tolist() == want and ncl.item() == sum(want)
    np.testing.assert_allclose(f64(gamma), g, rtol=1e-6)
    for n in w:
        assert_rounded_within(dev[n], out[n], 1e-6 * np.abs(out[n]), f"tau 30 {kind} {n}")


# ------------------------------------------------------------------ MuonClip step, tiny MHA
def test_tiny_mha_fp32_full_step():
    """The tiny fp32 MHA workload end to end: S_max from the forward features,
    Muon on the 256x512 matrix, then QK-Clip of heads 1 and 3."""
    wl = synth.workload("tiny_mha_fp32")
    X, Wa = synth.attention_inputs(wl)
    Wm, Gm, Mm = synth.muon_inputs(wl)
    q, k = forward.project_mha(X.cuda(), Wa["Wq"].cuda(), Wa["Wk"].cuda(), wl.attention.H)
    hp = mc.Hparams()
    smax, _ = mc.qk_max_logit(q.cuda(), k.cuda())
    ref_s, _ = O.max_logit(f64(q), f64(k))
    np.testing.assert_allclose(f64(smax), ref_s, rtol=1e-5)
    assert list(ref_s > 100.0) == [False, True, False, True]
    W, G, M = [Wm["W"].cuda()], [Gm["W"].cuda()], [Mm["W"].cuda()]
    Wq, Wk = Wa["Wq"].cuda(), Wa["Wk"].cuda()
    layer = mc.ClipLayer(smax, mc.mha_segments(Wq, Wk, wl.attention.H))
    mc.muonclip_step(W, G, M, hp, layers=[layer])
    torch.cuda.synchronize()
    (Wn, _, Od), _ = oracle_muon(Wm["W"], Gm["W"], Mm["W"], hp)
    assert_rounded_within(W[0], Wn, 1e-5 * rms(fp32(hp.lr) * Od), "tiny W")
    out, _, mask = O.qk_clip({"Wq": f64(Wa["Wq"]), "Wk": f64(Wa["Wk"])},
                             O.mha_segments(4, 64), ref_s, 100.0)
    assert_rounded_within(Wq, out["Wq"], 1e-6 * np.abs(out["Wq"]), "Wq")
    assert_rounded_within(Wk, out["Wk"], 1e-6 * np.abs(out["Wk"]), "Wk")
    # re-measured max logit after the clip is min(S, tau)
    # on the library: the projection with the clipped weights, then S_max
    q2, k2 = forward.project_mha(X.cuda(), Wq, Wk, 4)
    s2, _ = mc.qk_max_logit(q2, k2)
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(s2), np.minimum(ref_s, 100.0), rtol=1e-5)


def test_tiny_mha_step_tau30():
    """The tiny fp32 MHA workload with heads 1 and 3 scaled x12 (max logit
    ~67) stepped with tau = 30: both heads clip, which tau = 100 would not,
    and the re-measured max logit after the step's clip is min(S, 30)."""
    wl = synth.scaled(synth.workload("tiny_mha_fp32", "literal"), scaled_heads={1: 12.0, 3: 12.0})
    X, Wa = synth.attention_inputs(wl, seed=5)
    Wm, Gm, Mm = synth.muon_inputs(wl, seed=5)
    q, k = forward.project_mha(X.cuda(), Wa["Wq"].cuda(), Wa["Wk"].cuda(), wl.attention.H)
    hp = mc.Hparams(tau=30.0)
    smax, _ = mc.qk_max_logit(q.cuda(), k.cuda())
    ref_s, _ = O.max_logit(f64(q), f64(k))
    np.testing.assert_allclose(f64(smax), ref_s, rtol=1e-5)
    assert list(ref_s > 30.0) == [False, True, False, True]
    assert np.all(ref_s < 100.0) and np.all(np.abs(ref_s - 30.0) > 5.0)
    W, G, M = [Wm["W"].cuda()], [Gm["W"].cuda()], [Mm["W"].cuda()]
    Wq, Wk = Wa["Wq"].cuda(), Wa["Wk"].cuda()
    ncl = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer = mc.ClipLayer(smax, mc.mha_segments(Wq, Wk, wl.attention.H), nclipped=ncl)
    mc.muonclip_step(W, G, M, hp, layers=[layer])
    torch.cuda.synchronize()
    assert ncl.item() == 2
    (Wn, _, Od), _ = oracle_muon(Wm["W"], Gm["W"], Mm["W"], hp)
    assert_rounded_within(W[0], Wn, 1e-5 * rms(fp32(hp.lr) * Od), "tiny W")
    out, _, mask = O.qk_clip({"Wq": f64(Wa["Wq"]), "Wk": f64(Wa["Wk"])},
                             O.mha_segments(4, 64), ref_s, 30.0)
    assert_rounded_within(Wq, out["Wq"], 1e-6 * np.abs(out["Wq"]), "Wq")
    assert_rounded_within(Wk, out["Wk"], 1e-6 * np.abs(out["Wk"]), "Wk")
    q2, k2 = forward.project_mha(X.cuda(), Wq, Wk, 4)
    s2, _ = mc.qk_max_logit(q2, k2)
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(s2), np.minimum(ref_s, 30.0), rtol=1e-5)


def test_dense_block_step_reduced_tokens():
    """dense_block weights (full 2048-wide Wq/Wk and one FFN matrix) updated by
    Muon and then clipped in the same muonclip_step call, with S_max from a
    reduced batch (1 x 512 tokens) of the layer's features."""
    wl = synth.scaled(synth.workload("dense_block"), B=1, S=512)
    W, G, M = synth.muon_inputs(wl, seed=12, only=("Wq", "Wk", "W_down"))
    X, _ = synth.attention_inputs(wl, seed=12)
    q, k = forward.project_mha(X.cuda(), W["Wq"].cuda(), W["Wk"].cuda(), 16)
    hp = mc.Hparams()
    names = ["Wq", "Wk", "W_down"]
    Wd = [W[n].cuda() for n in names]
    smax, _ = mc.qk_max_logit(q.cuda(), k.cuda())
    ncl = torch.zeros(1, dtype=torch.int32, device="cuda")
    layer = mc.ClipLayer(smax, mc.mha_segments(Wd[0], Wd[1], 16), nclipped=ncl)
    mc.muonclip_step(Wd, [G[n].cuda() for n in names], [M[n].cuda() for n in names], hp,
                     layers=[layer])
    torch.cuda.synchronize()
    s_ref, _ = O.max_logit(f64(q), f64(k))
    np.testing.assert_allclose(f64(smax), s_ref, rtol=1e-3)
    gamma, mask = O.clip_factors(s_ref, 100.0)
    assert sorted(np.nonzero(mask)[0].tolist()) == [2, 7, 11] and ncl.item() == 3
    assert np.all(np.abs(s_ref - 100.0) > 5.0)          # clear margin for the mask
    for i, n in enumerate(names):
        (Wn, _, Od), _ = oracle_muon(W[n], G[n], M[n], hp)
        tol = 2e-2 * rms(fp32(hp.lr) * Od)
        if n == "W_down":
            assert_rounded_within(Wd[i], Wn, tol, n)
            continue
        factor = np.repeat(np.where(mask, np.sqrt(gamma), 1.0), 128)
        s_rel = float(np.max(np.abs(f64(smax) / s_ref - 1.0))) + 1e-7   # device gamma error
        lo, hi = update_then_clip_band(Wn, tol, factor, O.round_to_bf16, gamma_rel=s_rel)
        g = f64(Wd[i])
        assert np.all((g >= lo) & (g <= hi)), n


def test_step_beyond_the_fused_apply_table():
    """More matrices than the last Newton-Schulz launch can apply in its
    epilogue (192): the step falls back to the separate apply pass; a sample
    of the 200 matrices, both orientations, against the oracle."""
    hp = mc.Hparams()
    shapes = [(64, 96) if i % 2 == 0 else (96, 64) for i in range(200)]
    W0 = [synth.normal(s, 0.02, f"bw{i}", 19).to(BF16) for i, s in enumerate(shapes)]
    G0 = [synth.normal(s, 1.0, f"bg{i}", 19) for i, s in enumerate(shapes)]
    W = [w.cuda() for w in W0]
    G = [g.cuda() for g in G0]
    M = [torch.zeros(s, device="cuda") for s in shapes]
    st = new_status()
    mc.muonclip_step(W, G, M, hp, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for i in (0, 1, 117, 199):
        (Wn, _, Od), _ = oracle_muon(W0[i], G0[i], torch.zeros(shapes[i]), hp)
        assert_rounded_within(W[i], Wn, 2e-2 * rms(fp32(hp.lr) * Od), f"W {i}")


# ------------------------------------------------------------------ ZeRO-1 ranks on the library
def test_zero1_single_rank_equals_direct_step():
    """A ZeRO-1 step on one rank (momentum on the flat slice, then
    muonclip_step with mu = 0 on the full momentum) is bit-identical to the
    direct step, clip included."""
    from muon_qk_clip_gb300.dist import LibraryOps, Zero1Layout, zero1_state, zero1_step
    shapes = [(64, 96), (128, 40), (96, 64), (64, 32), (64, 32)]
    W0 = [synth.normal(s, 0.02, f"zw{i}", 17).to(BF16) for i, s in enumerate(shapes)]
    hp = mc.Hparams()
    W1 = [w.cuda() for w in W0]
    W2 = [w.cuda() for w in W0]
    M1 = [torch.zeros(s, device="cuda") for s in shapes]
    L = Zero1Layout(shapes, 1)
    M2 = zero1_state(L, device="cuda")
    smax = torch.tensor([150.0, 20.0, 400.0, 99.0], device="cuda")
    for step in range(2):
        G = [synth.normal(s, 1.0, f"zg{i}_{step}", 17).cuda() for i, s in enumerate(shapes)]
        layer = mc.ClipLayer(smax.clone(), mc.mha_segments(W1[3], W1[4], 4))
        mc.muonclip_step(W1, G, M1, hp, layers=[layer])
        zero1_step(W2, G, M2, L, [(smax.clone(), [(3, 0, 16, 16, 0.5), (4, 0, 16, 16, 0.5)])],
                   LibraryOps(W2), hp)
    torch.cuda.synchronize()
    for a, b in zip(W1, W2):
        assert torch.equal(a, b)
    for i, m in enumerate(M1):
        a = L.offsets[i]
        assert torch.equal(M2[a:a + m.numel()].view(m.shape), m)


def test_step_with_many_shape_groups():
    """Eleven distinct shapes (more shape groups than one launch takes, split
    over two streams): tiny, one-row, ragged and tall matrices in one call,
    two with a column count that is not a multiple of 4 (the element-wise
    edge of the streaming kernels, in both orientations), each equal to its
    own oracle step."""
    shapes = [(8, 8), (1, 64), (24, 40), (129, 64), (64, 129 + 7), (200, 48), (48, 200), (513, 256),
              (256, 513 + 7), (40, 130), (131, 37)]
    hp = mc.Hparams()
    W, G, M, want = [], [], [], []
    for i, (r, c) in enumerate(shapes):
        w = synth.normal((r, c), 0.02, f"mw{i}", 18).to(BF16)
        g = synth.normal((r, c), 1.0, f"mg{i}", 18)
        m = synth.normal((r, c), 1.0, f"mm{i}", 18)
        (Wn, Mn, Od), _ = oracle_muon(w, g, m, hp)
        want.append((Wn, Mn, Od))
        W.append(padded(r, c, BF16)); W[-1].copy_(w)
        G.append(padded(r, c, F32)); G[-1].copy_(g)
        M.append(padded(r, c, F32)); M[-1].copy_(m)
    st = new_status()
    mc.muonclip_step(W, G, M, hp, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    for (Wn, Mn, Od), w, m, s in zip(want, W, M, shapes):
        assert_rounded_within(m, Mn, 0.0, f"momentum {s}")
        assert_rounded_within(w, Wn, 2e-2 * rms(fp32(hp.lr) * Od), f"W {s}")


@pytest.mark.parametrize("kind", ["gauss", "few64"])
def test_ns_fast_iterations_2048(kind):
    """Three leading one-product iterations (the default) on a 2048 x 2048
    input, Gaussian or 64 unit directions over a 1e-3 rest.  float64
    emulation of the arithmetic (tests/ns_emulation.py, the same inputs)
    gives 4.3e-3 and 1.02e-2 of RMS: inside the 2e-2 bound.  A larger
    ns_fast_steps acts as three (a fourth one-product iteration emulates at
    2.0-2.3e-2 on 1024 x 4096 and 1024 x 16384 Gaussian inputs), so its
    output is bit-identical."""
    m = n = 2048
    rng = np.random.default_rng(4096 + len(kind))
    G = rng.standard_normal((m, n))
    if kind == "few64":
        U, s, Vt = np.linalg.svd(G, full_matrices=False)
        s2 = np.full(len(s), 1e-3)
        s2[:64] = 1.0
        G = (U * s2) @ Vt
    M = torch.tensor(G, dtype=torch.float32)
    outs = {}
    for fast in (3, 4):
        hp = mc.Hparams(ns_precision=abi.MC_NS_SPLIT_BF16, ns_fast_steps=fast)
        O_dev = torch.empty(m, n, dtype=torch.float32, device="cuda")
        mc.muon_newton_schulz([M.cuda()], [O_dev], hp)
        torch.cuda.synchronize()
        outs[fast] = f64(O_dev)
    ohp = O.Hparams(rms_scale=fp32(hp.rms_scale), ns_coeffs=tuple(fp32(c) for c in hp.ns_coeffs),
                    ns_eps=fp32(hp.ns_eps), ns_steps=hp.ns_steps)
    ref = O.muon_direction(f64(M), ohp)
    err = np.abs(outs[3] - ref).max() / rms(ref)
    assert err <= 2e-2, f"max |O - O_exact| = {err:.4g} of RMS"
    assert np.array_equal(outs[3], outs[4])


@pytest.mark.parametrize("m,n,k", [(1024, 2048, 16), (256, 512, 16), (1024, 16384, 64)])
def test_ns_adversarial_spectrum(m, n, k):
    """A spectrum of k unit directions over a near-null rest (1e-3), an
    adversarial case for the split arithmetic (three one-product leading
    iterations at every size; two-product trailing updates from a smaller
    side of 512).  The directions 1e-3 below the largest are amplified ~500x
    by the iteration, so their rounding matters most.  float64 emulation of
    the arithmetic (tests/ns_emulation.py, the same inputs) gives 8.4e-3 of
    RMS at 1024 x 2048, 7.7e-3 at 256 x 512 and 1.3e-2 at 1024 x 16384 with
    64 directions, near the plan's worst case: within the 2e-2 bound."""
    rng = np.random.default_rng(m if k == 16 else m + n)
    G = rng.standard_normal((m, n))
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    s2 = np.full(len(s), 1e-3)
    s2[:k] = 1.0
    M = torch.tensor((U * s2) @ Vt, dtype=torch.float32)
    hp = mc.Hparams(ns_precision=abi.MC_NS_SPLIT_BF16)
    O_dev = torch.empty(m, n, dtype=torch.float32, device="cuda")
    mc.muon_newton_schulz([M.cuda()], [O_dev], hp)
    torch.cuda.synchronize()
    ohp = O.Hparams(rms_scale=fp32(hp.rms_scale), ns_coeffs=tuple(fp32(c) for c in hp.ns_coeffs),
                    ns_eps=fp32(hp.ns_eps), ns_steps=hp.ns_steps)
    ref = O.muon_direction(f64(M), ohp)
    err = np.abs(f64(O_dev) - ref).max() / rms(ref)
    assert err <= 2e-2, f"max |O - O_exact| = {err:.4g} of RMS"
