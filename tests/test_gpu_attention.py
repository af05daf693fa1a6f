"""GPU parity of the attention forward with the fused per-head max logit
(qk_attention_forward) against the CPU oracle's attention_forward.

Tolerances (floating point, derived from the kernel's arithmetic):
  * O: the softmax numerators are rounded to bf16 (relative 2^-9) before the
    P V product and O is rounded to bf16 once, so
        |O - O_exact| <= 2^-8 * (P |V|) + 2^-8 * |O_exact|
    (twice the first-order bound; P |V| is the oracle's attention of |V|)
  * lse: 1e-3 * max(1, S_max^h) absolute (fp32 logits and row sums)
  * S_max: relative 1e-3 against the oracle (bf16 features, fp32 accumulate),
    and equal to qk_max_logit's value on the same features to 1e-6
"""
import numpy as np
import pytest
import torch

import oracle as O
from muon_qk_clip_gb300 import abi, build
from muon_qk_clip_gb300 import binding as mc
from muon_qk_clip_gb300 import synth
from tests.gpu_helpers import f64

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    abi.load()


def features(B, S, H, dh, dr, dv, seed, key_growth=0.0, head_scale=None):
    """bf16 q [B,S,H,dh+dr], k [B,S,H,dh], k_shared [B,S,dr] or None, v [B,S,H,dv]."""
    q = synth.normal((B, S, H, dh + dr), 1.0, "aq", seed)
    k = synth.normal((B, S, H, dh), 1.0, "ak", seed)
    ks = synth.normal((B, S, dr), 1.0, "aks", seed) if dr else None
    v = synth.normal((B, S, H, dv), 1.0, "av", seed)
    if head_scale is not None:
        q = q * torch.tensor(head_scale, dtype=q.dtype)[None, None, :, None]
    if key_growth:
        g = 1.0 + key_growth * torch.arange(S, dtype=torch.float32) / S
        k = k * g[None, :, None, None]
        if ks is not None:
            ks = ks * g[None, :, None]
    cast = lambda t: None if t is None else t.to(BF16)
    return cast(q), cast(k), cast(ks), cast(v)


def check_against_oracle(q, k, ks, v, out, lse, smax, causal=True, heads=None):
    Q, K, V = f64(q), f64(k), f64(v)
    Ks = None if ks is None else f64(ks)
    if heads is not None:
        Q, K, V = Q[:, :, heads], K[:, :, heads], V[:, :, heads]
    Oref, lref, sref = O.attention_forward(Q, K, V, Ks, causal=causal)
    A, _, _ = O.attention_forward(Q, K, np.abs(V), Ks, causal=causal)
    got = f64(out) if heads is None else f64(out)[:, :, heads]
    bound = 2.0 ** -8 * A + 2.0 ** -8 * np.abs(Oref) + 1e-7
    err = np.abs(got - Oref)
    assert np.all(err <= bound), f"O: worst excess {np.max(err - bound):.3g}, max err {err.max():.3g}"
    gl = f64(lse) if heads is None else f64(lse)[:, heads]
    tol = 1e-3 * np.maximum(1.0, sref)[None, :, None]
    assert np.all(np.abs(gl - lref) <= tol), f"lse: max err {np.max(np.abs(gl - lref)):.3g}"
    gs = f64(smax) if heads is None else f64(smax)[heads]
    np.testing.assert_allclose(gs, sref, rtol=1e-3)
    return sref


@pytest.mark.parametrize("B,S,H,dh,dr,dv,causal", [
    (2, 300, 3, 128, 0, 128, True),       # MHA, ragged last block
    (1, 128, 2, 128, 0, 128, True),       # exactly one block
    (1, 257, 2, 128, 64, 128, True),      # MLA: k^C + shared k^R, d_v 128
    (2, 200, 2, 64, 0, 64, True),         # d = 64, d_v = 64
    (1, 333, 2, 128, 0, 128, False),      # no mask
    (1, 97, 3, 128, 64, 128, False),      # MLA, no mask, shorter than a block
])
def test_attention_forward_parity(B, S, H, dh, dr, dv, causal):
    q, k, ks, v = features(B, S, H, dh, dr, dv, seed=50 + S)
    dq = lambda t: None if t is None else t.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, smax = mc.qk_attention_forward(dq(q), dq(k), dq(v), dq(ks), causal=causal, lse=True,
                                             status=st)
    ref_s, _ = mc.qk_max_logit(dq(q), dq(k), dq(ks), causal=causal)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_against_oracle(q, k, ks, v, out.cpu(), lse.cpu(), smax.cpu(), causal)
    np.testing.assert_allclose(f64(smax), f64(ref_s), rtol=1e-6)


def test_attention_forward_heavy_logits_rescale():
    """Logits up to ~300 whose row maxima keep growing along the sequence:
    the lazily updated running maximum must rescale O and the row sums."""
    q, k, ks, v = features(1, 640, 3, 128, 0, 128, seed=61, key_growth=3.0,
                           head_scale=[1.0, 12.0, 25.0])
    out, lse, smax = mc.qk_attention_forward(q.cuda(), k.cuda(), v.cuda(), lse=True)
    torch.cuda.synchronize()
    sref = check_against_oracle(q, k, ks, v, out.cpu(), lse.cpu(), smax.cpu())
    assert sref[2] > 100.0                 # the scaled head does exceed tau


def test_attention_forward_accumulates_smax_over_micro_batches():
    q, k, ks, v = features(4, 256, 2, 128, 64, 128, seed=62)
    qd, kd, ksd, vd = q.cuda(), k.cuda(), ks.cuda(), v.cuda()
    _, _, full = mc.qk_attention_forward(qd, kd, vd, ksd)
    _, _, part = mc.qk_attention_forward(qd[:2], kd[:2], vd[:2], ksd[:2])
    mc.qk_attention_forward(qd[2:], kd[2:], vd[2:], ksd[2:], smax=part, accumulate=True)
    torch.cuda.synchronize()
    assert torch.equal(full, part)


def test_attention_forward_flags_nonfinite_logit():
    q, k, _, v = features(1, 64, 2, 128, 0, 128, seed=63)
    q[0, 5, 1, 3] = float("inf")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.qk_attention_forward(q.cuda(), k.cuda(), v.cuda(), status=st)
    torch.cuda.synchronize()
    assert st.item() & abi.MC_STATUS_NONFINITE_LOGIT


def test_attention_forward_dense_block_full_size():
    """The dense_block layer (B 4, S 4096, H 16, d 128) in the launch the
    benchmark reports: S_max of every head equals qk_max_logit's, and two heads
    (one pre-scaled past tau) match the oracle on every row of batch 0."""
    wl = synth.workload("dense_block")
    att = wl.attention
    X, Wa = synth.attention_inputs(wl, seed=64, device="cuda")
    from muon_qk_clip_gb300 import forward
    q, k = forward.project_mha(X, Wa["Wq"], Wa["Wk"], att.H)
    v = synth.normal((att.B, att.S, att.H, att.d_head), 1.0, "dv", 64, BF16, "cuda")
    q, k = q.contiguous(), k.contiguous()
    del X
    out, lse, smax = mc.qk_attention_forward(q, k, v, lse=True)
    ref_s, _ = mc.qk_max_logit(q, k)
    torch.cuda.synchronize()
    np.testing.assert_allclose(f64(smax), f64(ref_s), rtol=1e-6)
    heads = [0, sorted(att.scaled_heads)[0]]
    Q, K, V = f64(q[:1]), f64(k[:1]), f64(v[:1])
    Oref, lref, sref = O.attention_forward(Q[:, :, heads], K[:, :, heads], V[:, :, heads])
    A, _, _ = O.attention_forward(Q[:, :, heads], K[:, :, heads], np.abs(V[:, :, heads]))
    got = f64(out[:1])[:, :, heads]
    assert np.all(np.abs(got - Oref) <= 2.0 ** -8 * A + 2.0 ** -8 * np.abs(Oref) + 1e-7)
    gl = f64(lse[:1])[:, heads]
    assert np.all(np.abs(gl - lref) <= 1e-3 * np.maximum(1.0, sref)[None, :, None])
    assert f64(smax)[heads[1]] > 100.0
