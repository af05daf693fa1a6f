"""Untimed setup: query/key features of an attention layer from its weights.

This is the model forward that produces Q and K (Q^h = X W_q^h, K^h = X W_k^h
for MHA; the MLA latent projections with RMSNorm and RoPE, [K2-internals]
"MLA 的特殊处理"), run on the library's own kernels (mc_matmul on the tcgen05
GEMM core for bf16, mc_rms_norm, mc_rope) to build inputs for qk_max_logit
and to re-measure S_max after a clip.  It is not part of the MuonClip step: in
training, S_max comes from the forward pass.  Device tensors only.
"""
from __future__ import annotations

from . import binding as mc


def _on_device(*ts):
    for t in ts:
        if t.device.type != "cuda":
            raise ValueError("the projection runs on the library's CUDA kernels: pass device tensors")


def project_mha(X, Wq, Wk, H: int):
    """Q = X Wq^T, K = X Wk^T as [B, S, H, d] views (fp32 accumulate, X dtype out)."""
    _on_device(X, Wq, Wk)
    B, S, D = X.shape
    x2 = X.reshape(B * S, D)
    q = mc.matmul(x2, Wq.contiguous())
    k = mc.matmul(x2, Wk.contiguous())
    return q.reshape(B, S, H, -1), k.reshape(B, S, H, -1)


def project_mla(X, W, H: int, d_nope=128, d_rope=64, d_v=128, with_v=False):
    """MLA features: Q [B,S,H,d_nope+d_rope] = [q^C || RoPE(q^R)], K^C a
    [B,S,H,d_nope] strided view into the [B,S,H,d_nope+d_v] key/value
    projection, and the shared rotary key K^R = RoPE(X W_KR^T) [B,S,d_rope];
    with_v adds the values V, the other strided view [B,S,H,d_v] of that
    projection.  The latents c_Q = RMSNorm(X W_DQ^T) and c_KV =
    RMSNorm(X W_DKV^T) are rounded to X's dtype before their up-projections."""
    _on_device(X, *W.values())
    B, S, D = X.shape
    x2 = X.reshape(B * S, D)
    cq = mc.rms_norm(mc.matmul(x2, W["W_DQ"].contiguous()))
    q = mc.matmul(cq, W["W_UQ"].contiguous()).reshape(B, S, H, d_nope + d_rope)
    mc.rope_(q[..., d_nope:])
    ckv = mc.rms_norm(mc.matmul(x2, W["W_DKV"].contiguous()))
    kv = mc.matmul(ckv, W["W_UKV"].contiguous()).reshape(B, S, H, d_nope + d_v)
    kr = mc.matmul(x2, W["W_KR"].contiguous()).reshape(B, S, d_rope)
    mc.rope_(kr)
    if with_v:
        return q, kv[..., :d_nope], kr, kv[..., d_nope:]
    return q, kv[..., :d_nope], kr
