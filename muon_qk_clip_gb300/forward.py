"""Untimed setup: query/key features of an attention layer from its weights.

This is the model forward that produces Q and K (Q^h = X W_q^h, K^h = X W_k^h
for MHA; the MLA latent projections with RMSNorm and RoPE), run with torch
matmuls to build inputs for qk_max_logit.  It is not part of the MuonClip
step: in training, S_max comes from the forward pass.
"""
from __future__ import annotations

import torch


def project_mha(X, Wq, Wk, H: int):
    """Q = X Wq^T, K = X Wk^T as [B, S, H, d] views (fp32 accumulate, X dtype out)."""
    B, S, D = X.shape
    x2 = X.reshape(B * S, D)
    q = (x2.float() @ Wq.float().t()) if X.device.type == "cpu" else (x2 @ Wq.t())
    k = (x2.float() @ Wk.float().t()) if X.device.type == "cpu" else (x2 @ Wk.t())
    return q.to(X.dtype).reshape(B, S, H, -1), k.to(X.dtype).reshape(B, S, H, -1)


def _rms(x, eps=1e-6):
    x = x.float()
    return x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + eps)


def _rope(x, theta=10000.0):
    """Interleaved-pair rotary embedding along axis 1 (positions 0..S-1)."""
    S, d = x.shape[1], x.shape[-1]
    inv = theta ** (-torch.arange(0, d, 2, dtype=torch.float64, device=x.device) / d)
    ang = torch.arange(S, dtype=torch.float64, device=x.device)[:, None] * inv[None, :]
    shape = [1, S] + [1] * (x.dim() - 3) + [d // 2]
    cos, sin = ang.cos().float().reshape(shape), ang.sin().float().reshape(shape)
    x = x.float()
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = torch.empty_like(x)
    out[..., 0::2] = x0 * cos - x1 * sin
    out[..., 1::2] = x0 * sin + x1 * cos
    return out


def project_mla(X, W, H: int, d_nope=128, d_rope=64, d_v=128, chunk=4096, with_v=False):
    """MLA features: Q [B,S,H,d_nope+d_rope] = [q^C || q^R], K^C a [B,S,H,d_nope]
    strided view into the [B,S,H,d_nope+d_v] key/value projection, and the
    shared rotary key K^R [B,S,d_rope]; with_v adds the values V, the other
    strided view [B,S,H,d_v] of that projection."""
    B, S, D = X.shape
    dt = X.dtype
    mm = (lambda a, w: a.float() @ w.float().t()) if X.device.type == "cpu" else (lambda a, w: a @ w.t())
    x2 = X.reshape(B * S, D)
    cq = _rms(mm(x2, W["W_DQ"])).to(dt)
    q = mm(cq, W["W_UQ"]).float().reshape(B, S, H, d_nope + d_rope)
    q[..., d_nope:] = _rope(q[..., d_nope:])
    ckv = _rms(mm(x2, W["W_DKV"])).to(dt)
    kv = mm(ckv, W["W_UKV"]).to(dt).reshape(B, S, H, d_nope + d_v)
    kr = _rope(mm(x2, W["W_KR"]).float().reshape(B, S, d_rope)).to(dt)
    if with_v:
        return q.to(dt), kv[..., :d_nope], kr, kv[..., d_nope:]
    return q.to(dt), kv[..., :d_nope], kr
