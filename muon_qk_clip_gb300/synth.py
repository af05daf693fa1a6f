"""Seeded synthetic inputs for the MuonClip workloads.

This module only draws random numbers and lays out shapes; it holds none of
the method's arithmetic.  Tests, the benchmark and the oracle-side checks all
take their inputs from here.  Every tensor is drawn from its own
torch.Generator seeded with crc32(f"{seed}:{key}"), so a tensor does not
depend on which other tensors were drawn.  The stream differs between CPU and
CUDA generators: tests that compare CPU and GPU results draw on the CPU and
copy.

Workloads (sizes and distributions of the Kimi K2 model that MuonClip trained):
  tiny_mha_fp32    d_model 256, 4 heads x 64, one 256x512 Muon matrix, fp32
  dense_block      d_model 2048, 16 heads x 128, FFN 2048->5632->2048, bf16
  k2_mla_layer     hidden 7168, 64 heads, q_lora 1536, kv_lora 512,
                   nope 128 / rope 64 / v 128, bf16
  moe_experts      64 experts 2048x7168 + 64 experts 7168x2048, bf16
  long_mla         k2_mla_layer at 32768 tokens
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field

import torch


def generator(seed: int, key: str, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(zlib.crc32(f"{seed}:{key}".encode()) & 0x7FFFFFFF)
    return g


def normal(shape, std: float, key: str, seed: int = 0, dtype=torch.float32, device="cpu"):
    """N(0, std^2) draws, generated in fp32 then cast to `dtype`."""
    g = generator(seed, key, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def uniform(shape, lo: float, hi: float, key: str, seed: int = 0, device="cpu"):
    g = generator(seed, key, device)
    return torch.rand(*shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


@dataclass
class MatrixSpec:
    name: str
    rows: int
    cols: int
    g_scale: float = 1.0       # extra factor on this matrix's gradient


@dataclass
class AttentionSpec:
    kind: str                  # "mha" or "mla"
    d_model: int
    H: int
    B: int
    S: int
    w_std: float
    d_head: int = 0            # MHA head dim
    q_lora: int = 0            # MLA dims
    kv_lora: int = 0
    d_nope: int = 0
    d_rope: int = 0
    d_v: int = 0
    scaled_heads: dict = field(default_factory=dict)   # head -> row multiplier
    scale_rows: str = "qk"     # MLA: "qc_kc_qr" (all head-specific q/k rows) or "qc"


@dataclass
class Workload:
    name: str
    dtype: torch.dtype         # weight dtype (momentum is always fp32)
    matrices: list
    w_std: float
    g_std: float
    attention: AttentionSpec | None = None
    muon_on_attention: bool = True   # the Muon set contains the attention weights


def _mla_matrices(D, H, ql, kl, dn, dr, dv):
    return [MatrixSpec("W_DQ", ql, D), MatrixSpec("W_UQ", H * (dn + dr), ql),
            MatrixSpec("W_DKV", kl, D), MatrixSpec("W_KR", dr, D),
            MatrixSpec("W_UKV", H * (dn + dv), kl), MatrixSpec("W_O", D, H * dv)]


def workload(name: str, variant: str = "calibrated") -> Workload:
    """The five workloads.  `variant` picks the head pre-scale: "literal" uses
    the configs' stated multipliers (x8 tiny, x6 MLA, x10 long), under which
    no head exceeds tau=100; "calibrated" uses multipliers that put the named
    heads' max logit near 3 tau (S grows as the square of the multiplier)."""
    cal = variant == "calibrated"
    if name == "tiny_mha_fp32":
        att = AttentionSpec("mha", 256, 4, 2, 128, 0.02, d_head=64,
                            scaled_heads={1: 25.0, 3: 25.0} if cal else {1: 8.0, 3: 8.0})
        return Workload(name, torch.float32, [MatrixSpec("W", 256, 512)], 0.02, 1.0, att,
                        muon_on_attention=False)
    if name == "dense_block":
        mats = [MatrixSpec(n, 2048, 2048) for n in ("Wq", "Wk", "Wv", "Wo")] + [
            MatrixSpec("W_up", 5632, 2048), MatrixSpec("W_gate", 5632, 2048),
            MatrixSpec("W_down", 2048, 5632)]
        att = AttentionSpec("mha", 2048, 16, 4, 4096, 0.02, d_head=128,
                            scaled_heads={2: 8.0, 7: 8.0, 11: 8.0})
        return Workload(name, torch.bfloat16, mats, 0.02, 1e-3, att)
    if name in ("k2_mla_layer", "long_mla"):
        D, H, ql, kl, dn, dr, dv = 7168, 64, 1536, 512, 128, 64, 128
        if name == "k2_mla_layer":
            heads = {5: 50.0, 17: 50.0, 33: 50.0, 50: 50.0} if cal else {5: 6.0, 17: 6.0, 33: 6.0, 50: 6.0}
            S, rows = 4096, "qc_kc_qr"
        else:
            named = (3, 11, 19, 27, 35, 43, 51, 59)
            heads = ({h: 35.0 + 5.0 * i for i, h in enumerate(named)} if cal
                     else {h: 10.0 for h in named})
            S, rows = 32768, ("qc_kc_qr" if cal else "qc")
        att = AttentionSpec("mla", D, H, 1, S, 0.006, q_lora=ql, kv_lora=kl, d_nope=dn,
                            d_rope=dr, d_v=dv, scaled_heads=heads, scale_rows=rows)
        return Workload(name, torch.bfloat16, _mla_matrices(D, H, ql, kl, dn, dr, dv), 0.006,
                        1e-3, att)
    if name == "moe_experts":
        u = uniform((128,), -1.0, 1.0, "expert_grad_scale")       # log10 of the scale
        mats = [MatrixSpec(f"E{i}_up", 2048, 7168, float(10 ** u[i])) for i in range(64)] + [
            MatrixSpec(f"E{i}_down", 7168, 2048, float(10 ** u[64 + i])) for i in range(64)]
        return Workload(name, torch.bfloat16, mats, 0.006, 1e-3, None)
    raise KeyError(name)


WORKLOADS = ("tiny_mha_fp32", "dense_block", "k2_mla_layer", "moe_experts", "long_mla")


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of `wl` with attention fields replaced (smaller S/B for tests)."""
    import copy
    w = copy.deepcopy(wl)
    for k, v in kw.items():
        setattr(w.attention, k, v)
    return w


def muon_inputs(wl: Workload, seed: int = 0, device="cpu", warm_momentum: bool = False,
                only=None):
    """Weights W (wl.dtype), gradients G (fp32) and momentum M (fp32) per matrix.
    Attention head multipliers are applied to the weights' head rows."""
    W, G, M = {}, {}, {}
    for ms in wl.matrices:
        if only is not None and ms.name not in only:
            continue
        w = normal((ms.rows, ms.cols), wl.w_std, f"W:{ms.name}", seed, torch.float32, device)
        W[ms.name] = w
        G[ms.name] = normal((ms.rows, ms.cols), wl.g_std * ms.g_scale, f"G:{ms.name}", seed,
                            torch.float32, device)
        M[ms.name] = (normal((ms.rows, ms.cols), wl.g_std * ms.g_scale * 3.0, f"M:{ms.name}", seed,
                             torch.float32, device) if warm_momentum
                      else torch.zeros(ms.rows, ms.cols, device=device))
    if wl.attention is not None and wl.muon_on_attention:
        _apply_head_scales(wl.attention, W)
    return {k: v.to(wl.dtype) for k, v in W.items()}, G, M


def _apply_head_scales(att: AttentionSpec, W: dict):
    for h, r in att.scaled_heads.items():
        if att.kind == "mha":
            d = att.d_head
            if "Wq" in W:
                W["Wq"][h * d:(h + 1) * d] *= r
                W["Wk"][h * d:(h + 1) * d] *= r
        else:
            dq, dkv = att.d_nope + att.d_rope, att.d_nope + att.d_v
            if "W_UQ" in W:
                if att.scale_rows == "qc":
                    W["W_UQ"][h * dq:h * dq + att.d_nope] *= r
                else:
                    W["W_UQ"][h * dq:(h + 1) * dq] *= r
                    W["W_UKV"][h * dkv:h * dkv + att.d_nope] *= r


def attention_inputs(wl: Workload, seed: int = 0, device="cpu"):
    """Token features X [B, S, d_model] ~ N(0,1) and the attention weights.
    For workloads whose Muon set excludes the attention weights (tiny MHA),
    the attention weights are drawn here.  Returns (X, weights dict)."""
    att = wl.attention
    X = normal((att.B, att.S, att.d_model), 1.0, "X", seed, torch.float32, device).to(wl.dtype)
    if wl.muon_on_attention:
        W, _, _ = muon_inputs(wl, seed, device, only=_attn_names(att))
        return X, W
    W = {}
    for n in ("Wq", "Wk", "Wv", "Wo"):
        W[n] = normal((att.d_model, att.d_model), att.w_std, f"W:{n}", seed, torch.float32, device)
    _apply_head_scales(att, W)
    return X, {k: v.to(wl.dtype) for k, v in W.items()}


def _attn_names(att: AttentionSpec):
    return ("Wq", "Wk") if att.kind == "mha" else ("W_DQ", "W_UQ", "W_DKV", "W_UKV", "W_KR")


def ns_test_matrix(rows: int, cols: int, seed: int = 0, key: str = "ns", device="cpu"):
    """A gradient-like fp32 matrix for Newton-Schulz tests."""
    return normal((rows, cols), 1e-3, key, seed, torch.float32, device)


def attention_features(B, S, H, dq, dk, dr, dtype, seed=0, device="cpu", std=1.0, key="qk"):
    """Random Q [B,S,H,dq], K [B,S,H,dk], K_shared [B,S,dr] (or None) features."""
    q = normal((B, S, H, dq), std, key + ":q", seed, torch.float32, device).to(dtype)
    k = normal((B, S, H, dk), std, key + ":k", seed, torch.float32, device).to(dtype)
    ks = normal((B, S, dr), std, key + ":ks", seed, torch.float32, device).to(dtype) if dr else None
    return q, k, ks


def flops_ns(rows: int, cols: int, steps: int = 5) -> float:
    """Algorithmic flops of `steps` Newton-Schulz iterations on one matrix:
    4 m^2 n + 2 m^3 per iteration, m = min, n = max."""
    m, n = min(rows, cols), max(rows, cols)
    return steps * (4.0 * m * m * n + 2.0 * m ** 3)


def flops_max_logit(B, S, H, d, causal=True) -> float:
    pairs = S * (S + 1) / 2 if causal else S * S
    return 2.0 * d * B * H * pairs


__all__ = ["generator", "normal", "uniform", "workload", "WORKLOADS", "muon_inputs",
           "attention_inputs", "ns_test_matrix", "attention_features", "flops_ns",
           "flops_max_logit", "scaled", "math"]
