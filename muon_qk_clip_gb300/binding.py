"""Python binding of the MuonClip C ABI, with the same call names.

Each function converts torch tensors into the C descriptors (device pointers,
shapes, strides) and calls libmuonclip.so on the current CUDA stream.  Torch
provides device memory and streams only; no arithmetic of the method happens
here.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from . import abi
from .abi import McAttnDesc, McAttnOut, McClipLayer, McClipSeg, McHparams, McMat, check

_DT = {torch.float32: abi.MC_F32, torch.bfloat16: abi.MC_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def mat(t: torch.Tensor) -> McMat:
    """Descriptor of a 2-D row-major tensor (unit column stride)."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return McMat(ctypes.c_void_p(t.data_ptr()), _DT[t.dtype], 0, t.shape[0], t.shape[1],
                 max(t.stride(0), t.shape[1]))


def _mats(ts):
    arr = (McMat * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = mat(t)
    return arr


@dataclass
class Hparams:
    """Mirror of mc_hparams; defaults follow mc_default_hparams."""
    mu: float = 0.95
    lr: float = 2e-4
    weight_decay: float = 0.1
    rms_scale: float = 0.2
    ns_steps: int = 5
    ns_coeffs: tuple = (3.4445, -4.7750, 2.0315)
    ns_eps: float = 1e-7
    tau: float = 100.0
    alpha: float = 0.5
    ns_precision: int = abi.MC_NS_AUTO
    ns_fast_steps: int = 3
    scale_mode: int = abi.MC_SCALE_RMS

    def c(self) -> McHparams:
        a, b, c = self.ns_coeffs
        return McHparams(self.mu, self.lr, self.weight_decay, self.rms_scale, self.ns_steps,
                         a, b, c, self.ns_eps, self.tau, self.alpha, self.ns_precision,
                         self.ns_fast_steps, self.scale_mode)


def default_hparams() -> Hparams:
    h = McHparams()
    abi.load().mc_default_hparams(ctypes.byref(h))
    return Hparams(h.mu, h.lr, h.weight_decay, h.rms_scale, h.ns_steps, (h.ns_a, h.ns_b, h.ns_c),
                   h.ns_eps, h.tau, h.alpha, h.ns_precision, h.ns_fast_steps, h.scale_mode)


def workspace_size(shapes_or_tensors, hp: Hparams | None = None) -> int:
    hp = hp or Hparams()
    arr = (McMat * len(shapes_or_tensors))()
    for i, s in enumerate(shapes_or_tensors):
        r, c = (s.shape if isinstance(s, torch.Tensor) else s)
        arr[i] = McMat(None, abi.MC_F32, 0, r, c, c)
    n = ctypes.c_size_t(0)
    hc = hp.c()
    check(abi.load().mc_workspace_size(arr, len(arr), ctypes.byref(hc), ctypes.byref(n)),
          "mc_workspace_size")
    return n.value


def ns_products(rows: int, cols: int, hp: Hparams | None = None) -> list:
    """Products per k-step of each Newton-Schulz iteration's (Gram, polynomial,
    update) on the split-bf16 tensor-core path: a list of ns_steps triples."""
    hp = hp or Hparams()
    out = (ctypes.c_int32 * (3 * hp.ns_steps))()
    hc = hp.c()
    check(abi.load().mc_ns_products(ctypes.byref(hc), rows, cols, out), "mc_ns_products")
    return [tuple(out[3 * i:3 * i + 3]) for i in range(hp.ns_steps)]


def alloc_workspace(shapes_or_tensors, hp=None, device="cuda") -> torch.Tensor:
    n = workspace_size(shapes_or_tensors, hp)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def muon_momentum(M, G, mu: float, status=None, stream=None):
    """M_t = mu M_{t-1} + G_t in place for every pair of matrices."""
    lib = abi.load()
    check(lib.muon_momentum(_mats(M), _mats(G), len(M), mu, _ptr(status), _stream(stream)),
          "muon_momentum")


def muon_newton_schulz(M, O, hp: Hparams | None = None, workspace=None, status=None, stream=None):
    """O = NewtonSchulz(M) * sqrt(max(rows, cols)) * rms_scale for every matrix."""
    hp = hp or Hparams()
    if workspace is None:
        workspace = alloc_workspace(M, hp, M[0].device)
    hc = hp.c()
    check(abi.load().muon_newton_schulz(_mats(M), _mats(O), len(M), ctypes.byref(hc),
                                        _ptr(workspace), workspace.numel(), _ptr(status),
                                        _stream(stream)), "muon_newton_schulz")


def attn_desc(q, k, k_shared=None, causal=True, scale=None) -> McAttnDesc:
    """q: [B,S,H,dq], k: [B,S,H,dk], k_shared: [B,S,dr] (dq = dk + dr); any
    strides with a contiguous feature axis."""
    B, S, H, dq = q.shape
    dk = k.shape[-1]
    dr = 0 if k_shared is None else k_shared.shape[-1]
    if dq != dk + dr:
        raise ValueError("q feature length must equal k + k_shared lengths")
    if q.stride(3) != 1 or k.stride(3) != 1 or (k_shared is not None and k_shared.stride(2) != 1):
        raise ValueError("feature axis must be contiguous")
    if q.dtype not in _DT or k.dtype != q.dtype or (k_shared is not None and k_shared.dtype != q.dtype):
        raise ValueError("q, k, k_shared must share a supported dtype")
    d = McAttnDesc()
    d.B, d.S, d.H, d.d_head, d.d_shared = B, S, H, dk, dr
    d.dtype = _DT[q.dtype]
    d.causal = 1 if causal else 0
    d.scale = (1.0 / math.sqrt(dq)) if scale is None else scale
    d.q, d.k = q.data_ptr(), k.data_ptr()
    d.k_shared = None if k_shared is None else k_shared.data_ptr()
    for i in range(3):
        d.q_strides[i] = q.stride(i)
        d.k_strides[i] = k.stride(i)
    if k_shared is not None:
        d.ks_strides[0], d.ks_strides[1] = k_shared.stride(0), k_shared.stride(1)
    return d


def qk_max_logit(q, k, k_shared=None, causal=True, scale=None, smax=None, argmax=None,
                 accumulate=False, status=None, stream=None):
    """Per-head max logit S_max^h; returns (smax [H] f32, argmax [H] int64 or None)."""
    H = q.shape[2]
    if smax is None:
        smax = torch.empty(H, dtype=torch.float32, device=q.device)
    d = attn_desc(q, k, k_shared, causal, scale)
    check(abi.load().qk_max_logit(ctypes.byref(d), _ptr(smax), _ptr(argmax), int(bool(accumulate)),
                                  _ptr(status), _stream(stream)), "qk_max_logit")
    return smax, argmax


def qk_attention_forward(q, k, v, k_shared=None, causal=True, scale=None, out=None, lse=None,
                         smax=None, accumulate=False, status=None, stream=None):
    """Attention forward O = softmax(scale Q K^T) V with the per-head max logit
    fused in.  q: [B,S,H,dq], k: [B,S,H,dk], k_shared: [B,S,dr] or None,
    v: [B,S,H,dv] (bf16, contiguous feature axes).  Returns (out [B,S,H,dv],
    lse [B,H,S] f32 or None, smax [H] f32); pass lse=True to allocate it."""
    B, S, H, _ = q.shape
    dv = v.shape[-1]
    if v.shape[:3] != (B, S, H) or v.stride(3) != 1 or v.dtype != q.dtype:
        raise ValueError("v must be [B, S, H, d_v] with a contiguous feature axis and q's dtype")
    if out is None:
        out = torch.empty((B, S, H, dv), dtype=q.dtype, device=q.device)
    if out.shape != v.shape or out.stride(3) != 1 or out.dtype != q.dtype:
        raise ValueError("out must be [B, S, H, d_v] with a contiguous feature axis")
    if lse is True:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if lse is not None and (tuple(lse.shape) != (B, H, S) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous [B, H, S] float32 tensor")
    if smax is None:
        smax = torch.empty(H, dtype=torch.float32, device=q.device)
    d = attn_desc(q, k, k_shared, causal, scale)
    o = McAttnOut()
    o.v, o.d_v = v.data_ptr(), dv
    o.o = out.data_ptr()
    for i in range(3):
        o.v_strides[i] = v.stride(i)
        o.o_strides[i] = out.stride(i)
    o.lse = None if lse is None else lse.data_ptr()
    check(abi.load().qk_attention_forward(ctypes.byref(d), ctypes.byref(o), _ptr(smax),
                                          int(bool(accumulate)), _ptr(status), _stream(stream)),
          "qk_attention_forward")
    return out, lse, smax


@dataclass
class ClipSegment:
    """Rows [offset + h*stride, +rows) of `w` belong to head h; scaled by gamma^exponent."""
    w: torch.Tensor
    offset: int
    stride: int
    rows: int
    exponent: float

    def c(self) -> McClipSeg:
        return McClipSeg(mat(self.w), self.offset, self.stride, self.rows, self.exponent, 0)


def _segs(segs):
    arr = (McClipSeg * max(len(segs), 1))()
    for i, s in enumerate(segs):
        arr[i] = s.c()
    return arr


def qk_clip_apply(smax, tau: float, segments, gamma_out=None, nclipped=None, status=None,
                  stream=None, mode: int = abi.MC_CLIP_PER_HEAD):
    """Rescale the rows of every head whose smax exceeds tau (in place); with
    mode=MC_CLIP_TOTAL every head takes one gamma from the layer's max."""
    arr = _segs(segments)
    check(abi.load().qk_clip_apply(_ptr(smax), smax.numel(), tau, mode, arr, len(segments),
                                   _ptr(gamma_out), _ptr(nclipped), _ptr(status), _stream(stream)),
          "qk_clip_apply")


@dataclass
class ClipLayer:
    smax: torch.Tensor
    segments: list
    gamma_out: torch.Tensor | None = None
    nclipped: torch.Tensor | None = None
    mode: int = abi.MC_CLIP_PER_HEAD


def muonclip_step(W, G, M, hp: Hparams | None = None, layers=(), workspace=None, status=None,
                  stream=None):
    """One MuonClip step: Muon on every (W, G, M) triple, then per-head QK-Clip."""
    hp = hp or Hparams()
    if workspace is None:
        workspace = alloc_workspace(W, hp, W[0].device)
    larr = (McClipLayer * max(len(layers), 1))()
    keep = []
    for i, L in enumerate(layers):
        segs = _segs(L.segments)
        keep.append(segs)
        larr[i] = McClipLayer(_ptr(L.smax), L.smax.numel(), len(L.segments),
                              ctypes.cast(segs, ctypes.POINTER(McClipSeg)),
                              _ptr(L.gamma_out), _ptr(L.nclipped), L.mode, 0)
    hc = hp.c()
    check(abi.load().muonclip_step(_mats(W), _mats(G), _mats(M), len(W), ctypes.byref(hc), larr,
                                   len(layers), _ptr(workspace), workspace.numel(), _ptr(status),
                                   _stream(stream)), "muonclip_step")


def _rows(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name}: expected a 2-D tensor with unit column stride")
    if t.dtype not in _DT:
        raise ValueError(f"{name}: unsupported dtype {t.dtype}")
    return max(t.stride(0), t.shape[1])


def matmul(A, B, out=None, scratch=None, status=None, stream=None):
    """Setup: D = A B^T on the library's GEMM core (bf16: tcgen05; fp32: CUDA
    cores).  A [M, K] and B [N, K] row-major device tensors of one dtype."""
    lda, ldb = _rows(A, "A"), _rows(B, "B")
    if A.dtype != B.dtype or A.shape[1] != B.shape[1]:
        raise ValueError("A and B need one dtype and one K")
    M, K, N = A.shape[0], A.shape[1], B.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=A.dtype, device=A.device)
    ldd = _rows(out, "out")
    if scratch is None and A.dtype == torch.bfloat16:
        scratch = torch.empty(4, dtype=torch.int32, device=A.device)
    check(abi.load().mc_matmul(_ptr(A), lda, _ptr(B), ldb, _ptr(out), ldd, M, N, K, _DT[A.dtype],
                               _ptr(scratch), _ptr(status), _stream(stream)), "mc_matmul")
    return out


def rms_norm(x, out=None, eps: float = 1e-6, stream=None):
    """Setup: weightless RMSNorm of each row of a 2-D device tensor (out may be x)."""
    ldx = _rows(x, "x")
    if out is None:
        out = torch.empty_like(x)
    ldy = _rows(out, "out")
    check(abi.load().mc_rms_norm(_ptr(x), ldx, _ptr(out), ldy, x.shape[0], x.shape[1], _DT[x.dtype],
                                 float(eps), _stream(stream)), "mc_rms_norm")
    return out


def rope_(x, theta: float = 10000.0, stream=None):
    """Setup: rotary embedding in place on interleaved pairs of x [B, S, d] or
    [B, S, heads, d] (unit stride along d), positions 0..S-1."""
    if x.stride(-1) != 1 or x.dtype not in _DT or x.dim() not in (3, 4):
        raise ValueError("x: [B, S, d] or [B, S, heads, d] with unit stride along d")
    B, S, d = x.shape[0], x.shape[1], x.shape[-1]
    nh, sh = (x.shape[2], x.stride(2)) if x.dim() == 4 else (1, 0)
    check(abi.load().mc_rope(_ptr(x), B, S, nh, d, x.stride(0), x.stride(1), sh, _DT[x.dtype],
                             float(theta), _stream(stream)), "mc_rope")
    return x


def profiler_enable(on: bool = True):
    """Bracket every library launch with CUDA events (per kernel class)."""
    abi.load().mc_profiler_enable(1 if on else 0)


def selftest_bounded_wait(budget_ns: int, abort_after_ns: int = 0, status=None, stream=None):
    """Run the bounded-wait self-check; returns (status int32[1], waited_ns
    int64[1]) device tensors, filled once the stream reaches the launch."""
    dev = torch.device("cuda", torch.cuda.current_device())
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    waited = torch.zeros(1, dtype=torch.int64, device=dev)
    check(abi.load().mc_selftest_bounded_wait(int(budget_ns), int(abort_after_ns), _ptr(status),
                                              _ptr(waited), _stream(stream)),
          "mc_selftest_bounded_wait")
    return status, waited


def profiler_read(reset: bool = True) -> dict:
    """{class: (launches, milliseconds)} accumulated since the last reset."""
    buf = (abi.McKernelTime * 16)()
    n = abi.load().mc_profiler_read(buf, 16, 1 if reset else 0)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].ms) for i in range(n)}


def mha_segments(Wq, Wk, H: int, alpha: float = 0.5):
    """QK-Clip segments of an MHA layer: head h owns rows [h d, (h+1) d)."""
    d = Wq.shape[0] // H
    return [ClipSegment(Wq, 0, d, d, alpha), ClipSegment(Wk, 0, d, d, 1.0 - alpha)]


def mla_segments(W_UQ, W_UKV, H: int, d_nope=128, d_rope=64, d_v=128):
    """QK-Clip segments of an MLA layer: q^C and k^C by sqrt(gamma), q^R by
    gamma; the shared rotary key (W_KR) and the value rows get none."""
    dq, dkv = d_nope + d_rope, d_nope + d_v
    return [ClipSegment(W_UQ, 0, dq, d_nope, 0.5), ClipSegment(W_UQ, d_nope, dq, d_rope, 1.0),
            ClipSegment(W_UKV, 0, dkv, d_nope, 0.5)]
