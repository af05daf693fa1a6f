"""MuonClip (Muon + per-head QK-Clip) optimizer step for GB300 (sm_103a).

The compute lives in libmuonclip.so (CUDA, built by muon_qk_clip_gb300.build);
this package is its binding plus seeded synthetic inputs for tests and the
benchmark.
"""
from .abi import MuonClipError  # noqa: F401
from .binding import (ClipLayer, ClipSegment, Hparams, alloc_workspace,  # noqa: F401
                      default_hparams, mha_segments, mla_segments, muon_momentum,
                      muon_newton_schulz, muonclip_step, qk_attention_forward, qk_clip_apply,
                      qk_max_logit, workspace_size)

__all__ = ["ClipLayer", "ClipSegment", "Hparams", "MuonClipError", "alloc_workspace",
           "default_hparams", "mha_segments", "mla_segments", "muon_momentum",
           "muon_newton_schulz", "muonclip_step", "qk_attention_forward", "qk_clip_apply",
           "qk_max_logit", "workspace_size"]
