"""ctypes mirror of include/muonclip.h and loader for the in-tree libmuonclip.so.

Argument marshalling only: every step of the MuonClip path runs in the CUDA
library.  If the library is missing this module raises; there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmuonclip.so")

MC_OK, MC_ERR_INVALID_ARG, MC_ERR_UNSUPPORTED, MC_ERR_WORKSPACE, MC_ERR_CUDA, \
    MC_ERR_NONFINITE, MC_ERR_TIMEOUT = range(7)
STATUS_NAMES = {0: "MC_OK", 1: "MC_ERR_INVALID_ARG", 2: "MC_ERR_UNSUPPORTED", 3: "MC_ERR_WORKSPACE",
                4: "MC_ERR_CUDA", 5: "MC_ERR_NONFINITE", 6: "MC_ERR_TIMEOUT"}

MC_STATUS_NONFINITE_UPDATE = 1
MC_STATUS_NONFINITE_LOGIT = 2
MC_STATUS_NONFINITE_SMAX = 4
MC_STATUS_TIMEOUT = 8

MC_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

MC_F32, MC_BF16 = 0, 1
MC_NS_AUTO, MC_NS_SPLIT_BF16, MC_NS_BF16, MC_NS_FP32 = 0, 1, 2, 3
MC_SCALE_RMS, MC_SCALE_SPECTRAL = 0, 1
MC_CLIP_PER_HEAD, MC_CLIP_TOTAL = 0, 1


class McMat(ctypes.Structure):
    _fields_ = [("ptr", c_void_p), ("dtype", c_int32), ("_pad", c_int32),
                ("rows", c_int64), ("cols", c_int64), ("ld", c_int64)]


class McHparams(ctypes.Structure):
    _fields_ = [("mu", c_float), ("lr", c_float), ("weight_decay", c_float), ("rms_scale", c_float),
                ("ns_steps", c_int32), ("ns_a", c_float), ("ns_b", c_float), ("ns_c", c_float),
                ("ns_eps", c_float), ("tau", c_float), ("alpha", c_float), ("ns_precision", c_int32),
                ("ns_fast_steps", c_int32), ("scale_mode", c_int32)]


class McClipSeg(ctypes.Structure):
    _fields_ = [("w", McMat), ("head_row_offset", c_int64), ("head_row_stride", c_int64),
                ("rows_per_head", c_int64), ("exponent", c_float), ("_pad", c_int32)]


class McClipLayer(ctypes.Structure):
    _fields_ = [("smax", c_void_p), ("H", c_int32), ("nsegs", c_int32),
                ("segs", POINTER(McClipSeg)), ("gamma_out", c_void_p), ("nclipped", c_void_p),
                ("mode", c_int32), ("_pad", c_int32)]


class McAttnDesc(ctypes.Structure):
    _fields_ = [("B", c_int32), ("S", c_int32), ("H", c_int32), ("d_head", c_int32),
                ("d_shared", c_int32), ("dtype", c_int32), ("causal", c_int32), ("scale", c_float),
                ("q", c_void_p), ("k", c_void_p), ("k_shared", c_void_p),
                ("q_strides", c_int64 * 3), ("k_strides", c_int64 * 3), ("ks_strides", c_int64 * 2)]


class McAttnOut(ctypes.Structure):
    _fields_ = [("v", c_void_p), ("d_v", c_int32), ("_pad", c_int32), ("v_strides", c_int64 * 3),
                ("o", c_void_p), ("o_strides", c_int64 * 3), ("lse", c_void_p)]


class McKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", c_int32), ("ms", c_float)]


# name -> (restype, argtypes), exactly the declarations of include/muonclip.h
SIGNATURES = {
    "mc_default_hparams": (None, [POINTER(McHparams)]),
    "mc_workspace_size": (c_int32, [POINTER(McMat), c_int32, POINTER(McHparams), POINTER(c_size_t)]),
    "mc_ns_products": (c_int32, [POINTER(McHparams), c_int64, c_int64, c_void_p]),
    "muon_momentum": (c_int32, [POINTER(McMat), POINTER(McMat), c_int32, c_float, c_void_p, c_void_p]),
    "muon_newton_schulz": (c_int32, [POINTER(McMat), POINTER(McMat), c_int32, POINTER(McHparams),
                                     c_void_p, c_size_t, c_void_p, c_void_p]),
    "muon_newton_schulz_noalloc": (c_int32, [POINTER(McMat), POINTER(McMat), c_int32,
                                             POINTER(McHparams), c_void_p, c_void_p]),
    "qk_max_logit": (c_int32, [POINTER(McAttnDesc), c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
    "qk_attention_forward": (c_int32, [POINTER(McAttnDesc), POINTER(McAttnOut), c_void_p, c_int32,
                                       c_void_p, c_void_p]),
    "qk_clip_apply": (c_int32, [c_void_p, c_int32, c_float, c_int32, POINTER(McClipSeg), c_int32,
                                c_void_p, c_void_p, c_void_p, c_void_p]),
    "muonclip_step": (c_int32, [POINTER(McMat), POINTER(McMat), POINTER(McMat), c_int32,
                                POINTER(McHparams), POINTER(McClipLayer), c_int32, c_void_p,
                                c_size_t, c_void_p, c_void_p]),
    "mc_matmul": (c_int32, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64, c_int32, c_int32,
                            c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    "mc_rms_norm": (c_int32, [c_void_p, c_int64, c_void_p, c_int64, c_int64, c_int32, c_int32, c_float,
                              c_void_p]),
    "mc_rope": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_int32, c_int64, c_int64, c_int64, c_int32,
                          c_double, c_void_p]),
    "mc_selftest_bounded_wait": (c_int32, [c_uint64, c_uint64, c_void_p, c_void_p, c_void_p]),
    "mc_profiler_enable": (None, [c_int32]),
    "mc_profiler_read": (c_int32, [POINTER(McKernelTime), c_int32, c_int32]),
    "mc_last_error": (c_char_p, []),
    "mc_version": (c_char_p, []),
}

_lib = None


def load():
    """Load libmuonclip.so and declare every entry point; raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built: run `python -m muon_qk_clip_gb300.build` "
                "(nvcc, sm_103a). There is no non-CUDA implementation.")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class MuonClipError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


def check(code: int, where: str):
    if code != MC_OK:
        raise MuonClipError(code, where, load().mc_last_error().decode())
