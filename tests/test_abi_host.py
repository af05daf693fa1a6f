"""Host-only checks of the C ABI: the library loads, exports every entry point
include/muonclip.h declares, its struct layouts match the ctypes mirror, and
argument errors are rejected on the host before any launch (these calls use
fake, aligned device addresses that are never dereferenced)."""
import ctypes
import os
import re
import subprocess

import pytest

from muon_qk_clip_gb300 import abi
from muon_qk_clip_gb300.abi import McAttnDesc, McAttnOut, McClipLayer, McClipSeg, McHparams, McMat

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muonclip.h")


@pytest.fixture(scope="module")
def lib():
    from muon_qk_clip_gb300 import build
    build.build()
    return abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_five_calls():
    fns = declared_functions()
    for name in ("muon_momentum", "muon_newton_schulz", "qk_max_logit", "qk_clip_apply",
                 "muonclip_step", "qk_attention_forward", "mc_workspace_size", "mc_last_error"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    missing = [f for f in declared_functions() if f not in exported]
    assert not missing, missing
    assert set(abi.SIGNATURES) <= exported


def test_struct_layouts_match_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(f'''
#include <stdio.h>
#include <stddef.h>
#include "{HEADER}"
int main(void) {{
  printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(mc_mat), sizeof(mc_hparams), sizeof(mc_clip_seg),
         sizeof(mc_clip_layer), sizeof(mc_attn_desc), sizeof(mc_attn_out));
  printf("%zu %zu %zu %zu %zu %zu\\n", offsetof(mc_attn_desc, q), offsetof(mc_attn_desc, ks_strides),
         offsetof(mc_clip_seg, exponent), offsetof(mc_hparams, ns_precision),
         offsetof(mc_attn_out, o), offsetof(mc_attn_out, lse));
  return 0;
}}''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", str(src), "-o", str(exe)], check=True)
    sizes, offs = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")[:2]
    assert [int(x) for x in sizes.split()] == [ctypes.sizeof(t) for t in
                                               (McMat, McHparams, McClipSeg, McClipLayer, McAttnDesc,
                                                McAttnOut)]
    assert [int(x) for x in offs.split()] == [McAttnDesc.q.offset, McAttnDesc.ks_strides.offset,
                                              McClipSeg.exponent.offset, McHparams.ns_precision.offset,
                                              McAttnOut.o.offset, McAttnOut.lse.offset]


def test_default_hparams(lib):
    h = McHparams()
    lib.mc_default_hparams(ctypes.byref(h))
    assert (h.mu, h.weight_decay, h.rms_scale, h.ns_steps, h.tau, h.alpha) == pytest.approx(
        (0.95, 0.1, 0.2, 5, 100.0, 0.5))
    assert (h.ns_a, h.ns_b, h.ns_c) == pytest.approx((3.4445, -4.7750, 2.0315))
    assert h.ns_fast_steps == 3
    assert lib.mc_version().decode().startswith("muonclip")


FAKE = 0x7f0000000000   # 256-byte aligned, never dereferenced


def m(rows, cols, dtype=abi.MC_F32, ld=None, ptr=FAKE):
    return McMat(ctypes.c_void_p(ptr), dtype, 0, rows, cols, cols if ld is None else ld)


def arr(*ms):
    a = (McMat * len(ms))()
    for i, x in enumerate(ms):
        a[i] = x
    return a


def hp(**kw):
    h = McHparams()
    abi.load().mc_default_hparams(ctypes.byref(h))
    for k, v in kw.items():
        setattr(h, k, v)
    return h


@pytest.mark.parametrize("bad,code", [
    (m(4, 8, ptr=0), abi.MC_ERR_INVALID_ARG),                 # null
    (m(4, 8, ptr=FAKE + 4), abi.MC_ERR_INVALID_ARG),          # misaligned
    (m(4, 8, ld=6), abi.MC_ERR_INVALID_ARG),                  # ld < cols
    (m(4, 6, ld=6), abi.MC_ERR_INVALID_ARG),                  # 24-byte pitch
    (m(0, 8), abi.MC_ERR_INVALID_ARG),                        # empty
    (m(4, 8, dtype=abi.MC_BF16), abi.MC_ERR_INVALID_ARG),     # momentum must be f32
    (m(4, 8, dtype=7), abi.MC_ERR_INVALID_ARG),               # unknown dtype
])
def test_momentum_rejects_bad_matrix(lib, bad, code):
    assert lib.muon_momentum(arr(bad), arr(m(4, 8)), 1, 0.9, None, None) == code
    assert lib.mc_last_error().decode()


def test_momentum_rejects_shape_mismatch_and_bad_mu(lib):
    assert lib.muon_momentum(arr(m(4, 8)), arr(m(4, 16)), 1, 0.9, None, None) == abi.MC_ERR_INVALID_ARG
    assert lib.muon_momentum(arr(m(4, 8)), arr(m(4, 8)), 1, float("nan"), None, None) == abi.MC_ERR_INVALID_ARG
    assert lib.muon_momentum(arr(m(4, 8)), arr(m(4, 8)), 0, 0.9, None, None) == abi.MC_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value", [("ns_steps", -1), ("ns_steps", 33), ("tau", 0.0),
                                         ("tau", -3.0), ("alpha", 1.5), ("ns_eps", -1.0),
                                         ("lr", float("inf")), ("ns_precision", 9),
                                         ("ns_fast_steps", -1), ("ns_fast_steps", 40),
                                         ("scale_mode", 3)])
def test_newton_schulz_rejects_bad_hparams(lib, field, value):
    h = hp(**{field: value})
    rc = lib.muon_newton_schulz(arr(m(64, 128)), arr(m(64, 128)), 1, ctypes.byref(h),
                                ctypes.c_void_p(FAKE), 1 << 30, None, None)
    assert rc == abi.MC_ERR_INVALID_ARG


def test_workspace_size_and_checks(lib):
    h = hp()
    n = ctypes.c_size_t(0)
    assert lib.mc_workspace_size(arr(m(64, 128), m(256, 64)), 2, ctypes.byref(h), ctypes.byref(n)) == 0
    need = n.value
    assert need > 4 * (64 * 128 + 64 * 256)
    hb = hp(ns_precision=abi.MC_NS_BF16)
    nb = ctypes.c_size_t(0)
    lib.mc_workspace_size(arr(m(64, 128), m(256, 64)), 2, ctypes.byref(hb), ctypes.byref(nb))
    assert nb.value < need
    M, O = arr(m(64, 128), m(256, 64)), arr(m(64, 128), m(256, 64))
    assert lib.muon_newton_schulz(M, O, 2, ctypes.byref(h), ctypes.c_void_p(FAKE), need - 1,
                                  None, None) == abi.MC_ERR_WORKSPACE
    assert lib.muon_newton_schulz(M, O, 2, ctypes.byref(h), None, need, None, None) == abi.MC_ERR_WORKSPACE
    assert lib.muon_newton_schulz(M, O, 2, ctypes.byref(h), ctypes.c_void_p(FAKE + 16), need,
                                  None, None) == abi.MC_ERR_WORKSPACE
    assert lib.muon_newton_schulz(M, arr(m(64, 128), m(64, 256)), 2, ctypes.byref(h),
                                  ctypes.c_void_p(FAKE), need, None, None) == abi.MC_ERR_INVALID_ARG


def attn(**kw):
    d = McAttnDesc()
    d.B, d.S, d.H, d.d_head, d.d_shared, d.dtype, d.causal = 1, 16, 2, 64, 0, abi.MC_BF16, 1
    d.scale = 0.125
    d.q = d.k = FAKE
    d.q_strides[:] = [16 * 2 * 64, 2 * 64, 64]
    d.k_strides[:] = [16 * 2 * 64, 2 * 64, 64]
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("kw,code", [
    (dict(S=0), abi.MC_ERR_INVALID_ARG), (dict(H=0), abi.MC_ERR_INVALID_ARG),
    (dict(d_head=0), abi.MC_ERR_INVALID_ARG), (dict(scale=0.0), abi.MC_ERR_INVALID_ARG),
    (dict(dtype=5), abi.MC_ERR_INVALID_ARG), (dict(q=None), abi.MC_ERR_INVALID_ARG),
    (dict(d_shared=64), abi.MC_ERR_INVALID_ARG),            # k_shared missing
    (dict(d_head=300), abi.MC_ERR_UNSUPPORTED),
])
def test_max_logit_rejects(lib, kw, code):
    d = attn(**kw)
    assert lib.qk_max_logit(ctypes.byref(d), ctypes.c_void_p(FAKE), None, 0, None, None) == code


def attn_out(**kw):
    o = McAttnOut()
    o.v = o.o = FAKE
    o.d_v = 64
    o.v_strides[:] = [16 * 2 * 64, 2 * 64, 64]
    o.o_strides[:] = [16 * 2 * 64, 2 * 64, 64]
    for k, v in kw.items():
        setattr(o, k, v)
    return o


@pytest.mark.parametrize("dkw,okw,code", [
    (dict(dtype=abi.MC_F32), {}, abi.MC_ERR_UNSUPPORTED),           # bf16 only
    (dict(S=0), {}, abi.MC_ERR_INVALID_ARG),
    (dict(scale=-1.0), {}, abi.MC_ERR_INVALID_ARG),
    ({}, dict(v=None), abi.MC_ERR_INVALID_ARG),
    ({}, dict(o=None), abi.MC_ERR_INVALID_ARG),
    (dict(d_head=256), {}, abi.MC_ERR_UNSUPPORTED),                 # q.k length > 192
    ({}, dict(d_v=256), abi.MC_ERR_UNSUPPORTED),
    (dict(d_head=96, d_shared=64, k_shared=FAKE), {}, abi.MC_ERR_UNSUPPORTED),  # split off a chunk
    ({}, dict(o=FAKE + 8), abi.MC_ERR_UNSUPPORTED),                 # misaligned output
])
def test_attention_forward_rejects(lib, dkw, okw, code):
    d, o = attn(**dkw), attn_out(**okw)
    assert lib.qk_attention_forward(ctypes.byref(d), ctypes.byref(o), ctypes.c_void_p(FAKE), 0,
                                    None, None) == code


def test_max_logit_argmax_rules(lib):
    d = attn()
    assert lib.qk_max_logit(ctypes.byref(d), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1,
                            None, None) == abi.MC_ERR_INVALID_ARG          # accumulate + argmax
    big = attn(B=2, S=65536)
    assert lib.qk_max_logit(ctypes.byref(big), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 0,
                            None, None) == abi.MC_ERR_UNSUPPORTED          # index overflow


def seg(w, off, stride, rows, e):
    return McClipSeg(w, off, stride, rows, e, 0)


def segarr(*ss):
    a = (McClipSeg * len(ss))()
    for i, s in enumerate(ss):
        a[i] = s
    return a


@pytest.mark.parametrize("s,H,tau,code", [
    (seg(m(64, 32), 0, 16, 16, 0.5), 5, 100.0, abi.MC_ERR_INVALID_ARG),   # runs past the rows
    (seg(m(64, 32), 0, 16, 16, 0.5), 0, 100.0, abi.MC_ERR_INVALID_ARG),   # H = 0
    (seg(m(64, 32), 0, 16, 16, 5.0), 4, 100.0, abi.MC_ERR_INVALID_ARG),   # exponent
    (seg(m(64, 32), -1, 16, 16, 0.5), 4, 100.0, abi.MC_ERR_INVALID_ARG),  # negative offset
    (seg(m(64, 32), 0, 16, 16, 0.5), 4, 0.0, abi.MC_ERR_INVALID_ARG),     # tau
])
def test_clip_rejects(lib, s, H, tau, code):
    assert lib.qk_clip_apply(ctypes.c_void_p(FAKE), H, tau, 0, segarr(s), 1, None, None, None, None) == code


def test_clip_rejects_unknown_mode(lib):
    s = seg(m(64, 32), 0, 16, 16, 0.5)
    assert lib.qk_clip_apply(ctypes.c_void_p(FAKE), 4, 100.0, 7, segarr(s), 1, None, None, None,
                             None) == abi.MC_ERR_INVALID_ARG


def test_step_rejects_mismatch_and_bad_layer(lib):
    h = hp()
    W, G, M = arr(m(64, 128, abi.MC_BF16)), arr(m(64, 128)), arr(m(64, 64))
    assert lib.muonclip_step(W, G, M, 1, ctypes.byref(h), None, 0, ctypes.c_void_p(FAKE), 1 << 30,
                             None, None) == abi.MC_ERR_INVALID_ARG
    L = (McClipLayer * 1)()
    L[0] = McClipLayer(None, 4, 0, None, None, None, 0, 0)
    assert lib.muonclip_step(W, G, arr(m(64, 128)), 1, ctypes.byref(h), L, 1, ctypes.c_void_p(FAKE),
                             1 << 30, None, None) == abi.MC_ERR_INVALID_ARG


def test_binding_raises_with_message(lib):
    with pytest.raises(abi.MuonClipError) as ei:
        abi.check(lib.muon_momentum(arr(m(4, 8, ptr=0)), arr(m(4, 8)), 1, 0.9, None, None), "muon_momentum")
    assert "null pointer" in str(ei.value)


@pytest.mark.parametrize("budget,abort_after,status,needle", [
    (0, 0, FAKE, "budget_ns"),
    (2_000_000_000, 0, FAKE, "budget_ns"),
    (1_000_000, 2_000_000_000, FAKE, "abort_after_ns"),
    (1_000_000, 0, None, "null status"),
])
def test_bounded_wait_selftest_rejects(lib, budget, abort_after, status, needle):
    st = None if status is None else ctypes.c_void_p(status)
    assert lib.mc_selftest_bounded_wait(budget, abort_after, st, None, None) == abi.MC_ERR_INVALID_ARG
    assert needle in lib.mc_last_error().decode()


# setup calls (Q/K projection): every rejection happens on the host, before a launch
P = ctypes.c_void_p(FAKE)


@pytest.mark.parametrize("args,needle", [
    ((P, 64, P, 64, P, 64, 4, 4, 64, 7, P, None, None), "dtype"),
    ((P, 64, P, 64, P, 64, 4, 4, 0, abi.MC_BF16, P, None, None), "K 0"),
    ((P, 32, P, 64, P, 64, 4, 4, 64, abi.MC_BF16, P, None, None), "pitch"),
    ((P, 68, P, 64, P, 64, 4, 4, 64, abi.MC_BF16, P, None, None), "16-byte"),
    ((ctypes.c_void_p(FAKE + 2), 64, P, 64, P, 64, 4, 4, 64, abi.MC_BF16, P, None, None), "16-byte"),
    ((P, 64, P, 64, P, 64, 4, 4, 64, abi.MC_BF16, None, None, None), "scratch"),
    ((None, 64, P, 64, P, 64, 4, 4, 64, abi.MC_F32, None, None, None), "null operand"),
])
def test_matmul_rejects(lib, args, needle):
    assert lib.mc_matmul(*args) == abi.MC_ERR_INVALID_ARG
    assert needle in lib.mc_last_error().decode()


def test_matmul_empty_is_a_no_op(lib):
    assert lib.mc_matmul(None, 64, None, 64, None, 64, 0, 4, 64, abi.MC_BF16, None, None, None) == abi.MC_OK


@pytest.mark.parametrize("args,needle", [
    ((P, 64, P, 64, 4, 64, 5, 1e-6, None), "dtype"),
    ((P, 32, P, 64, 4, 64, abi.MC_BF16, 1e-6, None), "pitches"),
    ((P, 64, P, 64, 4, 0, abi.MC_BF16, 1e-6, None), "cols 0"),
    ((P, 64, P, 64, 4, 64, abi.MC_BF16, -1.0, None), "eps"),
    ((None, 64, P, 64, 4, 64, abi.MC_BF16, 1e-6, None), "null"),
])
def test_rms_norm_rejects(lib, args, needle):
    assert lib.mc_rms_norm(*args) == abi.MC_ERR_INVALID_ARG
    assert needle in lib.mc_last_error().decode()


@pytest.mark.parametrize("args,needle", [
    ((P, 1, 8, 2, 63, 1024, 128, 64, abi.MC_BF16, 1e4, None), "d 63"),
    ((P, 1, 8, 0, 64, 1024, 128, 64, abi.MC_BF16, 1e4, None), "heads 0"),
    ((P, 1, 8, 2, 64, 1024, 128, 64, abi.MC_BF16, 0.0, None), "theta"),
    ((P, 1, 8, 2, 64, 1024, 128, 64, 9, 1e4, None), "dtype"),
    ((None, 1, 8, 2, 64, 1024, 128, 64, abi.MC_BF16, 1e4, None), "null"),
])
def test_rope_rejects(lib, args, needle):
    assert lib.mc_rope(*args) == abi.MC_ERR_INVALID_ARG
    assert needle in lib.mc_last_error().decode()
