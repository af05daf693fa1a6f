"""muon_newton_schulz_noalloc: the Newton-Schulz entry point for callers that
cannot give the library device memory (an allocator that owns the GPU's
memory, a loop that cannot afford cudaFree's device-wide synchronisation, a
plugin without an allocator).  Its scratch is a fixed array inside the
library, so these tests check that two calls in a row, each reusing whatever
the previous call left in that array, give the same results as the
workspace entry point, bit for bit: both run the same kernels on the same
plan, so any difference would be a stale read of the shared array.  The
larger call goes first, so the second runs over its leftovers.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from muon_qk_clip_gb300 import abi, build
from muon_qk_clip_gb300 import binding as mc
from muon_qk_clip_gb300 import synth


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def noalloc(lib, M, O, hp, status=None):
    hc = hp.c()
    rc = lib.muon_newton_schulz_noalloc(mc._mats(M), mc._mats(O), len(M), ctypes.byref(hc),
                                        None if status is None else ctypes.c_void_p(status.data_ptr()),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    abi.check(rc, "muon_newton_schulz_noalloc")


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    assert torch.cuda.is_available()
    hp = mc.Hparams()
    calls = [
        ([(512, 1024), (1024, 512), (256, 256)], torch.float32, 21),
        ([(384, 640), (200, 328)], torch.bfloat16, 22),
    ]
    for shapes, odt, seed in calls:
        M = [synth.ns_test_matrix(r, c, seed, f"na{i}").cuda() for i, (r, c) in enumerate(shapes)]
        O_na = [torch.full(s, float("nan"), dtype=odt, device="cuda") for s in shapes]
        O_ws = [torch.full(s, float("nan"), dtype=odt, device="cuda") for s in shapes]
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        noalloc(lib, M, O_na, hp, st)
        mc.muon_newton_schulz(M, O_ws, hp)
        torch.cuda.synchronize()
        assert st.item() == 0
        for a, b in zip(O_na, O_ws):
            assert torch.isfinite(a).all()
            assert torch.equal(a, b)


def test_noalloc_rejects_oversize_before_any_launch(lib):
    """A request beyond the static scratch is refused on the host with
    MC_ERR_WORKSPACE (no device needed: nothing is launched)."""
    fake = 0x7f0000000000
    m = abi.McMat(ctypes.c_void_p(fake), abi.MC_F32, 0, 2048, 4096, 4096)
    arr = (abi.McMat * 1)(m)
    out = (abi.McMat * 1)(m)
    hc = mc.Hparams().c()
    rc = lib.muon_newton_schulz_noalloc(arr, out, 1, ctypes.byref(hc), None, None)
    assert rc == abi.MC_ERR_WORKSPACE
    assert "static" in lib.mc_last_error().decode()
    need = mc.workspace_size([(2048, 4096)])
    assert need > abi.MC_NOALLOC_SCRATCH_BYTES
