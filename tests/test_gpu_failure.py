"""Failure detection on the GPU without a fault: the bounded device wait that
every tcgen05 kernel of the library uses for its mbarrier phases gives up on a
phase that nothing completes, reports MC_STATUS_TIMEOUT through the status
word, and leaves the context usable.  The wait is made to run out through
mc_selftest_bounded_wait (a flag that nothing sets); no kernel is broken on
purpose, nothing traps and every loop is bounded by %globaltimer."""
import numpy as np
import pytest
import torch

import oracle as O
from muon_qk_clip_gb300 import abi, build
from muon_qk_clip_gb300 import binding as mc
from muon_qk_clip_gb300 import synth
from tests.gpu_helpers import f64, rms

pytestmark = pytest.mark.gpu
MS = 1_000_000


def fp32(x):
    return float(np.float32(x))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    abi.load()


def test_wait_runs_out_of_budget():
    st, waited = mc.selftest_bounded_wait(20 * MS)
    torch.cuda.synchronize()
    assert st.item() & abi.MC_STATUS_TIMEOUT
    w = waited.item()
    assert 20 * MS <= w < 500 * MS, f"waited {w / MS:.2f} ms for a 20 ms budget"


def test_wait_gives_up_when_a_peer_raises_abort():
    st, waited = mc.selftest_bounded_wait(800 * MS, abort_after_ns=10 * MS)
    torch.cuda.synchronize()
    assert st.item() & abi.MC_STATUS_TIMEOUT
    w = waited.item()
    assert 10 * MS <= w < 400 * MS, f"waited {w / MS:.2f} ms; the abort came at 10 ms"


def test_status_bits_accumulate_and_context_stays_usable():
    """The status word is OR-ed (a second give-up keeps the bit, other bits
    stay), and the next call on the same stream computes correctly."""
    st = torch.full((1,), abi.MC_STATUS_NONFINITE_LOGIT, dtype=torch.int32, device="cuda")
    mc.selftest_bounded_wait(5 * MS, status=st)
    mc.selftest_bounded_wait(5 * MS, status=st)
    torch.cuda.synchronize()
    assert st.item() == abi.MC_STATUS_NONFINITE_LOGIT | abi.MC_STATUS_TIMEOUT
    M0 = synth.ns_test_matrix(256, 512, 0, "after_timeout")
    O_dev = torch.empty(256, 512, dtype=torch.float32, device="cuda")
    hp = mc.Hparams(ns_precision=abi.MC_NS_SPLIT_BF16)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.muon_newton_schulz([M0.cuda()], [O_dev], hp, status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    ohp = O.Hparams(rms_scale=fp32(hp.rms_scale), ns_coeffs=tuple(fp32(c) for c in hp.ns_coeffs),
                    ns_eps=fp32(hp.ns_eps), ns_steps=hp.ns_steps)
    ref = O.muon_direction(f64(M0), ohp)
    assert np.abs(f64(O_dev) - ref).max() <= 2e-2 * rms(ref)
