"""The tensor-core Newton-Schulz result does not depend on how its tiles are
scheduled: dynamic or round-robin tile order, one or two streams, single CTAs,
B-multicast clusters or CTA pairs (for every launch, the default, or the
one-product ones),
32- or 64-deep one-product k-steps give bit-identical outputs (every output
tile is computed by the same sequence of MMAs whichever CTA or stream takes
it).  The 1024 x 1152 matrix takes the one-product leading iterations.  The
switches are read once per process, so each variant runs in a subprocess."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
from muon_qk_clip_gb300 import binding as mc, synth
shapes = [(640, 384), (384, 640), (256, 256), (1000, 520), (520, 1000), (96, 136), (1024, 1152)]
G = [synth.normal(s, 1e-3, f"sg{i}", 71).cuda() for i, s in enumerate(shapes)]
O = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in shapes]
st = torch.zeros(1, dtype=torch.int32, device="cuda")
mc.muon_newton_schulz(G, O, mc.Hparams(ns_precision=1), status=st)
torch.cuda.synchronize()
assert st.item() == 0
np.savez(sys.argv[2], *[o.view(torch.int16).cpu().numpy() for o in O])
'''

VARIANTS = {
    "default": {},
    "static": {"MC_NS_SCHED": "static"},
    "one_stream": {"MC_NS_STREAMS": "1"},
    "single_cta": {"MC_NS_CTA": "1"},
    "cta_pairs": {"MC_NS_CTA": "2"},
    "clusters": {"MC_NS_PAIR": "none"},
    "pairs_fast": {"MC_NS_PAIR": "fast"},
    "pairs_all": {"MC_NS_PAIR": "all"},
    "pairs_fast_bk32": {"MC_NS_PAIR": "fast", "MC_NS_BK_FAST": "32"},
    "clusters_bk32": {"MC_NS_PAIR": "none", "MC_NS_BK_FAST": "32"},
    "bk32": {"MC_NS_BK_FAST": "32"},
}


def test_newton_schulz_bit_identical_across_schedules(tmp_path):
    from muon_qk_clip_gb300 import build
    build.build()
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    outs = {}
    for name, env in VARIANTS.items():
        out = tmp_path / f"{name}.npz"
        e = dict(os.environ, **env)
        subprocess.run([sys.executable, str(script), ROOT, str(out)], env=e, check=True, timeout=300)
        z = np.load(out)
        outs[name] = [z[k] for k in sorted(z.files, key=lambda k: int(k.split("_")[1]))]
    ref = outs["default"]
    for name, got in outs.items():
        for i, (a, b) in enumerate(zip(ref, got)):
            assert np.array_equal(a, b), f"{name}: matrix {i} differs"
