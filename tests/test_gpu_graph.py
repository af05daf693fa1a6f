"""A whole MuonClip step (max logit + muonclip_step with the clip) captured in
a CUDA graph and replayed equals the same steps run eagerly, bit for bit: the
library's launches, its tile-counter memset and its second Newton-Schulz
stream (forked and joined with events) are all capturable."""
import pytest
import torch

from muon_qk_clip_gb300 import build
from muon_qk_clip_gb300 import binding as mc
from muon_qk_clip_gb300 import forward, synth

pytestmark = pytest.mark.gpu


def _setup(seed):
    wl = synth.scaled(synth.workload("dense_block"), B=1, S=512)
    names = ["Wq", "Wk", "W_up", "W_down"]
    W, G, M = synth.muon_inputs(wl, seed=seed, only=names, device="cuda")
    X, _ = synth.attention_inputs(wl, seed=seed, device="cuda")
    q, k = forward.project_mha(X, W["Wq"], W["Wk"], 16)
    return ([W[n] for n in names], [G[n] for n in names], [M[n] for n in names],
            q.contiguous(), k.contiguous())


def test_step_in_cuda_graph_equals_eager():
    build.build()
    hp = mc.Hparams()
    # eager: two steps
    We, Ge, Me, qe, ke = _setup(19)
    ws_e = mc.alloc_workspace(We, hp, "cuda")
    sm_e = torch.empty(16, device="cuda")
    for _ in range(2):
        mc.qk_max_logit(qe, ke, smax=sm_e)
        mc.muonclip_step(We, Ge, Me, hp, layers=[mc.ClipLayer(sm_e, mc.mha_segments(We[0], We[1], 16))],
                         workspace=ws_e)
    torch.cuda.synchronize()
    # graph: capture one step, replay twice
    Wg, Gg, Mg, qg, kg = _setup(19)
    ws_g = mc.alloc_workspace(Wg, hp, "cuda")
    sm_g = torch.empty(16, device="cuda")
    layer = mc.ClipLayer(sm_g, mc.mha_segments(Wg[0], Wg[1], 16))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        mc.qk_max_logit(qg, kg, smax=torch.empty(16, device="cuda"))   # warm-up outside the graph
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            mc.qk_max_logit(qg, kg, smax=sm_g, stream=side)
            mc.muonclip_step(Wg, Gg, Mg, hp, layers=[layer], workspace=ws_g, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(We + Me, Wg + Mg):
        assert torch.equal(a, b)
    assert torch.equal(sm_e, sm_g)
