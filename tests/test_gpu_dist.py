"""ZeRO-1 MuonClip through the library in two ranks ("Muon's Infra
Scalability" sections 2.1-2.2 of the zhihu answer: reduce-scatter the
gradients, momentum on each rank's slice, boundary matrices gathered whole,
Newton-Schulz and the update of every matrix a rank owns a piece of, QK-Clip
with the S_max all-reduced over the ranks, all-gather of the parameters).

Both ranks run as processes on the one GPU (their kernels never wait on each
other); the collectives are gloo on host copies.  Two steps are compared with
two single-process oracle steps on the rank-averaged gradients, with fp32
weights (the library's fp32 Newton-Schulz, 1e-5 of the update's RMS)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O

pytestmark = pytest.mark.gpu

SHAPES = [(8, 8), (40, 40), (16, 24), (24, 16), (32, 20), (32, 20)]
SMAX = [[50.0, 300.0, 20.0, 90.0], [120.0, 80.0, 10.0, 95.0]]
SEGS = [(4, 0, 8, 8, 0.5), (5, 0, 8, 8, 0.5)]        # matrices 4 and 5: W_q, W_k of 4 heads


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def grads(rank, step):
    rng = np.random.default_rng(100 * step + rank)
    return [rng.standard_normal(s) for s in SHAPES]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from muon_qk_clip_gb300 import binding as mc
        from muon_qk_clip_gb300.dist import LibraryOps, Zero1Layout, zero1_state, zero1_step
        torch.cuda.set_device(0)
        rng = np.random.default_rng(0)
        W = [torch.tensor(rng.standard_normal(s) * 0.02, dtype=torch.float32, device="cuda") for s in SHAPES]
        L = Zero1Layout(SHAPES, world, align=64)
        M = zero1_state(L, device="cuda")
        hp = mc.Hparams()
        smaxes = []
        for step in range(2):
            G = [torch.tensor(g, dtype=torch.float32, device="cuda") for g in grads(rank, step)]
            smax = torch.tensor(SMAX[rank] if step == 0 else [10.0] * 4, device="cuda")
            zero1_step(W, G, M, L, [(smax, SEGS)], LibraryOps(W), hp)
            smaxes.append(smax.cpu().numpy().copy())
        torch.cuda.synchronize()
        out[rank] = ([w.cpu().double().numpy() for w in W], M.cpu().double().numpy(), smaxes)
    finally:
        dist.destroy_process_group()


def test_zero1_two_ranks_through_the_library_match_the_oracle():
    from muon_qk_clip_gb300 import build
    from muon_qk_clip_gb300 import binding as mc
    from muon_qk_clip_gb300.dist import Zero1Layout
    build.build()
    world, port = 2, free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    hp = mc.Hparams()
    f32 = lambda x: float(np.float32(x))  # noqa: E731
    ohp = O.Hparams(mu=f32(hp.mu), lr=f32(hp.lr), weight_decay=f32(hp.weight_decay),
                    rms_scale=f32(hp.rms_scale), ns_coeffs=tuple(f32(c) for c in hp.ns_coeffs),
                    ns_eps=f32(hp.ns_eps))
    rng = np.random.default_rng(0)
    W = {str(i): O.round_to_f32(rng.standard_normal(s) * 0.02) for i, s in enumerate(SHAPES)}
    M = {k: np.zeros_like(v) for k, v in W.items()}
    segs = [O.ClipSegment("4", 0, 8, 8, 0.5), O.ClipSegment("5", 0, 8, 8, 0.5)]
    upd = 0.0
    for step in range(2):
        gr = [[O.round_to_f32(g) for g in grads(r, step)] for r in range(world)]
        G = {str(i): sum(g[i] for g in gr) / world for i in range(len(SHAPES))}
        smax = np.max(np.array(SMAX), axis=0) if step == 0 else np.full(4, 10.0)
        for r in range(world):
            np.testing.assert_array_equal(out[r][2][step], smax)
        W_prev = W
        W, M, _ = O.muonclip_step(W, G, M, ohp, [(smax, segs)])
        upd = max(upd, max(float(np.sqrt(np.mean((W[k] - W_prev[k]) ** 2))) for k in W))
    L = Zero1Layout(SHAPES, world, align=64)
    flat_m = np.zeros(L.shard * world)
    for i in range(len(SHAPES)):
        flat_m[L.offsets[i]:L.offsets[i] + L.numel(i)] = M[str(i)].reshape(-1)
    # fp32 storage of W and M, the fp32 Newton-Schulz at 1e-5 of the update,
    # and the clip's gamma in fp32: 5e-8 absolute on weights of ~0.02 whose
    # per-step update is ~1e-4 (a missed or doubled update is off by ~1e-4)
    for r in range(world):
        w_r, m_r, _ = out[r]
        for i in range(len(SHAPES)):
            np.testing.assert_allclose(w_r[i], W[str(i)], rtol=0, atol=5e-8)
        lo, hi = L.slice(r)
        np.testing.assert_allclose(m_r, flat_m[lo:hi], rtol=2e-6, atol=1e-6)
    assert upd > 1e-5
    assert any(len(L.pieces(i)) > 1 for i in range(len(SHAPES)))   # boundary matrices occurred
    for a, b in zip(out[0][0], out[1][0]):                         # both ranks end identical
        np.testing.assert_array_equal(a, b)
