"""Multi-rank host logic on CPU (gloo, world size 2): the S_max MAX all-reduce,
the matrix partition, and a sharded MuonClip step whose result equals the
single-process step.  The per-rank step here is the CPU oracle; on GPUs it is
the library's muonclip_step."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
from muon_qk_clip_gb300.dist import partition_matrices, sharded_step
from muon_qk_clip_gb300.synth import flops_ns


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_partition_balances_and_is_deterministic():
    shapes = [(2048, 2048)] * 4 + [(5632, 2048)] * 2 + [(2048, 5632)]
    owner = partition_matrices(shapes, 2)
    assert owner == partition_matrices(shapes, 2)
    loads = [sum(flops_ns(*shapes[i]) for i in range(len(shapes)) if owner[i] == r) for r in range(2)]
    assert max(loads) / min(loads) < 1.25
    assert partition_matrices(shapes, 1) == [0] * len(shapes)
    moe = [(2048, 7168)] * 64 + [(7168, 2048)] * 64
    assert sorted(np.bincount(partition_matrices(moe, 8))) == [16] * 8


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(0)               # same weights on every rank
        shapes = [(16, 24), (24, 16), (32, 32), (8, 40)]
        W = [torch.tensor(rng.standard_normal(s) * 0.02) for s in shapes]
        G = [torch.tensor(rng.standard_normal(s)) for s in shapes]
        M = [torch.zeros(s, dtype=torch.float64) for s in shapes]
        # each rank saw a different micro-batch: local S_max differ
        local = np.array([[50.0, 300.0], [120.0, 80.0]])[rank]
        smax = torch.tensor(local)
        H, d = 2, 8
        segs = [(0, 0, d, d, 0.5), (2, 0, 16, 16, 0.5)]
        hp = O.Hparams()

        def step_fn(idx, layers):
            for i in idx:
                Wn, Mn, _ = O.muon_step(W[i].numpy(), G[i].numpy(), M[i].numpy(), hp)
                W[i].copy_(torch.tensor(Wn)); M[i].copy_(torch.tensor(Mn))
            for sm, sg in layers:
                gamma, mask = O.clip_factors(sm.numpy(), hp.tau)
                for (i, off, stride, rows, e) in sg:
                    for h in np.nonzero(mask)[0]:
                        W[i][off + h * stride: off + h * stride + rows] *= gamma[h] ** e

        sharded_step(W, G, M, [(smax, segs)], step_fn)
        out[rank] = ([w.numpy().copy() for w in W], smax.numpy().copy())
    finally:
        dist.destroy_process_group()


def test_sharded_step_matches_single_process():
    world, port = 2, free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    w0, s0 = out[0]
    w1, s1 = out[1]
    np.testing.assert_array_equal(s0, [120.0, 300.0])   # global max over both ranks
    np.testing.assert_array_equal(s1, s0)
    for a, b in zip(w0, w1):                              # every rank ends identical
        np.testing.assert_array_equal(a, b)
    # equal to the single-process oracle step with the global S_max
    rng = np.random.default_rng(0)
    shapes = [(16, 24), (24, 16), (32, 32), (8, 40)]
    W = {str(i): rng.standard_normal(s) * 0.02 for i, s in enumerate(shapes)}
    G = {str(i): rng.standard_normal(s) for i, s in enumerate(shapes)}
    M = {k: np.zeros_like(v) for k, v in W.items()}
    segs = [O.ClipSegment("0", 0, 8, 8, 0.5), O.ClipSegment("2", 0, 16, 16, 0.5)]
    Wn, _, _ = O.muonclip_step(W, G, M, O.Hparams(), [(np.array([120.0, 300.0]), segs)])
    for i in range(len(shapes)):
        np.testing.assert_allclose(w0[i], Wn[str(i)], rtol=0, atol=1e-15)


# ------------------------------------------------------------------ ZeRO-1
from muon_qk_clip_gb300.dist import Zero1Layout, zero1_state, zero1_step   # noqa: E402


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7])
def test_zero1_layout_owns_every_element_once(world):
    rng = np.random.default_rng(world)
    shapes = [tuple(int(x) for x in rng.integers(1, 70, 2)) for _ in range(9)] + [(40, 40)]
    L = Zero1Layout(shapes, world)
    assert L.shard % L.align == 0 and L.shard * world >= L.total
    for i in range(len(shapes)):
        assert L.offsets[i] % L.align == 0
        pcs = L.pieces(i)
        # contiguous, in rank order, covering [0, numel) exactly once
        assert pcs[0][1] == 0 and pcs[-1][2] == L.numel(i)
        for (r0, _, h0), (r1, l1, _) in zip(pcs, pcs[1:]):
            assert r1 == r0 + 1 and l1 == h0
        assert (len(pcs) > 1) == (i in L.boundary())
        for r, lo, hi in pcs:
            s0, s1 = L.slice(r)
            assert s0 <= L.offsets[i] + lo and L.offsets[i] + hi <= s1
    owned = sum(hi - lo for r in range(world) for i in range(len(shapes))
                for (rr, lo, hi) in L.pieces(i) if rr == r)
    assert owned == sum(L.numel(i) for i in range(len(shapes)))


def test_zero1_layout_matrix_across_three_ranks():
    L = Zero1Layout([(8, 8), (40, 40), (16, 24)], 3)
    assert [p[0] for p in L.pieces(1)] == [0, 1, 2]
    assert L.boundary() == [1] and L.touched(1) == [1]


class _OracleOps:
    """zero1_step's per-rank operations done by the CPU oracle (fp64)."""

    def __init__(self, W):
        self.W = W

    def momentum(self, M, G, hp):
        M.copy_(torch.from_numpy(O.momentum(M.numpy(), G.numpy(), hp.mu)))

    def step(self, Ws, mfull, layers, hp):
        for w, m in zip(Ws, mfull):
            Od = O.muon_direction(m.numpy(), hp)
            w.copy_(torch.from_numpy(O.muon_apply(w.numpy(), Od, hp.lr, hp.weight_decay)))
        self.clip(layers, hp)

    def clip(self, layers, hp):
        for smax, segs in layers:
            gamma, mask = O.clip_factors(smax.numpy(), hp.tau)
            for (i, off, stride, rows, e) in segs:
                for h in np.nonzero(mask)[0]:
                    self.W[i][off + h * stride: off + h * stride + rows] *= gamma[h] ** e


Z_SHAPES = [(8, 8), (40, 40), (16, 24), (24, 16), (32, 20), (32, 20)]
Z_SMAX = [[50.0, 300.0, 20.0, 90.0], [120.0, 80.0, 10.0, 95.0], [60.0, 70.0, 30.0, 99.0]]
Z_SEGS = [(4, 0, 8, 8, 0.5), (5, 0, 8, 8, 0.5)]      # matrices 4 and 5: W_q, W_k of 4 heads


def _z_inputs(rank, step):
    rng = np.random.default_rng(100 * step + rank)
    return [rng.standard_normal(s) for s in Z_SHAPES]


def _zero1_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(0)
        W = [torch.tensor(rng.standard_normal(s) * 0.02) for s in Z_SHAPES]
        L = Zero1Layout(Z_SHAPES, world, align=16)
        M = zero1_state(L, dtype=torch.float64)
        hp = O.Hparams()
        ops = _OracleOps(W)
        smaxes = []
        for step in range(2):
            G = [torch.tensor(g) for g in _z_inputs(rank, step)]
            smax = torch.tensor(Z_SMAX[rank] if step == 0 else [10.0, 10.0, 10.0, 10.0])
            zero1_step(W, G, M, L, [(smax, Z_SEGS)], ops, hp)
            smaxes.append(smax.numpy().copy())
        out[rank] = ([w.numpy().copy() for w in W], M.numpy().copy(), smaxes)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_zero1_step_matches_single_process(world):
    port = free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_zero1_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    # the reference: two single-process MuonClip steps on the averaged gradients
    rng = np.random.default_rng(0)
    W = {str(i): rng.standard_normal(s) * 0.02 for i, s in enumerate(Z_SHAPES)}
    M = {k: np.zeros_like(v) for k, v in W.items()}
    segs = [O.ClipSegment("4", 0, 8, 8, 0.5), O.ClipSegment("5", 0, 8, 8, 0.5)]
    for step in range(2):
        grads = [_z_inputs(r, step) for r in range(world)]
        G = {str(i): sum(g[i] for g in grads) / world for i in range(len(Z_SHAPES))}
        smax = np.max(np.array(Z_SMAX[:world]), axis=0) if step == 0 else np.full(4, 10.0)
        W, M, _ = O.muonclip_step(W, G, M, O.Hparams(), [(smax, segs)])
        for r in range(world):
            np.testing.assert_array_equal(out[r][2][step], smax)
    L = Zero1Layout(Z_SHAPES, world, align=16)
    flat_m = np.zeros(L.shard * world)
    for i in range(len(Z_SHAPES)):
        flat_m[L.offsets[i]:L.offsets[i] + L.numel(i)] = M[str(i)].reshape(-1)
    for r in range(world):
        w_r, m_r, _ = out[r]
        for i in range(len(Z_SHAPES)):
            np.testing.assert_allclose(w_r[i], W[str(i)], rtol=0, atol=1e-14)
        lo, hi = L.slice(r)
        np.testing.assert_allclose(m_r, flat_m[lo:hi], rtol=0, atol=1e-14)
    assert any(len(L.pieces(i)) > 1 for i in range(len(Z_SHAPES)))   # boundary matrices occurred
