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
