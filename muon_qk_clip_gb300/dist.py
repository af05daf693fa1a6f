"""Data-parallel MuonClip across ranks (one process per GPU).

Muon needs each whole matrix for Newton-Schulz, so the matrices are
partitioned across ranks (each rank owns whole matrices, balanced by
Newton-Schulz flops) and every rank runs the step on the matrices it owns;
owners then broadcast their updated weights.  This is the "gather whole
matrices" ZeRO-1 scheme of the zhihu "Muon's Infra Scalability" answer
(sections 2.1-2.2) with a partition that never splits a matrix.

QK-Clip needs S_max over the whole global batch ([K2-internals] "核心数学":
max over X in B), so the per-rank S_max vectors are combined with one
all-reduce(MAX) of H floats per layer before the step; every rank then makes
the same clip decision.

The collectives run through torch.distributed (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations

import heapq

import torch
import torch.distributed as dist

from .synth import flops_ns


def partition_matrices(shapes, world: int, steps: int = 5):
    """Greedy longest-processing-time assignment of whole matrices to ranks by
    Newton-Schulz flops.  Returns owner[i] for every matrix i; deterministic
    (ties broken by matrix index, then rank)."""
    order = sorted(range(len(shapes)), key=lambda i: (-flops_ns(*shapes[i], steps), i))
    heap = [(0.0, r) for r in range(world)]
    owner = [0] * len(shapes)
    for i in order:
        load, r = heapq.heappop(heap)
        owner[i] = r
        heapq.heappush(heap, (load + flops_ns(*shapes[i], steps), r))
    return owner


def allreduce_smax(smax: torch.Tensor, group=None) -> torch.Tensor:
    """In place: S_max^h = max over every rank's micro-batches."""
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(smax, op=dist.ReduceOp.MAX, group=group)
    return smax


def sharded_step(W, G, M, layers, step_fn, hp=None, group=None, owner=None):
    """One data-parallel MuonClip step.

    W, G, M: per-matrix tensors (every rank holds all weights; G is already
    averaged across ranks; M is only read and written on the owner).
    layers: list of (smax tensor, segments) where each segment is
    (matrix index, offset, stride, rows, exponent).  step_fn(idx, smax_list,
    segs_list) runs the local step on the matrices `idx` with the clip
    segments that point into them.  Returns the owner list."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if owner is None:
        owner = partition_matrices([tuple(w.shape) for w in W], world)
    for smax, _ in layers:
        allreduce_smax(smax, group)
    mine = [i for i in range(len(W)) if owner[i] == rank]
    local_layers = []
    for smax, segs in layers:
        local_layers.append((smax, [s for s in segs if owner[s[0]] == rank]))
    step_fn(mine, local_layers)
    if world > 1:
        for i, w in enumerate(W):
            src = owner[i] if group is None else dist.get_global_rank(group, owner[i])
            dist.broadcast(w, src=src, group=group)
    return owner
