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

The collectives run through torch.distributed: NCCL on device tensors, or
gloo, which takes host tensors (device tensors then go through host copies,
so ranks sharing one GPU can run the library with gloo collectives).
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


def _host_staged(t: torch.Tensor, group) -> bool:
    """gloo collectives take host tensors: a device tensor is staged."""
    return t.device.type != "cpu" and dist.get_backend(group) == "gloo"


def _all_reduce(t: torch.Tensor, op, group=None):
    if _host_staged(t, group):
        h = t.cpu()
        dist.all_reduce(h, op=op, group=group)
        t.copy_(h)
    else:
        dist.all_reduce(t, op=op, group=group)


def _all_gather(bufs, t: torch.Tensor, group=None):
    if _host_staged(t, group):
        hb = [torch.empty(b.shape, dtype=b.dtype) for b in bufs]
        dist.all_gather(hb, t.cpu(), group=group)
        for b, h in zip(bufs, hb):
            b.copy_(h)
    else:
        dist.all_gather(bufs, t, group=group)


def allreduce_smax(smax: torch.Tensor, group=None) -> torch.Tensor:
    """In place: S_max^h = max over every rank's micro-batches."""
    if dist.is_available() and dist.is_initialized():
        _all_reduce(smax, dist.ReduceOp.MAX, group)
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
            if _host_staged(w, group):
                h = w.cpu()
                dist.broadcast(h, src=src, group=group)
                w.copy_(h)
            else:
                dist.broadcast(w, src=src, group=group)
    return owner


# ---------------------------------------------------------------------------
# ZeRO-1 over a flat concatenation of the Muon parameters
# ---------------------------------------------------------------------------
#
# The zhihu answer on Muon's infrastructure scalability (section 2.1) gives the
# ZeRO-1 optimizer lifecycle: reduce-scatter the gradients so each data-
# parallel rank holds its slice, update the slice, all-gather the parameters.
# Section 2.2 describes the flat-concatenated layout (all optimizer states
# flattened, concatenated and cut evenly across ranks) and, for Muon, the
# "gather" method used for matrices cut by a slice boundary: every rank that
# owns a piece gathers the whole momentum matrix, runs Newton-Schulz on all of
# it and keeps only its own piece.  Matrices inside one slice need nothing
# extra.  zero1_step follows those steps; QK-Clip adds the S_max all-reduce
# (MAX) and a clip that every rank applies identically.
#
# Every parameter starts at a multiple of `align` elements in the flat buffer
# (padding, never owned data), so each slice and every matrix inside it starts
# 16-byte aligned for the library's loads.


class Zero1Layout:
    """Flat layout of the Muon matrices across `world` ranks."""

    def __init__(self, shapes, world: int, align: int = 64):
        self.shapes = [tuple(int(x) for x in s) for s in shapes]
        self.world = int(world)
        self.align = int(align)
        self.offsets, off = [], 0
        for r, c in self.shapes:
            self.offsets.append(off)
            off += -(-(r * c) // align) * align
        self.total = off
        per = -(-off // self.world) if off else 0
        self.shard = -(-per // align) * align         # elements per rank

    def numel(self, i):
        r, c = self.shapes[i]
        return r * c

    def slice(self, rank):
        return rank * self.shard, (rank + 1) * self.shard

    def pieces(self, i):
        """[(rank, lo, hi)] of matrix i: element range [lo, hi) of the
        flattened matrix owned by each rank, in rank order."""
        a, n = self.offsets[i], self.numel(i)
        out = []
        if self.shard == 0:
            return out
        for r in range(a // self.shard, (a + n - 1) // self.shard + 1):
            s0, s1 = self.slice(r)
            lo, hi = max(a, s0) - a, min(a + n, s1) - a
            if hi > lo:
                out.append((r, lo, hi))
        return out

    def touched(self, rank):
        return [i for i in range(len(self.shapes)) if any(p[0] == rank for p in self.pieces(i))]

    def boundary(self):
        return [i for i in range(len(self.shapes)) if len(self.pieces(i)) > 1]

    def pack_order(self, rank):
        """(matrix, lo, hi) of every boundary piece this rank owns, in matrix order."""
        return [(i, lo, hi) for i in self.boundary() for (r, lo, hi) in self.pieces(i) if r == rank]


def zero1_state(layout: Zero1Layout, device=None, dtype=torch.float32):
    """This rank's momentum slice (zeros), `layout.shard` elements."""
    return torch.zeros(layout.shard, dtype=dtype, device=device)


def _flat(tensors, layout: Zero1Layout, dtype):
    flat = torch.zeros(layout.shard * layout.world, dtype=dtype, device=tensors[0].device)
    for i, t in enumerate(tensors):
        a = layout.offsets[i]
        flat[a:a + t.numel()].copy_(t.reshape(-1))
    return flat


def _reduce_scatter_mean(flat, layout: Zero1Layout, rank, group):
    """This rank's slice of the average of every rank's flat buffer."""
    world = layout.world
    if world == 1:
        return flat.clone()
    out = torch.empty(layout.shard, dtype=flat.dtype, device=flat.device)
    if dist.get_backend(group) == "nccl":
        dist.reduce_scatter_tensor(out, flat, op=dist.ReduceOp.SUM, group=group)
    else:                          # gloo has no reduce-scatter: all-reduce, keep the slice
        _all_reduce(flat, dist.ReduceOp.SUM, group)
        lo, hi = layout.slice(rank)
        out.copy_(flat[lo:hi])
    return out.div_(world)


def _gather_boundary(M_shard, layout: Zero1Layout, rank, group):
    """Full momentum of every boundary matrix this rank touches: one
    all-gather of each rank's packed boundary pieces."""
    world = layout.world
    lo_r = layout.slice(rank)[0]
    sizes = [sum(hi - lo for _, lo, hi in layout.pack_order(r)) for r in range(world)]
    width = max(sizes) if sizes else 0
    if width == 0 or world == 1:
        return {}
    pack = torch.zeros(width, dtype=M_shard.dtype, device=M_shard.device)
    pos = 0
    for i, lo, hi in layout.pack_order(rank):
        a = layout.offsets[i] + lo - lo_r
        pack[pos:pos + hi - lo].copy_(M_shard[a:a + hi - lo])
        pos += hi - lo
    bufs = [torch.empty_like(pack) for _ in range(world)]
    _all_gather(bufs, pack, group)
    where = {}                                   # (matrix, rank) -> (buffer, position)
    for r in range(world):
        pos = 0
        for i, lo, hi in layout.pack_order(r):
            where[(i, r)] = (bufs[r], pos)
            pos += hi - lo
    full = {}
    for i in layout.boundary():
        pcs = layout.pieces(i)
        if not any(p[0] == rank for p in pcs):
            continue
        m = torch.empty(layout.numel(i), dtype=M_shard.dtype, device=M_shard.device)
        for r, lo, hi in pcs:
            buf, pos = where[(i, r)]
            m[lo:hi].copy_(buf[pos:pos + hi - lo])
        full[i] = m.view(layout.shapes[i])
    return full


def zero1_step(W, G, M_shard, layout: Zero1Layout, layers, ops, hp, group=None):
    """One ZeRO-1 MuonClip step on this rank.

    W: the full (replicated) weight matrices, updated in place on every rank.
    G: this rank's local gradients (full matrices); they are averaged.
    M_shard: this rank's momentum slice (zero1_state), updated in place.
    layers: [(smax, [(matrix index, row offset, head stride, rows, exponent)])]
    with this rank's local S_max; they are all-reduced (MAX) in place.
    ops: momentum(M, G, mu) on 2-D views; step(W_list, M_full_list, layers, hp)
    = Newton-Schulz of each full momentum, update-RMS scale, decoupled weight
    decay and QK-Clip of the given layers; clip(layers, hp) = QK-Clip only.
    """
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    if world != layout.world:
        raise ValueError("layout world size differs from the process group")
    # 1. gradients: reduce-scatter (mean) to this rank's slice
    g_shard = _reduce_scatter_mean(_flat(G, layout, M_shard.dtype), layout, rank, group)
    # 2. momentum on the slice (an elementwise step: a [shard / align, align] view)
    shape2 = (layout.shard // layout.align, layout.align)
    if layout.shard:
        ops.momentum(M_shard.view(shape2), g_shard.view(shape2), hp)
    # QK-Clip needs S_max over the global batch
    for smax, _ in layers:
        allreduce_smax(smax, group)
    # 3. full momentum of every matrix this rank owns a piece of
    full = _gather_boundary(M_shard, layout, rank, group)
    lo_r = layout.slice(rank)[0]
    idx = layout.touched(rank)
    mfull = []
    for i in idx:
        if i in full:
            mfull.append(full[i])
        else:
            a = layout.offsets[i] - lo_r
            mfull.append(M_shard[a:a + layout.numel(i)].view(layout.shapes[i]))
    # 4. Newton-Schulz + update of the touched matrices, then QK-Clip (every
    # rank clips its copies identically; owners' slices are the ones kept)
    if idx:
        ops.step([W[i] for i in idx], mfull, layers, hp)
    else:
        ops.clip(layers, hp)
    # 5. parameters: all-gather the slices
    if world > 1:
        wflat = _flat(W, layout, W[0].dtype)
        lo, hi = layout.slice(rank)
        parts = [torch.empty(layout.shard, dtype=wflat.dtype, device=wflat.device) for _ in range(world)]
        _all_gather(parts, wflat[lo:hi].contiguous(), group)
        wfull = torch.cat(parts)
        for i, w in enumerate(W):
            a = layout.offsets[i]
            w.copy_(wfull[a:a + w.numel()].view(w.shape))
    return layout


class LibraryOps:
    """zero1_step's per-rank operations on a GPU rank: the C-ABI library."""

    def __init__(self, W):
        self.W = W                                   # matrices the clip segments index

    def _layers(self, layers):
        from . import binding as mc
        return [mc.ClipLayer(smax, [mc.ClipSegment(self.W[i], off, stride, rows, e)
                                    for (i, off, stride, rows, e) in segs])
                for smax, segs in layers]

    def momentum(self, M, G, hp):
        from . import binding as mc
        mc.muon_momentum([M], [G], hp.mu)

    def step(self, W, mfull, layers, hp):
        # momentum is already accumulated: mu = 0 and G = the full momentum
        from . import binding as mc
        from dataclasses import replace
        h = replace(hp, mu=0.0)
        scratch = [torch.zeros(m.shape, dtype=torch.float32, device=m.device) for m in mfull]
        mc.muonclip_step(W, [_lib_mat(m) for m in mfull], scratch, h, layers=self._layers(layers))

    def clip(self, layers, hp):
        from . import binding as mc
        for L in self._layers(layers):
            mc.qk_clip_apply(L.smax, hp.tau, L.segments)


def _lib_mat(t):
    """t, or a copy whose row pitch is a multiple of 16 bytes."""
    esz = t.element_size()
    if (t.stride(0) * esz) % 16 == 0 and t.data_ptr() % 16 == 0:
        return t
    r, c = t.shape
    pitch = -(-c * esz // 16) * 16 // esz
    out = torch.empty((r, pitch), dtype=t.dtype, device=t.device)[:, :c]
    out.copy_(t)
    return out
