"""Benchmark of one MuonClip step on GB300 (prints one JSON line on rank 0).

Default workload (moe_experts): the Muon half of MuonClip over one MoE expert
batch shaped like Kimi K2's experts, 64 matrices of 2048 x 7168 (up/gate) and
64 of 7168 x 2048 (down), bf16 weights, fp32 momentum and gradients (gradient
scale log-uniform in [0.1, 10] per expert).  One step = muonclip_step over
all 128 matrices (momentum, Newton-Schulz x5, RMS-matched update with weight
decay).  The expert batch has no attention, so the per-head max logit, the
attention forward with S_max fused in and QK-Clip are measured on the K2 MLA
layer at 32768 tokens (64 heads, q.k 128 + 64 with a shared rotary key,
8 heads with a heavy-tailed max logit) and reported under `components`.
Workloads with attention (--workload dense_block, k2_mla_layer, long_mla,
tiny_mha_fp32) put qk_max_logit and the clip inside the step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload NAME]

--impl reference times the CPU oracle (fp64 numpy) on a bounded sample of the
same workload on the host cores, scaled to the full step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MuonClip step ms per layer; NS & max-logit TFLOP/s (% BF16 peak); clip GB/s"
WORKLOAD = "moe_experts"
ATTN_WORKLOAD = "long_mla"        # attention components for workloads without attention
WORKLOAD_CONFIG = {
    "tiny_mha_fp32": {"matrices": "1x256x512 (fp32)", "attention": "B2 S128 H4 d64 causal (fp32)"},
    "dense_block": {"matrices": "4x2048x2048, 2x5632x2048, 1x2048x5632",
                    "attention": "B4 S4096 H16 d128 causal"},
    "k2_mla_layer": {"matrices": "W_DQ 1536x7168, W_UQ 12288x1536, W_DKV 512x7168, W_KR 64x7168, "
                                 "W_UKV 16384x512, W_O 7168x8192",
                     "attention": "MLA B1 S4096 H64 q.k 128+64 (shared k^R) causal"},
    "moe_experts": {"matrices": "64x2048x7168 + 64x7168x2048", "attention": "none"},
    "long_mla": {"matrices": "as k2_mla_layer", "attention": "MLA B1 S32768 H64 q.k 128+64 causal"},
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "of measured"
    return dict(FALLBACK_PEAKS), "of fallback"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


# ------------------------------------------------------------------ CPU oracle sample
# Per workload: the Muon matrices the oracle steps (momentum, Newton-Schulz,
# update), and how many of the attention heads it takes the max logit of.
# The time is scaled to the full step by Newton-Schulz flops and by heads.
ORACLE_SAMPLE = {
    "tiny_mha_fp32": {"mats": [(256, 512)], "heads": 4},
    "dense_block": {"mats": [(2048, 2048), (5632, 2048)], "heads": 1},
    "k2_mla_layer": {"mats": [(1536, 7168), (64, 7168)], "heads": 4},
    "moe_experts": {"mats": [(2048, 7168), (7168, 2048)], "heads": 0},
    "long_mla": {"mats": [(1536, 7168), (64, 7168)], "heads": 4},
}


def oracle_sample(workload, seed=0, small=False):
    """Time the oracle on a bounded sample of `workload`'s step and scale it
    to the full step.  small: one matrix (alternating with the seed) and one
    head, for the reference arm's per-step samples.  Returns (ms per full
    step, description)."""
    import numpy as np

    import oracle as O
    from muon_qk_clip_gb300 import synth
    wl = synth.workload(workload)
    plan = ORACLE_SAMPLE[workload]
    mats = plan["mats"]
    heads = plan["heads"]
    if small:
        mats = [mats[seed % len(mats)]]
        heads = min(heads, 1)
    rng = np.random.default_rng(seed)
    hp = O.Hparams()
    t0 = time.perf_counter()
    sample_flops = 0.0
    for (r, c) in mats:
        W = rng.standard_normal((r, c)) * wl.w_std
        G = rng.standard_normal((r, c)) * wl.g_std
        O.muon_step(W, G, np.zeros((r, c)), hp)
        sample_flops += synth.flops_ns(r, c)
    t_ns = time.perf_counter() - t0
    full_ns = sum(synth.flops_ns(m.rows, m.cols) for m in wl.matrices)
    ms = 1e3 * t_ns * full_ns / sample_flops
    shapes = " + ".join(f"{r}x{c}" for r, c in mats)
    desc = (f"extrapolated: oracle (fp64 numpy) Muon step of {shapes} ({t_ns:.1f} s), scaled by "
            f"Newton-Schulz flops x{full_ns / sample_flops:.1f} to all {len(wl.matrices)} matrices")
    att = wl.attention
    if att is not None and heads > 0:
        dq = att.d_head if att.kind == "mha" else att.d_nope + att.d_rope
        dk = att.d_head if att.kind == "mha" else att.d_nope
        q = rng.standard_normal((att.B, att.S, heads, dq))
        k = rng.standard_normal((att.B, att.S, heads, dk))
        ks = rng.standard_normal((att.B, att.S, att.d_rope)) if att.kind == "mla" else None
        t1 = time.perf_counter()
        O.max_logit(q, k, ks)
        t_ml = time.perf_counter() - t1
        ms += 1e3 * t_ml * att.H / heads
        desc += (f"; + max logit of {heads} of {att.H} heads over {att.B}x{att.S} tokens "
                 f"({t_ml:.1f} s, scaled x{att.H / heads:g})")
    return ms, desc


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    for i in range(args.warmup):
        oracle_sample(args.workload, seed=i, small=True)
    vals = []
    desc = ""
    for i in range(args.steps):
        v, desc = oracle_sample(args.workload, seed=i, small=True)
        vals.append(v)
    value = statistics.mean(vals)
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "ms",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": value,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload, **WORKLOAD_CONFIG[args.workload]},
            "cpu_baseline": {"value": value, "unit": "ms", "cores": cores, "kind": "oracle",
                             "sample": "each step: " + desc},
            "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# fp32 FMA peak of the part: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def ns_sym_entries(m, unit=256):
    """Entries of an m x m symmetric Newton-Schulz output (the Gram A = X X^T
    and the polynomial B) that the tensor-core kernel computes: every
    256 x 256 unit on or above the diagonal, edge units over their real rows
    and columns only."""
    total = 0
    for j in range(-(-m // unit)):
        c = min(unit, m - j * unit)
        total += c * min(unit * (j + 1), m)
    return total


def ns_flops_counted(rows, cols, steps, symmetric=True):
    """Newton-Schulz flops credited to the kernel: per iteration 2 n E for the
    Gram, 2 m E for the polynomial and 2 m^2 n for the update (m = min side,
    n = max side), with E the computed entries of the symmetric outputs
    (m^2 when the path does not exploit the symmetry).  Neither the skipped
    lower triangles nor the extra products of the split arithmetic count."""
    m, n = min(rows, cols), max(rows, cols)
    e = ns_sym_entries(m) if symmetric else m * m
    return steps * (2.0 * n * e + 2.0 * m * e + 2.0 * m * m * n)


def ns_products(rows, cols, steps, fast_steps, split=True):
    """Tensor-core products per k-step of each iteration's (Gram, polynomial,
    update) under the library's plan: one (hi*hi) in the leading iterations
    (up to three, keeping two three-term iterations after them, from a
    smaller side of 256), then one in the Gram and three (hi*hi + hi*lo +
    lo*hi) in the polynomial and update; matrices with a smaller side under
    256 take three everywhere.  The updates of the last two iterations take
    two (hi*hi + hi*lo of X) from a smaller side of 512 (iteration 2
    onwards)."""
    if not split:
        return [(1, 1, 1)] * steps
    side = min(rows, cols)
    nf = 0 if side < 256 else min(fast_steps, 3, max(0, steps - 2))
    trail = (1, 3, 3) if side >= 256 else (3, 3, 3)
    out = [(1, 1, 1) if it < nf else trail for it in range(steps)]
    if steps >= 2 and side >= 512:
        for it in range(max(1, steps - 2), steps):
            out[it] = (out[it][0], out[it][1], 2)
    return out


def ns_flops_executed(rows, cols, steps, fast_steps, split=True, symmetric=True):
    """What the tensor pipe executes: each phase's counted flops (Gram 2 n E,
    polynomial 2 m E, update 2 m^2 n) times its products per k-step."""
    m, n = min(rows, cols), max(rows, cols)
    e = ns_sym_entries(m) if symmetric else m * m
    ph = (2.0 * n * e, 2.0 * m * e, 2.0 * m * m * n)
    return sum(sum(p * f for p, f in zip(prod, ph))
               for prod in ns_products(rows, cols, steps, fast_steps, split))


# Sources that decide the Newton-Schulz GEMM's DRAM traffic: the kernel and
# the planner that picks each launch's products and shapes.
TRAFFIC_SOURCES = ("muon_qk_clip_gb300/csrc/ns_tc.cu", "muon_qk_clip_gb300/csrc/common.cuh",
                   "muon_qk_clip_gb300/csrc/api.cpp")


def traffic_sources_hash():
    """Hash of the code of TRAFFIC_SOURCES: comments and blank lines are
    dropped first, so an edit of a comment keeps the captured traffic."""
    import re
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())
        h.update(code.encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def traffic_for(workload, launches_per_call):
    """DRAM bytes per launch of the dominant kernel: the committed ncu total
    per Newton-Schulz call on this workload divided by this run's launches per
    call, or None when no capture exists for the workload or a source that
    decides the traffic changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or not launches_per_call:
        return None
    d = json.load(open(p)).get("ns_gemm", {}).get(workload)
    if not d or d.get("source_sha256_16") != traffic_sources_hash():
        return None
    return int(d["bytes_per_ns_call"] / launches_per_call)


def attention_setup(wname, seed, dev, hp, mc, forward, synth, W=None):
    """Q/K (and V) features of `wname`'s attention layer from its weights
    (untimed setup forward), and the layer's clip segments on the weights in
    W (the step's own weights) or on the setup weights."""
    wl = synth.workload(wname)
    att = wl.attention
    X, Wa = synth.attention_inputs(wl, seed=seed, device=dev)
    W = W if W is not None else Wa
    if att.kind == "mha":
        q, k = forward.project_mha(X, Wa["Wq"], Wa["Wk"], att.H)
        q, k = q.contiguous(), k.contiguous()
        Wv = W["Wv"] if "Wv" in W else Wa.get("Wv", Wa["Wq"])
        v, _ = forward.project_mha(X, Wv, Wv, att.H)
        v = v.contiguous()
        Wq = W["Wq"] if "Wq" in W else Wa["Wq"]
        Wk = W["Wk"] if "Wk" in W else Wa["Wk"]
        segs = mc.mha_segments(Wq, Wk, att.H, hp.alpha)
        ks = None
    else:
        q, kc, ks, v = forward.project_mla(X, Wa, att.H, att.d_nope, att.d_rope, att.d_v, with_v=True)
        q, ks = q.contiguous(), ks.contiguous()
        k = kc                                          # strided views of [k^C || v]
        segs = mc.mla_segments(W["W_UQ"], W["W_UKV"], att.H, att.d_nope, att.d_rope, att.d_v)
    del X
    return {"wl": wl, "att": att, "q": q, "k": k, "ks": ks, "v": v, "segs": segs,
            "weights": Wa}


def attention_components(A, args, hp, mc, dev, stream, flush, barrier, peak_t, hbm):
    # peak_t: the burst bf16 figure (each kernel is timed alone, a few ms per call)
    """The attention-side figures on layer A: qk_max_logit, the attention
    forward with S_max fused in, the clip of the layer's offending heads and
    an all-heads clip stress (L2 flushed before each timed call)."""
    import torch
    att, q, k, ks, v, segs = A["att"], A["q"], A["k"], A["ks"], A["v"], A["segs"]
    H = att.H
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    smax = torch.zeros(H, dtype=torch.float32, device=dev)
    d_qk = q.shape[-1]
    out = {"workload": A["wl"].name, "attention": WORKLOAD_CONFIG[A["wl"].name]["attention"]}

    def timed(fn, n, spin=False):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush.zero_()
            if spin:
                # a ~50 us device spin keeps the stream busy while the host
                # builds the call, so the interval holds the launch, not the host
                torch.cuda._sleep(100_000)
            a.record(stream)
            fn()
            b.record(stream)
        barrier()
        return sorted(a.elapsed_time(b) for a, b in evs)

    # max logit
    ml = lambda: mc.qk_max_logit(q, k, ks, smax=smax, status=status, stream=stream)  # noqa: E731
    for _ in range(2):
        ml()
    barrier()
    t = timed(ml, args.steps, spin=True)
    ml_ms = statistics.median(t)
    ml_flops = synth_flops_max_logit(att, d_qk)
    out["max_logit"] = {"ms": round(ml_ms, 4), "tflops": round(ml_flops / (ml_ms * 1e-3) / 1e12, 2),
                        "frac_bf16_peak": round(ml_flops / (ml_ms * 1e-3) / 1e12 / peak_t, 4),
                        "algorithmic_flops": ml_flops}
    # attention forward with S_max fused in
    if q.dtype == torch.bfloat16:
        o_buf = torch.empty(v.shape, dtype=v.dtype, device=dev)
        smax_f = torch.empty(H, dtype=torch.float32, device=dev)
        fw = lambda: mc.qk_attention_forward(q, k, v, ks, out=o_buf, smax=smax_f, status=status,  # noqa: E731
                                             stream=stream)
        for _ in range(2):
            fw()
        barrier()
        t = timed(fw, args.steps, spin=True)
        fwd_ms = statistics.median(t)
        fwd_flops = 2.0 * (d_qk + v.shape[-1]) * att.B * att.H * att.S * (att.S + 1) / 2
        out["attn_fwd_fused_smax"] = {
            "ms": round(fwd_ms, 4), "tflops": round(fwd_flops / (fwd_ms * 1e-3) / 1e12, 2),
            "frac_bf16_peak": round(fwd_flops / (fwd_ms * 1e-3) / 1e12 / peak_t, 4),
            "algorithmic_flops": fwd_flops,
            "smax_equals_max_logit": bool(torch.equal(smax_f, smax))}
        del o_buf
    # the clip of this layer's offending heads with the measured S_max (on
    # copies of the weights, restored before each call)
    copies = {}
    for sg in segs:
        copies.setdefault(sg.w.data_ptr(), (sg.w, sg.w.clone()))
    csegs = [mc.ClipSegment(copies[sg.w.data_ptr()][1], sg.offset, sg.stride, sg.rows, sg.exponent)
             for sg in segs]
    gamma = torch.zeros(H, dtype=torch.float32, device=dev)
    ncl = torch.zeros(1, dtype=torch.int32, device=dev)
    mc.qk_clip_apply(smax, hp.tau, csegs, gamma_out=gamma, nclipped=ncl, status=status, stream=stream)
    barrier()
    n_clipped = int(ncl.item())
    t = timed(lambda: mc.qk_clip_apply(smax, hp.tau, csegs, stream=stream), args.steps, spin=True)
    clip_ms = statistics.median(t)
    esz = q.element_size()
    per_head_rows = 2 * att.d_head if att.kind == "mha" else att.d_nope + att.d_rope + att.d_nope
    row_len = max(sg.w.shape[1] for sg in segs)
    clip_bytes = 2 * n_clipped * per_head_rows * row_len * esz          # read + write
    out["clip_layer"] = {"heads_clipped": n_clipped, "bytes": clip_bytes, "us": round(clip_ms * 1e3, 2),
                         "gbs": round(clip_bytes / (clip_ms * 1e-3) / 1e9, 1)}
    # every head over tau
    s_all = torch.full((H,), 4.0 * hp.tau, dtype=torch.float32, device=dev)
    stress_bytes = sum(2 * H * sg.rows * sg.w.shape[1] * sg.w.element_size() for sg in csegs)
    mc.qk_clip_apply(s_all, hp.tau, csegs, stream=stream)
    barrier()
    t = timed(lambda: mc.qk_clip_apply(s_all, hp.tau, csegs, stream=stream), args.steps, spin=True)
    cms = statistics.median(t)
    out["clip_stress_all_heads"] = {"heads_clipped": H, "bytes": stress_bytes, "ms": round(cms, 4),
                                    "gbs": round(stress_bytes / (cms * 1e-3) / 1e9, 1),
                                    "frac_hbm": round(stress_bytes / (cms * 1e-3) / 1e9 / hbm, 4)}
    out["smax_head_max"] = round(float(smax.max().item()), 3)
    out["device_status"] = int(status.item())
    del copies, csegs
    return out


def synth_flops_max_logit(att, d_qk):
    from muon_qk_clip_gb300 import synth
    return synth.flops_max_logit(att.B, att.S, att.H, d_qk)


def clip_stress_large(mc, hp, dev, stream, barrier, hbm):
    """The clip where HBM bandwidth, not launch latency, decides: 64 heads of
    8192 x 1024 bf16 rows (1 GiB), every head over tau."""
    import torch
    Hs, rows, cols = 64, 8192, 1024
    Wbig = torch.ones(Hs * rows, cols, dtype=torch.bfloat16, device=dev)
    segs_l = [mc.ClipSegment(Wbig, 0, rows, rows, 0.5)]
    s_l = torch.full((Hs,), 4.0 * hp.tau, dtype=torch.float32, device=dev)
    mc.qk_clip_apply(s_l, hp.tau, segs_l, stream=stream)
    barrier()
    ev_l = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
    for a, b in ev_l:
        torch.cuda._sleep(100_000)
        a.record(stream)
        mc.qk_clip_apply(s_l, hp.tau, segs_l, stream=stream)
        b.record(stream)
    barrier()
    ms_l = statistics.median(a.elapsed_time(b) for a, b in ev_l)
    nbytes = 2 * Wbig.numel() * Wbig.element_size()          # read + write
    del Wbig
    return {"heads_clipped": Hs, "bytes": nbytes, "ms": round(ms_l, 4),
            "gbs": round(nbytes / (ms_l * 1e-3) / 1e9, 1), "frac_hbm": round(nbytes / (ms_l * 1e-3) / 1e9 / hbm, 4)}


def gpu_arm(args):
    import torch

    from muon_qk_clip_gb300 import binding as mc
    from muon_qk_clip_gb300 import forward, synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    wl = synth.workload(args.workload)
    att = wl.attention
    # ---- inputs resident in HBM (each rank its own layer: weak scaling)
    seed = 1000 + rank
    W, G, M = synth.muon_inputs(wl, seed=seed, device=dev)
    names = [m.name for m in wl.matrices]
    Wl, Gl, Ml = [W[n] for n in names], [G[n] for n in names], [M[n] for n in names]
    hp = mc.Hparams()
    A = attention_setup(args.workload, seed, dev, hp, mc, forward, synth, W) if att is not None else None
    q = k = ks = None
    segs = []
    if A is not None:
        q, k, ks, segs = A["q"], A["k"], A["ks"], A["segs"]
    ws = mc.alloc_workspace(Wl, hp, dev)
    H = att.H if att is not None else 1
    smax = torch.zeros(H, dtype=torch.float32, device=dev)
    gamma = torch.zeros(H, dtype=torch.float32, device=dev)
    ncl = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    layers = [mc.ClipLayer(smax, segs, gamma, ncl)] if att is not None else []
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)   # > 129 MB L2
    stream = torch.cuda.current_stream()

    def step():
        if att is not None:
            mc.qk_max_logit(q, k, ks, smax=smax, status=status, stream=stream)
        mc.muonclip_step(Wl, Gl, Ml, hp, layers=layers, workspace=ws, status=status, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()

    # ---- timed region: K steps, L2 flushed before each (outside the events)
    mc.profiler_enable(True)
    mc.profiler_read(reset=True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        barrier()
        wall = time.perf_counter() - wall0
    prof = mc.profiler_read(reset=True)
    mc.profiler_enable(False)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    t_local = sum(step_ms)
    if dist is not None:
        t = torch.tensor([t_local], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        t_local = float(t.item())
    ms_per_step = t_local / args.steps
    stat = int(status.item())
    n_clipped_step = int(ncl.item()) if att is not None else 0

    # ---- end to end through the public API: pinned host G (and Q, K) in, metrics out.
    # The inputs are double-buffered on the device: step i+1's host-to-device
    # copies run on a copy stream while step i computes, and every copy, from
    # the first step's to the last one's, lies inside the timed region (one
    # region over the K steps: start event, then the first copy, ..., the last
    # step's result read back).  Each step's inputs (G and Q/K) are larger than
    # L2, so no flush runs in this region.
    feats = [t for t in (q, k, ks) if t is not None]
    host_block, host_in = pinned_block(Gl + feats)
    Gh, fh = host_in[:len(Gl)], host_in[len(Gl):]
    out_h = torch.empty(2 * H + 2, dtype=torch.float32).pin_memory()
    h2d = sum(g.numel() * g.element_size() for g in Gh) + sum(t.numel() * t.element_size() for t in fh)
    d2h = out_h.numel() * 4
    res = torch.empty(2 * H + 2, dtype=torch.float32, device=dev)
    G_slots = [Gl, [torch.empty_like(g) for g in Gl]]
    F_slots = [feats, [torch.empty_strided(t.size(), t.stride(), dtype=t.dtype, device=dev) for t in feats]]
    # the copies are spread over several streams (one copy engine each) in
    # about equal byte shares, so the host link is not left to one engine
    n_copy = args.copy_streams
    copy_streams = [torch.cuda.Stream(device=dev) for _ in range(n_copy)]
    pairs_of = [[] for _ in range(2)]
    for slot in range(2):
        items = list(zip(G_slots[slot], Gh)) + list(zip(F_slots[slot], fh))
        items.sort(key=lambda x: -x[1].numel() * x[1].element_size())
        loads = [0] * n_copy
        share = [[] for _ in range(n_copy)]
        for d, h in items:
            k = loads.index(min(loads))
            share[k].append((d, h))
            loads[k] += h.numel() * h.element_size()
        pairs_of[slot] = share
    ready = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]   # slot's inputs landed
    consumed = [torch.cuda.Event(), torch.cuda.Event()]   # slot's inputs read by its step
    used = [False, False]

    def issue_copies(slot):
        for k, cs in enumerate(copy_streams):
            with torch.cuda.stream(cs):
                if used[slot]:
                    cs.wait_event(consumed[slot])
                for d, h in pairs_of[slot][k]:
                    d.copy_(h, non_blocking=True)
                ready[slot][k].record(cs)

    # a step whose inputs fit in L2 flushes it inside the region (counted)
    e2e_flush = h2d < 129 * 2 ** 20

    def e2e_step(slot):
        for ev_k in ready[slot]:
            stream.wait_event(ev_k)
        if e2e_flush:
            flush.zero_()
        if att is not None:
            fq, fk = F_slots[slot][0], F_slots[slot][1]
            fks = F_slots[slot][2] if ks is not None else None
            mc.qk_max_logit(fq, fk, fks, smax=smax, status=status, stream=stream)
        mc.muonclip_step(Wl, G_slots[slot], Ml, hp, layers=layers, workspace=ws, status=status,
                         stream=stream)
        consumed[slot].record(stream)
        used[slot] = True
        # the step's result: S_max, gamma, heads clipped and the status word
        res[:H].copy_(smax)
        res[H:2 * H].copy_(gamma)
        res[2 * H:2 * H + 1].copy_(ncl.float())
        res[2 * H + 1:].copy_(status.float())
        out_h.copy_(res, non_blocking=True)

    def e2e_run(n):
        for cs in copy_streams:
            cs.wait_stream(stream)
        issue_copies(0)
        for i in range(n):
            if i + 1 < n:
                issue_copies((i + 1) % 2)
            e2e_step(i % 2)

    # warm-up: the pipeline runs ~1.5 s of steps untimed first (a count from
    # the max-over-ranks step time, the same on every rank)
    e2e_run(max(args.warmup, int(math.ceil(1500.0 / max(ms_per_step, 1e-3)))))
    barrier()
    e2e_t0, e2e_t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_t0.record(stream)
    e2e_run(args.steps)
    e2e_t1.record(stream)
    barrier()
    e2e_local = e2e_t0.elapsed_time(e2e_t1)
    if dist is not None:
        t = torch.tensor([e2e_local], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_local = float(t.item())
    del Gh, fh, host_in, host_block, G_slots, F_slots

    pk, pk_src = peaks()
    # a roofline kernel timed inside a second or more of back-to-back steps
    # runs in the regime of the sustained (power-capped) GEMM measurement; a
    # shorter timed loop is compared with the burst figure.  Both fractions
    # are reported.
    peak_burst = pk["bf16_tflops"]
    long_loop = wall >= 1.0
    peak_t = (pk.get("bf16_tflops_sustained") or peak_burst) if long_loop else peak_burst
    hbm = pk.get("hbm_gbs") or 6764.0

    # ---- attention-side components: this workload's layer, or for a
    # workload without attention the 32768-token K2 MLA layer
    comp_att = None
    if rank == 0 and not args.no_components:
        if A is None:
            A2 = attention_setup(ATTN_WORKLOAD, seed, dev, hp, mc, forward, synth)
            comp_att = attention_components(A2, args, hp, mc, dev, stream, flush, barrier, peak_burst, hbm)
            del A2
        else:
            comp_att = attention_components(A, args, hp, mc, dev, stream, flush, barrier, peak_burst, hbm)
        torch.cuda.empty_cache()
    clip_large = clip_stress_large(mc, hp, dev, stream, barrier, hbm) if rank == 0 and not args.no_components else None

    # ---- algorithmic work
    tc_path = wl.dtype == torch.bfloat16
    ns_flops_nominal = sum(synth.flops_ns(m.rows, m.cols, hp.ns_steps) for m in wl.matrices)
    ns_flops = sum(ns_flops_counted(m.rows, m.cols, hp.ns_steps, symmetric=tc_path) for m in wl.matrices)
    # what the tensor pipe executes: the counted flops times the products per k-step
    ns_flops_products = sum(ns_flops_executed(m.rows, m.cols, hp.ns_steps, hp.ns_fast_steps, tc_path,
                                              symmetric=tc_path) for m in wl.matrices)
    ml_flops = 0.0
    clip_bytes = 0
    if att is not None:
        d_qk = att.d_head if att.kind == "mha" else att.d_nope + att.d_rope
        ml_flops = synth.flops_max_logit(att.B, att.S, att.H, d_qk)
        esz = 2 if wl.dtype == torch.bfloat16 else 4
        per_head_rows = (2 * att.d_head if att.kind == "mha"
                         else att.d_nope + att.d_rope + att.d_nope)
        row_len = {s_.w.shape[1] for s_ in segs}
        clip_bytes = 2 * n_clipped_step * per_head_rows * max(row_len) * esz   # read + write
    n_gemm, t_gemm = prof.get("ns_gemm", (0, 0.0))
    n_ml, t_ml = prof.get("max_logit", (0, 0.0))
    n_clip, t_clip = prof.get("clip", (0, 0.0))
    ns_tflops = ns_flops * args.steps / (t_gemm * 1e-3) / 1e12 if t_gemm else None
    ml_tflops = ml_flops * args.steps / (t_ml * 1e-3) / 1e12 if t_ml else None
    clip_gbs = clip_bytes * args.steps / (t_clip * 1e-3) / 1e9 if t_clip and clip_bytes else None
    # streaming kernels' algorithmic bytes: momentum/prep reads G and M, writes M
    # and the oriented iterate; apply reads W and the iterate, writes W
    elems = sum(m.rows * m.cols for m in wl.matrices)
    g_b = Gl[0].element_size()
    x_b = 4                                            # (hi, lo) 16-bit planes, or one fp32 plane
    w_b = Wl[0].element_size()
    prep_bytes = elems * (g_b + 8 + x_b)
    apply_bytes = elems * (2 * w_b + x_b)
    n_prep, t_prep = prof.get("prep", (0, 0.0))
    n_apply, t_apply = prof.get("apply", (0, 0.0))
    prep_gbs = prep_bytes * args.steps / (t_prep * 1e-3) / 1e9 if t_prep else None
    apply_gbs = apply_bytes * args.steps / (t_apply * 1e-3) / 1e9 if t_apply else None
    per_launch_flops = ns_flops / (n_gemm / args.steps) if n_gemm else None
    achieved = per_launch_flops / (t_gemm / n_gemm * 1e-3) / 1e12 if n_gemm else None
    launches = sum(v[0] for v in prof.values())
    cfg = {"workload": args.workload, **WORKLOAD_CONFIG[args.workload], "ns_steps": hp.ns_steps,
           "ns_precision": ns_precision_text(hp) if tc_path else "fp32 CUDA cores",
           "ns_flops_counted": ("Gram and polynomial: the computed 256x256 units on or above the "
                                "diagonal (symmetry exploited); update 2 m^2 n; split products not "
                                "credited" if tc_path else "4 m^2 n + 2 m^3 per iteration"),
           "clipped_heads": n_clipped_step,
           "l2": "flushed (512 MB write) before each step; e2e: " + (
               "flushed inside the timed region before each step" if e2e_flush else
               "not flushed, each step's host inputs (G, Q/K) are larger than L2"),
           "e2e_pipeline": (f"inputs double-buffered: step i+1's host copies overlap step i, spread "
                            f"over {args.copy_streams} copy streams"),
           "parallelism": f"dp{world} (one layer per rank)"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    value = ms_per_step / world
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "ms", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": cfg,
        "clocks": clk.summary(),
        "e2e": {"value": round(e2e_local / args.steps / world, 4), "unit": "ms",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "roofline": {"bound": "tensor" if tc_path else "alu",
                     "kernel": ("ns_gemm (tcgen05 Newton-Schulz phase GEMM)" if tc_path else
                                "ns_gemm (fp32 CUDA-core Newton-Schulz phase)"),
                     "achieved": round(achieved, 2) if achieved else None,
                     "peak": peak_t if tc_path else FP32_ALU_TFLOPS, "unit": "TFLOP/s",
                     "frac": round(achieved / (peak_t if tc_path else FP32_ALU_TFLOPS), 4) if achieved else None,
                     "peak_source": ((f"bf16_tflops_sustained {pk_src}: the timed loop runs {wall:.1f} s of "
                                      f"back-to-back steps" if long_loop else
                                      f"bf16_tflops {pk_src} (burst): the timed loop runs {wall:.2f} s")
                                     + " (16-bit dense; fp16 and bf16 share the rate)"
                                     if tc_path else "152 SMs x 128 fp32 lanes x 2 flops (FMA) x 2.07 GHz"),
                     "frac_of_burst_peak": round(achieved / peak_burst, 4) if achieved and tc_path else None,
                     "traffic": traffic_for(args.workload, n_gemm // args.steps if n_gemm else 0)},
        "components": {
            "attention": comp_att,
            "clip_stress_1gib": clip_large,
            "ns_algorithmic_tflops": round(ns_tflops, 2) if ns_tflops else None,
            "ns_frac_bf16_peak": round(ns_tflops / peak_t, 4) if ns_tflops else None,
            "ns_frac_bf16_burst_peak": round(ns_tflops / peak_burst, 4) if ns_tflops else None,
            "ns_nominal_tflops": round(ns_flops_nominal * args.steps / (t_gemm * 1e-3) / 1e12, 2)
            if t_gemm else None,
            "ns_tensor_pipe_tflops": round(ns_flops_products * args.steps / (t_gemm * 1e-3) / 1e12, 2)
            if t_gemm and tc_path else None,
            "ns_tensor_pipe_frac": round(ns_flops_products * args.steps / (t_gemm * 1e-3) / 1e12 / peak_t, 4)
            if t_gemm and tc_path else None,
            "max_logit_tflops_in_step": round(ml_tflops, 2) if ml_tflops else None,
            "max_logit_frac_bf16_peak_in_step": round(ml_tflops / peak_t, 4) if ml_tflops else None,
            "clip_gbs_in_step": round(clip_gbs, 1) if clip_gbs else None,
            "prep_gbs": round(prep_gbs, 1) if prep_gbs else None,
            "prep_frac_hbm": round(prep_gbs / hbm, 4) if prep_gbs else None,
            "apply_gbs": round(apply_gbs, 1) if apply_gbs else None,
            "apply_frac_hbm": round(apply_gbs / hbm, 4) if apply_gbs else None,
            "kernel_ms_per_step": {k: round(v[1] / args.steps, 4) for k, v in prof.items()},
            "kernel_launches_per_step": {k: v[0] // args.steps for k, v in prof.items()},
            "step_ms_min": round(min(step_ms), 4), "step_ms_max": round(max(step_ms), 4),
            "wall_s_timed_loop": round(wall, 3), "device_status": stat,
        },
    }
    if not args.no_cpu_baseline:
        v, desc = oracle_sample(args.workload)
        line["cpu_baseline"] = {"value": round(v, 1), "unit": "ms", "cores": cpu_cores(),
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def pinned_block(tensors):
    """Contiguous host copies of `tensors`, as views into one pinned block
    (each at a 256-byte offset): one pinned allocation for the whole input
    set.  Beside a GEMM loop, copies out of it held ~210 GB/s where 128
    separately pinned 59 MB tensors were measured alternating between 26 and
    209 GB/s from pass to pass."""
    import torch
    sizes = [t.numel() * t.element_size() for t in tensors]
    offs, total = [], 0
    for n in sizes:
        offs.append(total)
        total += (n + 255) // 256 * 256
    block = torch.empty(max(total, 256), dtype=torch.uint8, pin_memory=True)
    views = []
    for t, o, n in zip(tensors, offs, sizes):
        h = block[o:o + n].view(t.dtype).view(t.shape)
        h.copy_(t)
        views.append(h)
    return block, views


def ns_precision_text(hp):
    return (f"16-bit (hi, lo) planes, fp32 accumulate: iteration 1 on bf16 planes, later ones on "
            f"fp16; one product (hi*hi) per k-step in the first {hp.ns_fast_steps} iterations "
            f"(smaller side >= 256) and in the Gram products after them, three "
            f"(hi*hi+hi*lo+lo*hi) in the later polynomials, two (hi*hi+hi*lo of X) in the later "
            f"updates (smaller side >= 512; else three)")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="streams the end-to-end run spreads its host-to-device copies over")
    ap.add_argument("--no-components", action="store_true",
                    help="skip the attention-side and clip-stress figures")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOAD_CONFIG),
                    help="moe_experts (the K2 expert batch) is the reported workload")
    args = ap.parse_args()
    if args.impl == "reference":
        reference_arm(args)
    else:
        from muon_qk_clip_gb300 import build
        build.build()
        gpu_arm(args)


if __name__ == "__main__":
    main()
