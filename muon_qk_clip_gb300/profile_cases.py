"""One-shot cases for profilers (ncu): run a single call of the library on
one workload's shapes (dense_block unless --workload says otherwise) and exit.

  python -m muon_qk_clip_gb300.profile_cases step        # one full MuonClip step
  python -m muon_qk_clip_gb300.profile_cases ns          # Newton-Schulz of the 7 matrices
  python -m muon_qk_clip_gb300.profile_cases max_logit   # S_max of B4 S4096 H16 d128
  python -m muon_qk_clip_gb300.profile_cases attn_fwd    # attention forward + fused S_max, same layer
  python -m muon_qk_clip_gb300.profile_cases momentum    # momentum of the 7 matrices

Each case warms up once (so the profiled launch is not the first) and runs
`--repeat` more times.
"""
from __future__ import annotations

import argparse

import torch

from . import binding as mc
from . import build, forward, synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["step", "ns", "max_logit", "attn_fwd", "momentum"])
    ap.add_argument("--repeat", type=int, default=1)
    ap.add_argument("--precision", type=int, default=0, help="mc_ns_precision")
    ap.add_argument("--fast-steps", type=int, default=None, help="ns_fast_steps (library default if unset)")
    ap.add_argument("--workload", default="dense_block", choices=list(synth.WORKLOADS))
    ap.add_argument("--experts", type=int, default=0,
                    help="moe_experts only: keep this many matrices of each shape (0: all 64)")
    args = ap.parse_args()
    build.build()
    dev = torch.device("cuda", 0)
    wl = synth.workload(args.workload)
    att = wl.attention
    if args.case in ("step", "max_logit", "attn_fwd") and (att is None or att.kind != "mha"):
        raise SystemExit(f"case {args.case} runs on an MHA layer; {args.workload} has none")
    if args.experts and args.workload != "moe_experts":
        raise SystemExit("--experts applies to moe_experts")
    names = [m.name for m in wl.matrices]
    if args.experts:
        names = [n for n in names if int(n[1:n.index("_")]) < args.experts]
    W, G, M = synth.muon_inputs(wl, device=dev, only=names)
    Wl, Gl, Ml = [W[n] for n in names], [G[n] for n in names], [M[n] for n in names]
    hp = mc.Hparams(ns_precision=args.precision)
    if args.fast_steps is not None:
        hp.ns_fast_steps = args.fast_steps
    if args.case in ("step", "max_logit", "attn_fwd"):
        X = synth.normal((att.B, att.S, att.d_model), 1.0, "X", 0, torch.bfloat16, dev)
        q, k = forward.project_mha(X, W["Wq"], W["Wk"], att.H)
        q, k = q.contiguous(), k.contiguous()
        if args.case == "attn_fwd":
            v, _ = forward.project_mha(X, W["Wv"], W["Wv"], att.H)
            v = v.contiguous()
            out = torch.empty_like(v)
        del X
        smax = torch.zeros(att.H, device=dev)
    if args.case in ("step", "ns"):
        ws = mc.alloc_workspace(Wl, hp, dev)
    if args.case == "ns":
        Ol = [torch.empty_like(w) for w in Wl]

    def once():
        if args.case == "step":
            mc.qk_max_logit(q, k, smax=smax)
            mc.muonclip_step(Wl, Gl, Ml, hp, workspace=ws,
                             layers=[mc.ClipLayer(smax, mc.mha_segments(W["Wq"], W["Wk"], att.H))])
        elif args.case == "ns":
            mc.muon_newton_schulz(Gl, Ol, hp, workspace=ws)
        elif args.case == "max_logit":
            mc.qk_max_logit(q, k, smax=smax)
        elif args.case == "attn_fwd":
            mc.qk_attention_forward(q, k, v, out=out, smax=smax)
        else:
            mc.muon_momentum(Ml, Gl, hp.mu)

    once()
    torch.cuda.synchronize()
    for _ in range(args.repeat):
        once()
    torch.cuda.synchronize()
    print(f"profile case {args.case} done")


if __name__ == "__main__":
    main()
