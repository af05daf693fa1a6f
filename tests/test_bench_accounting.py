"""The Newton-Schulz flop accounting bench.py reports its roofline with.

The tensor-core kernel computes only the 256 x 256 units of the symmetric
outputs (A = X X^T and the polynomial B) on or above the diagonal, so those
phases are credited with the entries of those units, never with the full
m x m output; the split products are not credited either."""
import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("m", [1, 100, 255, 256, 257, 300, 512, 1000, 2048, 2049])
def test_sym_entries_brute_force(bench, m):
    """Mark every entry (r, c) whose 256-unit block (r // 256, c // 256) lies on
    or above the diagonal and count them."""
    r = np.arange(m) // 256
    mask = r[:, None] <= r[None, :]
    assert bench.ns_sym_entries(m) == int(mask.sum())


def test_sym_entries_closed_form(bench):
    # m = 256 T: T (T + 1) / 2 full units
    for t in (1, 2, 8, 28):
        assert bench.ns_sym_entries(256 * t) == 256 * 256 * t * (t + 1) // 2


def test_counted_flops(bench):
    m, n, steps = 512, 1536, 5
    e = 256 * 256 * 3                      # units (0,0), (0,1), (1,1)
    want = steps * (2 * n * e + 2 * m * e + 2 * m * m * n)
    assert bench.ns_flops_counted(m, n, steps) == want
    assert bench.ns_flops_counted(n, m, steps) == want        # orientation
    # without symmetry it is the nominal 4 m^2 n + 2 m^3
    assert bench.ns_flops_counted(m, n, steps, symmetric=False) == steps * (4 * m * m * n + 2 * m ** 3)


def test_products_per_iteration(bench):
    # G2: the updates of the last two iterations of a plan keeping two
    # three-term iterations take two products (hi*hi + hi*lo of X) from a
    # smaller side of 512
    F, S, G1, G2 = (1, 1, 1), (3, 3, 3), (1, 3, 3), (1, 3, 2)
    assert bench.ns_products(128, 7168, 5, 3) == [S] * 5              # smaller side < 256
    assert bench.ns_products(256, 7168, 5, 3) == [F, F, F, G1, G1]    # < 512: three
    assert bench.ns_products(1024, 1536, 5, 3) == [F, F, F, G2, G2]
    assert bench.ns_products(1024, 1536, 5, 4) == [F, F, F, G2, G2]   # at most three
    assert bench.ns_products(512, 1536, 5, 4) == [F, F, F, G2, G2]
    assert bench.ns_products(2048, 5632, 5, 2) == [F, F, G1, G2, G2]
    assert bench.ns_products(2048, 5632, 4, 3) == [F, F, G2, G2]     # two three-term kept
    assert bench.ns_products(2048, 5632, 4, 4) == [F, F, G2, G2]
    assert bench.ns_products(2048, 2048, 5, 0) == [G1] * 3 + [G2] * 2
    assert bench.ns_products(2048, 2048, 2, 0) == [G1, G2]            # iteration 1: bf16 planes
    assert bench.ns_products(2048, 2048, 1, 0) == [G1]
    assert bench.ns_products(2048, 2048, 5, 3, split=False) == [F] * 5


def test_executed_flops_weight_each_phase_by_its_products(bench):
    m, n = 2048, 5632
    e = bench.ns_sym_entries(m)
    g, p, u = 2.0 * n * e, 2.0 * m * e, 2.0 * m * m * n
    # iterations: one-product x 3, then one-product Gram, three-product
    # polynomial and two-product update x 2
    want = 3 * (g + p + u) + 2 * (g + 3 * p + 2 * u)
    assert bench.ns_flops_executed(m, n, 5, 3) == want
    assert bench.ns_flops_executed(m, n, 5, 3, split=False) == bench.ns_flops_counted(m, n, 5)


def test_traffic_is_taken_only_for_the_profiled_source(bench, tmp_path, monkeypatch):
    """The roofline's DRAM traffic comes from the committed ncu total per
    Newton-Schulz call on the same workload, divided by this run's launches
    per call, and only while every source that decides the traffic (the
    kernel, its helpers and the planner) still hashes as when it was taken."""
    import json
    for rel in bench.TRAFFIC_SOURCES:
        f = tmp_path / rel
        f.parent.mkdir(parents=True, exist_ok=True)
        f.write_text(f"// {rel}\nint x = 1;  /* a\n comment */\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.traffic_sources_hash()
    (tmp_path / "profiles").mkdir()
    rec = {"ns_gemm": {"moe_experts": {"bytes_per_ns_call": 3000, "source_sha256_16": h}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.traffic_for("moe_experts", 30) == 100
    assert bench.traffic_for("moe_experts", 0) is None
    assert bench.traffic_for("dense_block", 30) is None           # no capture for it
    for rel in bench.TRAFFIC_SOURCES:                               # any code change voids it
        f = tmp_path / rel
        old = f.read_text()
        f.write_text(old + "int changed;\n")
        assert bench.traffic_for("moe_experts", 30) is None, rel
        f.write_text(old.replace("int x = 1;", "int x = 2;"))
        assert bench.traffic_for("moe_experts", 30) is None, rel
        f.write_text(old + "// a comment\n\n/* another */\n")     # comments do not
        assert bench.traffic_for("moe_experts", 30) == 100, rel
        f.write_text(old)
    assert bench.traffic_for("moe_experts", 30) == 100


def test_oracle_sample_covers_every_workload(bench):
    from muon_qk_clip_gb300 import synth
    for name in synth.WORKLOADS:
        plan = bench.ORACLE_SAMPLE[name]
        wl = synth.workload(name)
        shapes = {(m.rows, m.cols) for m in wl.matrices}
        assert all(s in shapes for s in plan["mats"]), name
        assert (plan["heads"] > 0) == (wl.attention is not None), name


@pytest.mark.parametrize("steps,fast", [(5, 2), (5, 3), (5, 4), (5, 0), (5, 1), (4, 3), (4, 4), (6, 5),
                                        (3, 2), (2, 4), (0, 2)])
def test_products_mirror_the_library_plan(bench, steps, fast):
    """bench.py's executed-flop accounting uses a copy of the library's plan of
    products per k-step; the library reports its own through mc_ns_products."""
    from muon_qk_clip_gb300 import abi, build
    from muon_qk_clip_gb300 import binding as mc
    build.build()
    abi.load()
    hp = mc.Hparams(ns_steps=steps, ns_fast_steps=fast)
    for r, c in [(64, 64), (255, 300), (256, 256), (512, 7168), (1023, 1536), (1024, 1536),
                 (1536, 1024), (2047, 4096), (2048, 2048), (2048, 5632), (7168, 2048), (8192, 7168)]:
        assert mc.ns_products(r, c, hp) == bench.ns_products(r, c, steps, fast), (r, c)


def test_products_call_rejects(bench):
    from muon_qk_clip_gb300 import abi, build
    from muon_qk_clip_gb300 import binding as mc
    build.build()
    lib = abi.load()
    hc = mc.Hparams().c()
    import ctypes
    out = (ctypes.c_int32 * 15)()
    assert lib.mc_ns_products(ctypes.byref(hc), 0, 5, out) == abi.MC_ERR_INVALID_ARG
    assert lib.mc_ns_products(ctypes.byref(hc), 5, 5, None) == abi.MC_ERR_INVALID_ARG
    bad = mc.Hparams(ns_fast_steps=-1).c()
    assert lib.mc_ns_products(ctypes.byref(bad), 5, 5, out) == abi.MC_ERR_INVALID_ARG
