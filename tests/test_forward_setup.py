"""The setup forward that builds Q/K for qk_max_logit (row a8: untimed, not part
of the MuonClip step) on the library's own kernels: mc_matmul (bf16 on the
tcgen05 GEMM core, fp32 on the CUDA-core GEMM), mc_rms_norm and mc_rope, each
against the oracle's fp64 definition on the same inputs, and the MHA and MLA
projections composed from them against the oracle's projections (whose RoPE
and RMSNorm are pinned in test_oracle_pins)."""
import numpy as np
import pytest
import torch

import oracle as O
from muon_qk_clip_gb300 import binding as mc
from muon_qk_clip_gb300 import forward, synth

pytestmark = pytest.mark.gpu
BF16, F32 = torch.bfloat16, torch.float32


def f64(t):
    return t.detach().double().cpu().numpy()


# one rounding of an fp32 accumulation to the output format, relative to the
# value, plus the accumulation's own error relative to sum |a||b|
TOL = {BF16: (2.0 ** -8, 4e-5), F32: (2.0 ** -23, 4e-6)}


@pytest.mark.parametrize("dtype", [BF16, F32])
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (300, 200, 96), (257, 513, 1000), (520, 264, 2048),
                                   (96, 1536, 7168)])
def test_matmul_parity(dtype, M, N, K):
    """D = A B^T element by element against fp64 on the same (rounded)
    inputs, across several 256 x 256 tiles and ragged tails."""
    A = synth.normal((M, K), 1.0, "mmA", M + N, F32, "cuda").to(dtype)
    B = synth.normal((N, K), 0.05, "mmB", M + N, F32, "cuda").to(dtype)
    # rows of D padded to a 16-byte pitch (a ragged N needs one)
    D = mc.matmul(A, B, out=torch.empty(M, (N + 7) // 8 * 8, dtype=dtype, device="cuda")[:, :N])
    torch.cuda.synchronize()
    a, b = f64(A), f64(B)
    ref = a @ b.T
    mag = np.abs(a) @ np.abs(b).T
    rt, at = TOL[dtype]
    assert np.all(np.abs(f64(D) - ref) <= rt * np.abs(ref) + at * mag)


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_matmul_pitched_operands(dtype):
    """Row pitches larger than the rows: A and B are column slices of wider
    tensors, D a column slice of a wider output."""
    M, N, K = 200, 136, 320
    Aw = synth.normal((M, K + 64), 1.0, "pA", 3, F32, "cuda").to(dtype)
    Bw = synth.normal((N, K + 32), 0.05, "pB", 3, F32, "cuda").to(dtype)
    Dw = torch.full((M, N + 24), 7.0, dtype=dtype, device="cuda")
    A, B, D = Aw[:, 16:16 + K], Bw[:, 8:8 + K], Dw[:, 8:8 + N]
    mc.matmul(A, B, out=D)
    torch.cuda.synchronize()
    a, b = f64(A), f64(B)
    ref = a @ b.T
    rt, at = TOL[dtype]
    assert np.all(np.abs(f64(D) - ref) <= rt * np.abs(ref) + at * (np.abs(a) @ np.abs(b).T))
    assert torch.all(Dw[:, :8] == 7.0) and torch.all(Dw[:, 8 + N:] == 7.0)


def test_matmul_flags_nonfinite():
    A = synth.normal((64, 64), 1.0, "nfA", 4, F32, "cuda").to(BF16)
    B = synth.normal((64, 64), 1.0, "nfB", 4, F32, "cuda").to(BF16)
    A[5, 3] = float("inf")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mc.matmul(A, B, status=st)
    torch.cuda.synchronize()
    assert st.item() & 1


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_rms_norm_parity(dtype):
    rows, cols = 1000, 1536
    x = synth.normal((rows, cols), 3.0, "rms", 5, F32, "cuda").to(dtype)
    y = mc.rms_norm(x, eps=1e-6)
    ref = O.rms_norm(f64(x), 1e-6)
    rt = 2.0 ** -8 if dtype == BF16 else 1e-5
    assert np.all(np.abs(f64(y) - ref) <= rt * np.abs(ref) + 1e-7)
    mc.rms_norm(x, out=x, eps=1e-6)                    # in place
    torch.cuda.synchronize()
    assert torch.equal(x, y)


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_rope_parity(dtype):
    """Interleaved pairs at positions up to 4095, in place on a strided view
    (the rotary tail of each head), the rest of each row untouched."""
    B, S, H, dn, dr = 2, 4096, 3, 16, 64
    full = synth.normal((B, S, H, dn + dr), 1.0, "rope", 6, F32, "cuda").to(dtype)
    before = full.clone()
    mc.rope_(full[..., dn:])
    torch.cuda.synchronize()
    ref = O.rope(f64(before[..., dn:]))
    x = f64(before[..., dn:])
    pair = np.repeat(np.abs(x[..., 0::2]) + np.abs(x[..., 1::2]), 2, axis=-1)
    rt = 2.0 ** -8 if dtype == BF16 else 4e-7
    assert np.all(np.abs(f64(full[..., dn:]) - ref) <= rt * pair + 1e-7)
    assert torch.equal(full[..., :dn], before[..., :dn])


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_project_mha_matches_oracle(dtype):
    B, S, D, H = 2, 40, 256, 4
    X = synth.normal((B, S, D), 1.0, "fx", 1, F32, "cuda").to(dtype)
    Wq = synth.normal((D, D), 0.1, "fq", 1, F32, "cuda").to(dtype)
    Wk = synth.normal((D, D), 0.1, "fk", 1, F32, "cuda").to(dtype)
    q, k = forward.project_mha(X, Wq, Wk, H)
    torch.cuda.synchronize()
    qo, ko = O.project_mha(f64(X), f64(Wq), f64(Wk), H)
    x, wq, wk = f64(X).reshape(B * S, D), f64(Wq), f64(Wk)
    rt, at = TOL[dtype]
    for got, ref, w in ((q, qo, wq), (k, ko, wk)):
        mag = (np.abs(x) @ np.abs(w).T).reshape(ref.shape)
        assert np.all(np.abs(f64(got) - ref) <= rt * np.abs(ref) + at * mag)


@pytest.mark.parametrize("dtype", [BF16, F32])
def test_project_mla_matches_oracle(dtype):
    """MLA features (R8 layout): q = [q^C || RoPE(q^R)] from the RMS-normed
    query latent, k^C from the RMS-normed key latent, the shared rotary key
    RoPE(X W_KR^T), and the values.  The library rounds each intermediate to
    the input dtype (the latents, the up-projections before RoPE), so bf16
    agrees to a few bf16 roundings and fp32 to a few fp32 ones."""
    B, S, D, H, ql, kl, dn, dr, dv = 1, 300, 256, 3, 96, 64, 16, 8, 16
    mk = lambda shape, std, key: synth.normal(shape, std, key, 2, F32, "cuda").to(dtype)  # noqa: E731
    W = {"W_DQ": mk((ql, D), 0.1, "dq"), "W_UQ": mk((H * (dn + dr), ql), 0.2, "uq"),
         "W_DKV": mk((kl, D), 0.1, "dkv"), "W_UKV": mk((H * (dn + dv), kl), 0.2, "ukv"),
         "W_KR": mk((dr, D), 0.1, "kr")}
    X = mk((B, S, D), 1.0, "mx")
    q, kc, kr, v = forward.project_mla(X, W, H, dn, dr, dv, with_v=True)
    torch.cuda.synchronize()
    Wd = {n: f64(w) for n, w in W.items()}
    qo, kco, kro = O.project_mla(f64(X), Wd["W_DQ"], Wd["W_UQ"], Wd["W_DKV"], Wd["W_UKV"],
                                 Wd["W_KR"], H, dn, dr, dv)
    ckv = O.rms_norm(f64(X) @ Wd["W_DKV"].T)
    vo = (ckv @ Wd["W_UKV"].T).reshape(B, S, H, dn + dv)[..., dn:]
    tol = 3e-2 if dtype == BF16 else 2e-5
    for got, ref in ((q, qo), (kc, kco), (kr, kro), (v, vo)):
        scale = np.sqrt(np.mean(ref ** 2))
        assert np.max(np.abs(f64(got) - ref)) <= tol * scale, (got.shape, np.max(np.abs(f64(got) - ref)) / scale)


def test_projection_rejects_host_tensors():
    X = torch.zeros(1, 4, 8)
    W = torch.zeros(8, 8)
    with pytest.raises(ValueError, match="device tensors"):
        forward.project_mha(X, W, W, 1)
