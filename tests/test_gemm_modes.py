"""GPU parity of the prefill GEMM's acc and swiglu modes against the oracle.

acc: y_new = y_old + Y with Y bounded as the store mode (1e-2 * S1 against the
exact product, 1e-5 * S2 against the bf16 product), plus one fp32 rounding
of the final add (2^-24 * |y_new|).
swiglu: h = silu(g) * u from the gate and up GEMM rows; against the bf16
references (g, u within e = 1e-5 * S2 + 1e-6, as the store mode):
|h - h2| <= 1.1 * e_g * |u| + (|silu(g)| + 1.1 * e_g) * e_u + 2e-6 * |h2|
(|silu'| <= 1.0998; fp32 silu and product), and within the same form with
e = 1e-2 * S1 + 1e-6 of the exact SwiGLU.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth
from tests.test_gemm import TOL_R1, TOL_R2

pytestmark = pytest.mark.gpu


def silu(z):
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_bound(g, u, sg, su, tol, hr):
    eg = tol * sg + 1e-6
    eu = tol * su + 1e-6
    return 1.1 * eg * np.abs(u) + (np.abs(silu(g)) + 1.1 * eg) * eu + 2e-6 * np.abs(hr)


@pytest.mark.parametrize("M,N,K,seed", [(5, 200, 512, 70), (300, 384, 896, 71), (600, 130, 256, 72)])
def test_gemm_acc_adds_to_y(qk, orc, M, N, K, seed):
    wq = synth.weights("q4_k", N, K, seed=seed)
    x = synth.activations(M, K, seed=seed)
    y0 = synth.activations(M, N, seed=seed + 100)
    yd = torch.from_numpy(y0.copy()).cuda()
    qk.qgemm_q4_k_acc(torch.from_numpy(wq).cuda(), 0, N, K, torch.from_numpy(x).cuda(), yd)
    torch.cuda.synchronize()
    y = yd.cpu().numpy().astype(np.float64)
    r1, s1 = orc.gemv("q4_k", wq, K, x)
    r2, s2 = orc.gemm_bf16("q4_k", wq, K, x)
    base = y0.astype(np.float64)
    assert np.all(np.abs(y - (base + r1)) <= TOL_R1 * s1 + 1e-6 + 2.0 ** -24 * np.abs(y))
    bad = ~(np.abs(y - (base + r2)) <= TOL_R2 * s2 + 1e-6 + 2.0 ** -24 * np.abs(y))
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside the bf16 bound"


def test_gemm_acc_twice_equals_store_plus_store(qk):
    """acc on a zeroed y gives the store result; a second acc doubles it exactly."""
    M, N, K = 64, 256, 1024
    wd = torch.from_numpy(synth.weights("q4_k", N, K, seed=73)).cuda()
    xd = torch.from_numpy(synth.activations(M, K, seed=73)).cuda()
    ys = qk.qgemm_q4_k(wd, 0, N, K, xd)
    ya = torch.zeros((M, N), device="cuda")
    qk.qgemm_q4_k_acc(wd, 0, N, K, xd, ya)
    torch.cuda.synchronize()
    assert torch.equal(ys, ya)
    qk.qgemm_q4_k_acc(wd, 0, N, K, xd, ya)
    torch.cuda.synchronize()
    assert torch.equal(ya, 2 * ys)


@pytest.mark.parametrize("M,F,K,gate,up,seed", [
    (5, 100, 512, 0, 100, 74),         # fused tensor [gate; up]
    (300, 250, 896, 0, 250, 75),       # ragged tiles, K = 3.5 super-blocks, two token passes
    (600, 130, 256, 130, 0, 76),       # up rows before the gate rows
    (64, 384, 2048, 10, 500, 77),      # gaps between the ranges
])
def test_gemm_swiglu_matches_oracle(qk, orc, M, F, K, gate, up, seed):
    rows = max(gate, up) + F
    wq = synth.weights("q4_k", rows, K, seed=seed)
    x = synth.activations(M, K, seed=seed)
    h = qk.qgemm_swiglu_q4_k(torch.from_numpy(wq).cuda(), gate, up, F, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    h = h.cpu().numpy().astype(np.float64)
    gr, ur = np.arange(gate, gate + F), np.arange(up, up + F)
    h2, g2, u2, sg2, su2 = orc.swiglu_gemm_bf16("q4_k", wq, K, x, gr, ur)
    bad2 = ~(np.abs(h - h2) <= swiglu_bound(g2, u2, sg2, su2, TOL_R2, h2))
    if bad2.any():
        i = tuple(np.argwhere(bad2)[0])
        raise AssertionError(f"{bad2.sum()} of {bad2.size} outside the bf16 bound; first {i}: gpu {h[i]!r} "
                             f"ref {h2[i]!r} g {g2[i]!r} u {u2[i]!r}")
    h1, g1, u1, sg1, su1 = orc.swiglu("q4_k", wq, K, x, gr, ur)
    assert np.all(np.abs(h - h1) <= swiglu_bound(g1, u1, sg1, su1, TOL_R1, h1))


def test_gemm_swiglu_equals_store_then_silu(qk):
    """g and u of the swiglu mode are the store mode's outputs bit for bit:
    h equals silu(y_gate) * y_up computed from two store calls, up to the
    fp32 evaluation of silu (the kernel divides with CUDA's fast division,
    within 2 ulp of the correctly rounded quotient)."""
    M, F, K = 256, 256, 1024
    wd = torch.from_numpy(synth.weights("q4_k", 2 * F, K, seed=78)).cuda()
    xd = torch.from_numpy(synth.activations(M, K, seed=78)).cuda()
    h = qk.qgemm_swiglu_q4_k(wd, 0, F, F, K, xd)
    g = qk.qgemm_q4_k(wd, 0, F, K, xd)
    u = qk.qgemm_q4_k(wd, F, F, K, xd)
    torch.cuda.synchronize()
    ref = (g / (1.0 + torch.exp(-g))) * u
    assert torch.allclose(h, ref, rtol=2e-6, atol=1e-30)


@pytest.mark.parametrize("fmt", ["q4_k", "q8_0"])
@pytest.mark.parametrize("mode", ["store", "acc", "swiglu"])
def test_gemm_epilogue_paths_give_the_same_bits(qk, fmt, mode):
    """Y rows 16-byte aligned (TMA-store epilogue) and not (direct stores): identical results."""
    M, N, K = 300, 256, 512
    wq = synth.weights(fmt, 2 * N, K, seed=74)
    wd = torch.from_numpy(wq).cuda()
    xd = torch.from_numpy(synth.activations(M, K, seed=74)).cuda()
    y0 = torch.from_numpy(synth.activations(M, N + 1, seed=75)).cuda()
    ya = y0[:, :N].contiguous()                # ldy = N: aligned rows
    yb = y0.clone()                            # ldy = N + 1: rows 4 bytes apart from alignment
    for y, ldy in ((ya, N), (yb, N + 1)):
        if mode == "store":
            qk._gemm({"q4_k": "qgemm_q4_k", "q8_0": "qgemm_q8_0"}[fmt], wd, 0, N, K, xd, y, ldy, None, None)
        elif mode == "acc":
            qk.qgemm_acc(fmt, wd, 0, N, K, xd, y, ldy)
        else:
            qk.qgemm_swiglu(fmt, wd, 0, N, N, K, xd, h=y, ldh=ldy)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb[:, :N])
    assert torch.equal(yb[:, N], y0[:, N])        # the column past N is not written
