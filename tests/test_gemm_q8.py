"""GPU parity of the Q8_0 prefill GEMM (store, acc and swiglu modes) against the oracle.

Bounds as the Q4_K GEMM: 1e-2 * S1 + 1e-6 against the exact product (two bf16
roundings), 1e-5 * S2 + 1e-6 against the product of bf16(fp32(w)) and
bf16(x) (fp32 accumulation only); SwiGLU with the bound derived in
test_gemm_modes.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth
from tests.test_gemm import TOL_R1, TOL_R2
from tests.test_gemm_modes import swiglu_bound

pytestmark = pytest.mark.gpu


def check(y, orc, wq, K, x, rows, what, base=None):
    r1, s1 = orc.gemv("q8_0", wq, K, x, rows=rows)
    r2, s2 = orc.gemm_bf16("q8_0", wq, K, x, rows=rows)
    extra = 0.0
    if base is not None:
        r1, r2 = base + r1, base + r2
        extra = 2.0 ** -24 * np.abs(y)
    bad1 = ~(np.abs(y - r1) <= TOL_R1 * s1 + 1e-6 + extra)
    assert not bad1.any(), f"{what}: {bad1.sum()} outside 1e-2 of the exact reference"
    bad2 = ~(np.abs(y - r2) <= TOL_R2 * s2 + 1e-6 + extra)
    if bad2.any():
        i = tuple(np.argwhere(bad2)[0])
        raise AssertionError(f"{what}: {bad2.sum()} of {bad2.size} outside {TOL_R2} of the bf16 reference; "
                             f"first {i}: gpu {y[i]!r} r2 {r2[i]!r} S2 {s2[i]!r}")


SHAPES = [
    # M tokens, N rows, K, seed
    (1, 128, 256, 80),
    (5, 200, 896, 81),        # K = 28 blocks: rows are not 16-byte multiples
    (300, 384, 576, 82),      # two token halves, K = 18 blocks
    (512, 128, 4096, 83),
    (600, 130, 2080, 84),     # ragged rows, K = 65 blocks (a chunk with one block)
    (64, 256, 40, 85),        # K inside two blocks
]


@pytest.mark.parametrize("M,N,K,seed", SHAPES)
def test_gemm_q8_0_matches_oracle(qk, orc, M, N, K, seed):
    wq = synth.weights("q8_0", N, K, seed=seed)
    x = synth.activations(M, K, seed=seed)
    y = qk.qgemm_q8_0(torch.from_numpy(wq).cuda(), 0, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    check(y.cpu().numpy().astype(np.float64), orc, wq, K, x, np.arange(N), f"q8_0 M{M} N{N} K{K}")


def test_gemm_q8_0_row_offset_and_odd_alignment(qk, orc):
    """A row range that starts 2 bytes past a 4-byte boundary (odd rows of a 34-byte-block tensor)."""
    M, K = 40, 96
    wq = synth.weights("q8_0", 300, K, seed=86)
    wd = torch.from_numpy(wq).cuda()
    x = synth.activations(M, K, seed=86)
    for off, N in ((1, 129), (77, 200)):
        y = qk.qgemm_q8_0(wd, off, N, K, torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        check(y.cpu().numpy().astype(np.float64), orc, wq, K, x, np.arange(off, off + N), f"offset {off}")


def test_gemm_q8_0_acc(qk, orc):
    M, N, K = 300, 200, 896
    wq = synth.weights("q8_0", N, K, seed=87)
    x = synth.activations(M, K, seed=87)
    y0 = synth.activations(M, N, seed=187)
    yd = torch.from_numpy(y0.copy()).cuda()
    qk.qgemm_acc("q8_0", torch.from_numpy(wq).cuda(), 0, N, K, torch.from_numpy(x).cuda(), yd)
    torch.cuda.synchronize()
    check(yd.cpu().numpy().astype(np.float64), orc, wq, K, x, np.arange(N), "q8_0 acc", base=y0.astype(np.float64))


@pytest.mark.parametrize("M,F,K,gate,up,seed", [(5, 100, 896, 0, 100, 88), (300, 130, 4096, 130, 0, 89)])
def test_gemm_q8_0_swiglu(qk, orc, M, F, K, gate, up, seed):
    wq = synth.weights("q8_0", max(gate, up) + F, K, seed=seed)
    x = synth.activations(M, K, seed=seed)
    h = qk.qgemm_swiglu("q8_0", torch.from_numpy(wq).cuda(), gate, up, F, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    h = h.cpu().numpy().astype(np.float64)
    gr, ur = np.arange(gate, gate + F), np.arange(up, up + F)
    h2, g2, u2, sg2, su2 = orc.swiglu_gemm_bf16("q8_0", wq, K, x, gr, ur)
    assert np.all(np.abs(h - h2) <= swiglu_bound(g2, u2, sg2, su2, TOL_R2, h2))
    h1, g1, u1, sg1, su1 = orc.swiglu("q8_0", wq, K, x, gr, ur)
    assert np.all(np.abs(h - h1) <= swiglu_bound(g1, u1, sg1, su1, TOL_R1, h1))


def test_gemm_q8_0_qwen_ffn_up_full(qk, orc):
    """Qwen2.5-0.5B-shaped ffn_up in Q8_0: 512 tokens x 4864 rows x 896, every output."""
    M, N, K = 512, 4864, 896
    wq = synth.weights("q8_0", N, K, seed=90)
    x = synth.activations(M, K, seed=90)
    y = qk.qgemm_q8_0(torch.from_numpy(wq).cuda(), 0, N, K, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    check(y.cpu().numpy().astype(np.float64), orc, wq, K, x, np.arange(N), "qwen ffn_up")


def test_gemm_q8_0_timeout_is_recorded(qk):
    M, N, K = 64, 256, 1024
    wd = torch.from_numpy(synth.weights("q8_0", N, K, seed=91)).cuda()
    xd = torch.from_numpy(synth.activations(M, K, seed=91)).cuda()
    assert qk.device_error() == 0
    old = qk.set_wait_limit_ns(20_000_000)
    qk.debug_gemm_skip_chunk(3)
    try:
        qk.qgemm_q8_0(wd, 0, N, K, xd)
        assert qk.device_error() == 6
    finally:
        qk.debug_gemm_skip_chunk(-1)
        qk.set_wait_limit_ns(old)
    y = qk.qgemm_q8_0(wd, 0, N, K, xd)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("K,shift", [(512, 0), (512, 2), (4096, 0)])
def test_gemm_q8_0_tma_and_direct_weight_paths(qk, orc, K, shift):
    """K a multiple of 256 with a 16-byte aligned tensor: weights by TMA; the same tensor
    2 bytes off alignment: read directly.  Both against the oracle, and store + acc."""
    M, N = 300, 260
    wq = synth.weights("q8_0", N, K, seed=90)
    buf = torch.zeros(wq.size + 16, dtype=torch.uint8, device="cuda")
    buf[shift:shift + wq.size] = torch.from_numpy(wq).cuda()
    wd = buf[shift:shift + wq.size]
    x = synth.activations(M, K, seed=90)
    xd = torch.from_numpy(x).cuda()
    y = qk.qgemm_q8_0(wd, 3, N - 3, K, xd)
    check(y.cpu().numpy().astype(np.float64), orc, wq, K, x, np.arange(3, N), f"q8_0 K{K} shift {shift}")
    y0 = synth.activations(M, N - 3, seed=91)
    yd = torch.from_numpy(y0.copy()).cuda()
    qk.qgemm_acc("q8_0", wd, 3, N - 3, K, xd, yd)
    check(yd.cpu().numpy().astype(np.float64), orc, wq, K, x, np.arange(3, N), "q8_0 acc", base=y0.astype(np.float64))
