"""GPU parity of the tcgen05 Q4_K prefill GEMM against the CPU oracle.

Two references: R1, the exact f64 dot of the decoded weights and the fp32
activations, and R2, the f64 dot of bf16(fp32(w)) and bf16(x).  The bound
against R1 is the stated 1e-2 relative (read per element against
sum|w*x|); against R2 only the fp32 accumulation differs, which pins that
both operands were rounded to nearest-even bf16 and w via fp32.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_R1 = 1e-2
TOL_R2 = 1e-5


def run_gemm(qk, wq, row_offset, N, K, x):
    wd = torch.from_numpy(np.ascontiguousarray(wq)).cuda()
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    y = qk.qgemm_q4_k(wd, row_offset, N, K, xd)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


def check(y, orc, wq, K, x, rows, what):
    r1, s1 = orc.gemv("q4_k", wq, K, x, rows=rows)
    r2, s2 = orc.gemm_bf16("q4_k", wq, K, x, rows=rows)
    bad1 = ~(np.abs(y - r1) <= TOL_R1 * s1 + 1e-6)
    assert not bad1.any(), f"{what}: {bad1.sum()} outside 1e-2 of the exact reference"
    bad2 = ~(np.abs(y - r2) <= TOL_R2 * s2 + 1e-6)
    if bad2.any():
        i = tuple(np.argwhere(bad2)[0])
        raise AssertionError(f"{what}: {bad2.sum()} of {bad2.size} outside {TOL_R2} of the bf16 reference; "
                             f"first {i}: gpu {y[i]!r} r2 {r2[i]!r} S2 {s2[i]!r}")
    rel = np.linalg.norm(y - r1) / max(np.linalg.norm(r1), 1e-30)
    assert rel < 5e-3, f"{what}: relative Frobenius error {rel}"


SHAPES = [
    # M tokens, N rows, K, seed
    (1, 128, 256, 1),
    (5, 200, 512, 2),        # ragged N tile
    (64, 128, 4096, 3),
    (256, 256, 1024, 4),     # exactly one token half
    (300, 384, 896, 5),      # K = 3.5 super-blocks, two token halves
    (512, 128, 2048, 6),
    (600, 130, 256, 7),      # two token passes, ragged rows
]


@pytest.mark.parametrize("M,N,K,seed", SHAPES)
def test_gemm_matches_oracle(qk, orc, M, N, K, seed):
    wq = synth.weights("q4_k", N, K, seed=seed)
    x = synth.activations(M, K, seed=seed)
    y = run_gemm(qk, wq, 0, N, K, x)
    check(y, orc, wq, K, x, np.arange(N), f"M{M} N{N} K{K}")


def test_gemm_row_offset(qk, orc):
    N_total, K, M, off, N = 600, 512, 40, 256, 200
    wq = synth.weights("q4_k", N_total, K, seed=8)
    x = synth.activations(M, K, seed=8)
    y = run_gemm(qk, wq, off, N, K, x)
    check(y, orc, wq, K, x, np.arange(off, off + N), "row offset")


def test_gemm_bf16_exact_inputs(qk, orc):
    """Weights and activations exactly representable in bf16 with small
    integer products: the GEMM equals the exact dot."""
    N, K, M = 128, 512, 32
    wq = synth.pow2_scaled_blocks(synth.weights("q4_k", N, K, seed=9), "q4_k", (-4,), 9)
    rec = wq.view(synth.Q4_K_DTYPE)
    rec["scales"] &= 0x0F       # small sc/m so that every weight fits in bf16
    x = synth.small_int_activations(M, K, seed=9, lo=-2, hi=2)
    y = run_gemm(qk, wq, 0, N, K, x)
    r1, _ = orc.gemv("q4_k", wq, K, x)
    r2, _ = orc.gemm_bf16("q4_k", wq, K, x)
    assert np.array_equal(r1, r2)
    assert np.array_equal(y, r1.astype(np.float32).astype(np.float64))


def test_gemm_full_size(qk, orc):
    """Llama-8B ffn_gate shape: M = 512 tokens, K = 4096, N = 14336, every output
    against both references (the oracle on all host cores over row bands)."""
    M, K, N = 512, 4096, 14336
    wq = synth.weights("q4_k", N, K, seed=4)
    x = synth.activations(M, K, seed=4)
    y = run_gemm(qk, wq, 0, N, K, x)
    rows = np.arange(N)
    r1, s1 = orc.gemv_threaded("q4_k", wq, K, x, rows, orc.host_cores())
    r2, s2 = orc.gemm_bf16_threaded("q4_k", wq, K, x, rows, orc.host_cores())
    assert not (~(np.abs(y - r1) <= TOL_R1 * s1 + 1e-6)).any(), "outside 1e-2 of the exact reference"
    bad2 = ~(np.abs(y - r2) <= TOL_R2 * s2 + 1e-6)
    if bad2.any():
        i = tuple(np.argwhere(bad2)[0])
        raise AssertionError(f"{bad2.sum()} of {bad2.size} outside {TOL_R2} of the bf16 reference; "
                             f"first {i}: gpu {y[i]!r} r2 {r2[i]!r}")
    assert np.linalg.norm(y - r1) / np.linalg.norm(r1) < 5e-3


def test_gemm_workspace_errors(qk):
    N, K, M = 128, 256, 4
    w = torch.zeros(qk.row_bytes("q4_k", K) * N, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), device="cuda")
    y = torch.full((M, N), 3.0, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qk.QKError) as ei:
        qk.qgemm_q4_k(w, 0, N, K, x, y=y, ldy=N, workspace=small)
    assert ei.value.status == 7
    assert torch.all(y == 3.0)


def test_gemm_bounded_wait_times_out(qk, orc):
    N, K, M = 512, 1024, 64
    wq = synth.weights("q4_k", N, K, seed=10)
    x = synth.activations(M, K, seed=10)
    assert qk.device_error() == 0
    old = qk.set_wait_limit_ns(20_000_000)
    qk.debug_gemm_skip_chunk(0)
    try:
        run_gemm(qk, wq, 0, N, K, x)
        assert qk.device_error() == 6
    finally:
        qk.debug_gemm_skip_chunk(-1)
        qk.set_wait_limit_ns(old)
    y = run_gemm(qk, wq, 0, N, K, x)
    check(y, orc, wq, K, x, np.arange(N), "after timeout")


def test_gemm_token_pass_does_not_change_bits(qk):
    """A call with few weight tiles lets each CTA pair take one 256-token
    block a pass instead of two; every output still sums its K chunks in
    the same order, so rows 0..511 of a 14336-row call (two blocks a pass)
    equal a 512-row call over the same rows (one block a pass) bit for bit."""
    M, K = 512, 2048
    wq = synth.weights("q4_k", 14336, K, seed=9)
    x = synth.activations(M, K, seed=9)
    wd = torch.from_numpy(wq).cuda()
    xd = torch.from_numpy(x).cuda()
    y_big = qk.qgemm_q4_k(wd, 0, 14336, K, xd)
    y_small = qk.qgemm_q4_k(wd, 0, 512, K, xd)
    torch.cuda.synchronize()
    assert torch.equal(y_big[:, :512], y_small)
