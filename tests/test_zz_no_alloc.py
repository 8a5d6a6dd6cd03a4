"""The workspace-free GEMM entry point agrees with qgemm_q4_k.

qgemm_q4_k_noalloc is for callers that cannot allocate device memory (for
example a plugin inside an engine that owns every device allocation, or code
with a fixed memory footprint), so they cannot pass the workspace that
qgemm_q4_k takes; its scratch is a fixed array inside the library.  This test
calls it through the C ABI three times in a row -- each call finds the
previous call's data still in the shared array -- and checks each result
against the ordinary entry point bit for bit (the same kernel on the same
operands) and against the bf16 reference with the GEMM tests' tolerance
(1e-5 of sum|w*x| of the bf16-rounded operands, plus 1e-6).  It also checks
that the argument checks give the ordinary entry point's statuses and that
a call too large for the array is refused before any launch.
"""
import ctypes

import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth

pytestmark = pytest.mark.gpu


def _entry(qk):
    f = qk.load().qgemm_q4_k_noalloc
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [P, I64, I64, I64, P, I64, P, I64, P]
    f.restype = ctypes.c_int
    return f


def test_noalloc_gemm_matches_workspace_gemm(qk, orc):
    f = _entry(qk)
    stream = torch.cuda.current_stream().cuda_stream
    # the third call is smaller than the second and has K % 8 != 0, so the
    # pad columns of its bf16 copy sit where the previous call left data; it
    # also reads rows from an offset and writes into a wider y
    for M, N, K, off, ldy, seed in ((96, 384, 1024, 0, 384, 40), (512, 256, 4096, 0, 256, 41),
                                    (40, 200, 1000, 56, 333, 42)):
        wq = synth.weights("q4_k", off + N, K, seed=seed)
        x = synth.activations(M, K, seed=seed)
        wd = torch.from_numpy(wq).cuda()
        xd = torch.from_numpy(x).cuda()
        ref = torch.full((M, ldy), -5.0, device="cuda")
        qk.qgemm_q4_k(wd, off, N, K, xd, y=ref, ldy=ldy)
        y = torch.full((M, ldy), -5.0, device="cuda")
        st = f(wd.data_ptr(), off, N, K, xd.data_ptr(), M, y.data_ptr(), ldy, stream)
        assert st == 0
        torch.cuda.synchronize()
        assert qk.device_error() == 0
        # the same kernel on the same operands: the same bits, and nothing past column N
        assert torch.equal(y, ref), f"M{M} N{N} K{K}"
        assert torch.all(y[:, N:] == -5.0)
        r2, s2 = orc.gemm_bf16("q4_k", wq, K, x, rows=np.arange(off, off + N))
        diff = np.abs(y[:, :N].cpu().numpy().astype(np.float64) - r2)
        assert np.all(diff <= 1e-5 * s2 + 1e-6), f"M{M} N{N} K{K}: max diff {diff.max()}"


def test_noalloc_gemm_argument_checks_match_the_workspace_gemm(qk):
    """The same statuses as qgemm_q4_k for the same bad arguments (the workspace aside)."""
    f = _entry(qk)
    lib = qk.load()
    K, N, M = 256, 8, 4
    w = torch.zeros(qk.row_bytes("q4_k", K) * N, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), device="cuda")
    y = torch.zeros((M, N), device="cuda")
    wsp = torch.empty(qk.gemm_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    cases = [(0, N, K, M, N), (-1, N, K, M, N), (0, 0, K, M, N), (0, N, K, M, N - 1),
             ((1 << 31) - 4, N, K, M, N)]          # the last row past 2^31 - 1: too large
    for off, n, k, m, ldy in cases:
        want = lib.qgemm_q4_k(w.data_ptr(), off, n, k, x.data_ptr(), m, y.data_ptr(), ldy, wsp.data_ptr(),
                              wsp.numel(), s)
        got = f(w.data_ptr(), off, n, k, x.data_ptr(), m, y.data_ptr(), ldy, s)
        if off == 0 and n == N and ldy == N:
            continue                                 # the valid call: both launch
        assert got == want, (off, n, k, m, ldy, got, want)
    torch.cuda.synchronize()


def test_noalloc_gemm_rejects_sizes_beyond_the_array(qk):
    f = _entry(qk)
    M, N, K = 2048, 128, 4096                      # bf16 copy of x: 16 MiB > 8 MiB
    w = torch.zeros(qk.row_bytes("q4_k", K) * N, dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), device="cuda")
    y = torch.full((M, N), 2.0, device="cuda")
    st = f(w.data_ptr(), 0, N, K, x.data_ptr(), M, y.data_ptr(), N, torch.cuda.current_stream().cuda_stream)
    assert st == 8
    torch.cuda.synchronize()
    assert torch.all(y == 2.0)


def test_noalloc_gemm_bounded_wait_times_out(qk):
    """The GEMM test hook reaches this entry point too: a withheld activation
    copy makes the bounded wait run out, and the next call works normally."""
    f = _entry(qk)
    M, N, K = 64, 512, 1024
    wd = torch.from_numpy(synth.weights("q4_k", N, K, seed=43)).cuda()
    xd = torch.from_numpy(synth.activations(M, K, seed=43)).cuda()
    s = torch.cuda.current_stream().cuda_stream
    y = torch.empty((M, N), device="cuda")
    assert qk.device_error() == 0
    old = qk.set_wait_limit_ns(20_000_000)
    qk.debug_gemm_skip_chunk(0)
    try:
        assert f(wd.data_ptr(), 0, N, K, xd.data_ptr(), M, y.data_ptr(), N, s) == 0
        torch.cuda.synchronize()
        assert qk.device_error() == 6
    finally:
        qk.debug_gemm_skip_chunk(-1)
        qk.set_wait_limit_ns(old)
    assert f(wd.data_ptr(), 0, N, K, xd.data_ptr(), M, y.data_ptr(), N, s) == 0
    torch.cuda.synchronize()
    assert qk.device_error() == 0
    assert torch.equal(y, qk.qgemm_q4_k(wd, 0, N, K, xd))
