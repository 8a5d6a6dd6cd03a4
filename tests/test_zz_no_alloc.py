"""The workspace-free GEMM entry point agrees with qgemm_q4_k.

qgemm_q4_k_noalloc is for callers that cannot allocate device memory (for
example a plugin inside an engine that owns every device allocation, or code
with a fixed memory footprint), so they cannot pass the workspace that
qgemm_q4_k takes; its scratch is a fixed array inside the library.  This test
calls it through the C ABI twice in a row -- the second call finds the first
call's data still in the shared array -- and checks each result against the
ordinary entry point with the GEMM tests' tolerance (1e-5 of sum|w*x| of the
bf16-rounded operands, plus 1e-6).  It also checks that a call too large for
the array is refused before any launch.
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
    for M, N, K, seed in ((96, 384, 1024, 40), (512, 256, 4096, 41)):
        wq = synth.weights("q4_k", N, K, seed=seed)
        x = synth.activations(M, K, seed=seed)
        wd = torch.from_numpy(wq).cuda()
        xd = torch.from_numpy(x).cuda()
        ref = qk.qgemm_q4_k(wd, 0, N, K, xd)
        y = torch.full((M, N), float("nan"), device="cuda")
        st = f(wd.data_ptr(), 0, N, K, xd.data_ptr(), M, y.data_ptr(), N, stream)
        assert st == 0
        torch.cuda.synchronize()
        assert qk.device_error() == 0
        _, s2 = orc.gemm_bf16("q4_k", wq, K, x)
        diff = np.abs(y.cpu().numpy().astype(np.float64) - ref.cpu().numpy().astype(np.float64))
        assert np.all(diff <= 1e-5 * s2 + 1e-6), f"M{M} N{N} K{K}: max diff {diff.max()}"


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
