"""GPU parity of the Q6_K GEMV (plain, SwiGLU and expert forms) against the oracle.

Tolerance as the other GEMVs: |y - y_ref| <= 1e-5 * sum|w*x| + 1e-6; where
every partial sum is exact in fp32 the GPU must equal the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth
from tests.test_gemv import assert_close, gpu_gemv
from tests.test_swiglu import assert_swiglu_close

pytestmark = pytest.mark.gpu

CASES = [
    # rows, K, batch, seed
    (1000, 4096, 1, 50), (1000, 4096, 2, 50), (600, 4096, 3, 50), (600, 4096, 4, 50),
    (300, 4096, 5, 50), (300, 4096, 6, 50), (300, 4096, 7, 50), (300, 4096, 8, 50),
    (896, 4864, 1, 51),          # 19 super-blocks: rows start 2 bytes off a 4-byte boundary
    (4864, 896, 1, 52),          # K = 3.5 super-blocks: the last block's second half is unused
    (333, 300, 5, 53), (1, 256, 1, 54), (3, 1, 1, 54), (5, 65, 8, 54), (7, 130, 2, 54),
    (900, 14336, 1, 55), (123, 14336, 2, 55), (40, 20480, 1, 55),
]


@pytest.mark.parametrize("rows,K,batch,seed", CASES)
def test_q6k_gemv_matches_oracle(qk, orc, rows, K, batch, seed):
    wq = synth.weights("q6_k", rows, K, seed=seed)
    x = synth.activations(batch, K, seed=seed)
    y = gpu_gemv(qk, "q6_k", wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv("q6_k", wq, K, x)
    assert_close(y, yr, s, f"q6_k {rows}x{K} b{batch}")


@pytest.mark.parametrize("batch", [1, 2, 3])
def test_q6k_bit_exact_when_sums_are_exact(qk, orc, batch):
    """d a power of two, |scale| <= 3, |x| <= 2: every product and partial sum
    is a multiple of 2^-3 below 2^20, so fp32 sums are exact in any order."""
    rows, K = 300, 1024
    wq = synth.pow2_scaled_blocks(synth.weights("q6_k", rows, K, seed=56), "q6_k", (-3, -2, -1, 0), 56)
    rec = wq.view(synth.Q6_K_DTYPE)
    rec["scales"] = synth.randint(56, 60, rec.size * 16, -3, 3).astype(np.int8).reshape(rec.size, 16)
    x = synth.small_int_activations(batch, K, seed=56, lo=-2, hi=2)
    y = gpu_gemv(qk, "q6_k", wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv("q6_k", wq, K, x)
    assert np.all(s < 2.0 ** 20)
    assert np.array_equal(y, yr.astype(np.float32))


def test_q6k_row_ranges_equal_one_call(qk):
    K = 4096
    wd = torch.from_numpy(synth.weights("q6_k", 3000, K, seed=57)).cuda()
    xd = torch.from_numpy(synth.activations(1, K, seed=57)).cuda()
    whole = qk.qmatvec_q6_k(wd, 0, 3000, K, xd)
    parts = torch.full((1, 3000), float("nan"), device="cuda")
    for off, n in ((0, 1000), (1000, 1999), (2999, 1)):
        qk.qmatvec_q6_k(wd, off, n, K, xd, y=parts[:, off:], ldy=3000)
    torch.cuda.synchronize()
    assert torch.equal(whole, parts)


def test_q6k_lm_head_full(qk, orc):
    """A Q6_K output head 128256 x 4096 (Llama-3 vocabulary), batch 1, every row."""
    rows, K, seed = 128256, 4096, 58
    wq = synth.weights("q6_k", rows, K, seed=seed)
    x = synth.activations(1, K, seed=seed)
    y = gpu_gemv(qk, "q6_k", wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv_threaded("q6_k", wq, K, x, np.arange(rows), orc.host_cores())
    assert_close(y, yr, s, "q6_k lm_head")


def test_q6k_nonfinite_scale_propagates(qk, orc):
    rows, K = 64, 512
    wq = synth.weights("q6_k", rows, K, seed=59)
    rec = wq.view(synth.Q6_K_DTYPE).reshape(rows, -1)
    rec["d"][5, 0] = np.float16(np.nan)
    rec["d"][9, 1] = np.float16(np.inf)
    x = synth.activations(1, K, seed=59)
    y = gpu_gemv(qk, "q6_k", wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv("q6_k", wq, K, x)
    assert np.isnan(y[0, 5]) and np.isnan(yr[0, 5])
    assert not np.isfinite(y[0, 9]) and not np.isfinite(yr[0, 9])
    keep = np.isfinite(yr[0])
    assert_close(y[:, keep], yr[:, keep], s[:, keep], "finite rows")


@pytest.mark.parametrize("F,K,batch", [(300, 4096, 1), (77, 14336, 2), (61, 300, 3)])
def test_q6k_swiglu_matches_oracle(qk, orc, F, K, batch):
    wq = synth.weights("q6_k", 2 * F, K, seed=60)
    x = synth.activations(batch, K, seed=60)
    wd = torch.from_numpy(wq).cuda()
    h = qk.qmatvec_swiglu("q6_k", wd, 0, F, F, K, torch.from_numpy(x).cuda()).cpu().numpy()
    ref = orc.swiglu("q6_k", wq, K, x, np.arange(F), np.arange(F, 2 * F))
    assert_swiglu_close(h, ref, f"q6_k swiglu F={F} K={K}")


def test_q6k_experts_match_oracle(qk, orc):
    E, rows, K, xk = 6, 300, 2048, 2
    wq = synth.weights("q6_k", E * rows, K, seed=61)
    x = synth.activations(3, K, seed=61)
    ids = np.array([5, 0, 3, 3, 1, 2], np.int32)
    y = qk.qmatvec_experts("q6_k", torch.from_numpy(wq).cuda(), E, rows, K, torch.from_numpy(x).cuda(), xk,
                           torch.from_numpy(ids).cuda()).cpu().numpy()
    yr, s = orc.experts("q6_k", wq, E, rows, K, x, xk, ids)
    assert_close(y, yr, s, "q6_k experts")


def test_q6k_bounded_wait_times_out_and_context_survives(qk, orc):
    rows, K = 2000, 4096
    wq = synth.weights("q6_k", rows, K, seed=62)
    x = synth.activations(1, K, seed=62)
    assert qk.device_error() == 0
    old = qk.set_wait_limit_ns(20_000_000)
    qk.debug_skip_item(0)
    try:
        gpu_gemv(qk, "q6_k", wq, 0, rows, K, x)
        assert qk.device_error() == 6
    finally:
        qk.debug_skip_item(-1)
        qk.set_wait_limit_ns(old)
    y = gpu_gemv(qk, "q6_k", wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv("q6_k", wq, K, x)
    assert_close(y, yr, s, "after timeout")
