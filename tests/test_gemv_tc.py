"""GPU parity of the batch 2..8 tensor-core GEMV (Q8_0 with K a multiple of
128, Q4_K) against the CPU oracle.

Tolerance as for every GEMV: |y - y_ref| <= 1e-5 * S + 1e-6 + A per element
(S the factorised magnitude sum of the oracle, A the activation-encoding term
stated in include/qk.h), checked here without A: the two fp16 pieces of the
scaled x and the exact outlier terms keep the error far inside 1e-5 * S.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-6


@pytest.fixture(autouse=True)
def tc_forced(qk):
    """Every call here takes the tensor-core form wherever the format and K
    allow it (by default only calls with a whole 128-row tile a SM do)."""
    prev = qk.debug_gemv_tc(2)
    yield
    qk.debug_gemv_tc(prev)


def _call(qk, fmt, wd, off, rows, K, xd, y=None, ldy=0):
    fn = qk.qmatvec_q8_0 if fmt == "q8_0" else qk.qmatvec_q4_k
    return fn(wd, off, rows, K, xd, y=y, ldy=ldy)


def _check(y, yr, s, what):
    y = np.asarray(y, dtype=np.float64)
    fin = np.isfinite(yr)
    assert np.array_equal(np.isfinite(y), fin), f"{what}: non-finite pattern differs"
    bad = fin & ~(np.abs(y - yr) <= REL * s + ABS)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {i}: "
                             f"gpu {y[i]!r} oracle {yr[i]!r} S {s[i]!r}")


def _sm():
    p = torch.cuda.get_device_properties(0)
    return p.multi_processor_count, getattr(p, "shared_memory_per_block_optin", 232448)


SHAPES = [
    # fmt, rows, K, batch: ragged tiles (1, 127, 129 rows), a short last item
    # (K = 640, 896: 128 columns), padded Q4_K super-blocks (K = 300, 896);
    # K split over CTA pairs (K = 2048, 4096: 8 and 16 items a tile) with one
    # row a pair (1 row), one tile a pair, and 4 or 5 tiles a pair (the odd
    # CTA's row sums reuse their two buffers)
    ("q8_0", 1, 128, 2), ("q8_0", 127, 896, 8), ("q8_0", 129, 896, 3), ("q8_0", 1000, 896, 5),
    ("q8_0", 300, 2048, 4), ("q8_0", 999, 640, 7), ("q8_0", 5000, 3840, 2), ("q8_0", 30000, 2048, 6),
    ("q4_k", 1, 256, 2), ("q4_k", 200, 300, 6), ("q4_k", 1000, 4096, 4), ("q4_k", 257, 896, 8),
    ("q4_k", 600, 4864, 3), ("q4_k", 20000, 1024, 5), ("q4_k", 1, 2048, 7), ("q4_k", 48640, 2048, 3),
]


@pytest.mark.parametrize("fmt,rows,K,batch", SHAPES)
def test_tensor_core_gemv_matches_oracle(qk, orc, fmt, rows, K, batch):
    sms, smem = _sm()
    assert qk.debug_gemv_tc_plan_for(fmt, rows, K, sms, smem) is not None   # this shape takes the form
    wq = synth.weights(fmt, rows, K, seed=40 + batch)
    x = synth.activations(batch, K, seed=40 + batch)
    y = _call(qk, fmt, torch.from_numpy(wq).cuda(), 0, rows, K, torch.from_numpy(x).cuda()).cpu().numpy()
    yr, s = (orc.gemv_threaded(fmt, wq, K, x, np.arange(rows), orc.host_cores()) if rows * K > 4_000_000
              else orc.gemv(fmt, wq, K, x))
    _check(y, yr, s, f"{fmt} {rows}x{K} b{batch}")


@pytest.mark.parametrize("fmt,K", [("q8_0", 896), ("q4_k", 4096)])
@pytest.mark.parametrize("kind", synth.WIDE_RANGE_KINDS)
def test_tensor_core_wide_range_activations(qk, orc, fmt, K, kind):
    """Outlier groups, 2^+-30 spreads, outlier channels, two large values a
    group and subnormal x, at batch 3."""
    rows = 700
    wq = synth.weights(fmt, rows, K, seed=41)
    x, _ = synth.wide_range_activations(3, K, 41, kind)
    y = _call(qk, fmt, torch.from_numpy(wq).cuda(), 0, rows, K, torch.from_numpy(x).cuda()).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    _check(y, yr, s, f"{fmt} {kind}")


@pytest.mark.parametrize("fmt,K", [("q8_0", 896), ("q4_k", 4096)])
def test_tensor_core_row_ranges_equal_fused_call(qk, fmt, K):
    """Row ranges 4096/1024/1024 of a fused tensor at batch 4 give the bits of one call."""
    wq = synth.weights(fmt, 6144, K, seed=42)
    x = synth.activations(4, K, seed=42)
    wd, xd = torch.from_numpy(wq).cuda(), torch.from_numpy(x).cuda()
    fused = _call(qk, fmt, wd, 0, 6144, K, xd)
    parts = torch.full((4, 6144), float("nan"), device="cuda")
    for off, n in ((0, 4096), (4096, 1024), (5120, 1024), (5120, 7)):
        _call(qk, fmt, wd, off, n, K, xd, y=parts[:, off:], ldy=6144)
    torch.cuda.synchronize()
    assert torch.equal(fused, parts)


def test_tensor_core_batch_rows_are_independent(qk):
    """Batch row b of a batch-8 call has the bits of the same row in a batch-2 call."""
    fmt, rows, K = "q4_k", 3000, 2048
    wq = synth.weights(fmt, rows, K, seed=43)
    x = synth.activations(8, K, seed=43)
    wd = torch.from_numpy(wq).cuda()
    y8 = _call(qk, fmt, wd, 0, rows, K, torch.from_numpy(x).cuda())
    y2 = _call(qk, fmt, wd, 0, rows, K, torch.from_numpy(np.ascontiguousarray(x[5:7])).cuda())
    torch.cuda.synchronize()
    assert torch.equal(y8[5:7], y2)


@pytest.mark.parametrize("fmt,K", [("q8_0", 1024), ("q4_k", 1024)])
def test_tensor_core_and_fp32_forms_agree_with_oracle(qk, orc, fmt, K):
    """The same call with the tensor-core form switched off (fp32 form) and on."""
    rows, batch = 2000, 6
    wq = synth.weights(fmt, rows, K, seed=44)
    x = synth.activations(batch, K, seed=44)
    wd, xd = torch.from_numpy(wq).cuda(), torch.from_numpy(x).cuda()
    yr, s = orc.gemv(fmt, wq, K, x)
    prev = qk.debug_gemv_tc(0)
    try:
        y32 = _call(qk, fmt, wd, 0, rows, K, xd).cpu().numpy()
    finally:
        qk.debug_gemv_tc(prev)
    ytc = _call(qk, fmt, wd, 0, rows, K, xd).cpu().numpy()
    _check(y32, yr, s, "fp32 form")
    _check(ytc, yr, s, "tensor-core form")


def test_tensor_core_exact_sums_are_bit_exact(qk, orc):
    """Power-of-two scales and |x| <= 2: every partial sum is exact, so the
    tensor-core form gives the oracle's bits."""
    for fmt, K in (("q8_0", 1024), ("q4_k", 512)):
        rows = 300
        wq = synth.pow2_scaled_blocks(synth.weights(fmt, rows, K, seed=45), fmt, (-4, -3, -2, -1), 45)
        x = synth.small_int_activations(5, K, seed=45, lo=-2, hi=2)
        y = _call(qk, fmt, torch.from_numpy(wq).cuda(), 0, rows, K, torch.from_numpy(x).cuda()).cpu().numpy()
        yr, s = orc.gemv(fmt, wq, K, x)
        assert np.all(s < 2.0 ** 20)
        assert np.array_equal(y, yr.astype(np.float32)), fmt


def test_default_form_choice(qk):
    """By default the tensor-core form serves calls with a whole 128-row tile a
    SM (Q8_0 from batch 2, Q4_K from batch 4); smaller calls and Q4_K at batch
    2..3 take the fp32 form.  Each call's bits are those of the form it takes."""
    sms, _ = _sm()
    cases = [("q8_0", 128 * sms, 896, 2, True), ("q8_0", 128 * sms - 1, 896, 2, False),
             ("q4_k", 128 * sms, 1024, 4, True), ("q4_k", 128 * sms, 1024, 3, False)]
    for fmt, rows, K, batch, tc in cases:
        wq = synth.weights(fmt, rows, K, seed=46)
        x = synth.activations(batch, K, seed=46)
        wd, xd = torch.from_numpy(wq).cuda(), torch.from_numpy(x).cuda()
        prev = qk.debug_gemv_tc(1)
        try:
            y_auto = _call(qk, fmt, wd, 0, rows, K, xd)
            qk.debug_gemv_tc(2)
            y_tc = _call(qk, fmt, wd, 0, rows, K, xd)
            qk.debug_gemv_tc(0)
            y_32 = _call(qk, fmt, wd, 0, rows, K, xd)
        finally:
            qk.debug_gemv_tc(prev)
        torch.cuda.synchronize()
        assert not torch.equal(y_tc, y_32), (fmt, rows, batch)      # the two forms differ in their bits
        assert torch.equal(y_auto, y_tc if tc else y_32), (fmt, rows, batch)


@pytest.mark.parametrize("fmt,K,item", [("q8_0", 896, 0), ("q4_k", 4096, 5)])
def test_tensor_core_bounded_wait_times_out_and_context_survives(qk, orc, fmt, K, item):
    """An item whose weights are never loaded (test hook, CTA 0) makes the
    converters' bounded wait run out: the launch records QK_ERR_TIMEOUT, the
    tensor memory is freed, and later launches work normally."""
    rows, batch = 3000, 4
    wq = synth.weights(fmt, rows, K, seed=47)
    x = synth.activations(batch, K, seed=47)
    wd, xd = torch.from_numpy(wq).cuda(), torch.from_numpy(x).cuda()
    assert qk.device_error() == 0
    old = qk.set_wait_limit_ns(20_000_000)
    qk.debug_skip_item(item)
    try:
        _call(qk, fmt, wd, 0, rows, K, xd)
        assert qk.device_error() == 6
    finally:
        qk.debug_skip_item(-1)
        qk.set_wait_limit_ns(old)
    assert qk.device_error() == 0
    for _ in range(3):                      # the tensor memory of every SM is free again
        y = _call(qk, fmt, wd, 0, rows, K, xd).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    _check(y, yr, s, "after timeout")
