"""GPU parity of the Q8_0 / Q4_K GEMV against the CPU oracle.

Tolerance (fp32 GEMV): |y - y_ref| <= 1e-5 * sum|w*x| + 1e-6 per element,
y_ref and sum|w*x| from the f64 oracle.  Where every partial sum is exact in
fp32 (power-of-two scales, small-integer activations) the GPU must be
bit-identical to the oracle whatever its summation order.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-6


def gpu_gemv(qk, fmt, wq, row_offset, rows, K, x, y=None, ldy=0):
    wd = torch.from_numpy(np.ascontiguousarray(wq)).cuda()
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    fn = {"q8_0": qk.qmatvec_q8_0, "q4_k": qk.qmatvec_q4_k, "q6_k": qk.qmatvec_q6_k}[fmt]
    out = fn(wd, row_offset, rows, K, xd, y=y, ldy=ldy)
    torch.cuda.synchronize()
    return out


def assert_close(y, yr, s, what=""):
    y = np.asarray(y, dtype=np.float64)
    bad = ~(np.abs(y - yr) <= REL * s + ABS)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu {y[tuple(i)]!r} oracle {yr[tuple(i)]!r} S {s[tuple(i)]!r}")


SMALL = [
    # fmt, rows, K, batch, seed
    ("q8_0", 576, 576, 1, 0),        # SmolLM-135M q-proj shape, seed 0
    ("q8_0", 1000, 896, 1, 5), ("q8_0", 1000, 896, 2, 5), ("q8_0", 1000, 896, 3, 5),
    ("q8_0", 1000, 896, 4, 5), ("q8_0", 1000, 896, 5, 5), ("q8_0", 1000, 896, 6, 5),
    ("q8_0", 1000, 896, 7, 5), ("q8_0", 1000, 896, 8, 5),
    ("q8_0", 333, 40, 3, 6),          # ragged K (partial block)
    ("q8_0", 1, 32, 1, 7), ("q8_0", 7, 1, 2, 7), ("q8_0", 2, 33, 8, 7),
    ("q8_0", 2000, 4096, 2, 8), ("q8_0", 150, 14336, 1, 8), ("q8_0", 61, 2080, 5, 8),
    ("q4_k", 4864, 896, 1, 1),        # Qwen2.5-0.5B ffn_up shape (K = 3.5 super-blocks)
    ("q4_k", 896, 4864, 1, 1),        # its ffn_down transpose (19 super-blocks)
    ("q4_k", 1000, 4096, 1, 9), ("q4_k", 1000, 4096, 2, 9), ("q4_k", 1000, 4096, 3, 9),
    ("q4_k", 1000, 4096, 4, 9), ("q4_k", 600, 4096, 5, 9), ("q4_k", 600, 4096, 6, 9),
    ("q4_k", 600, 4096, 7, 9), ("q4_k", 600, 4096, 8, 9),
    ("q4_k", 333, 300, 5, 10),        # ragged K inside a super-block
    ("q4_k", 1, 256, 1, 11), ("q4_k", 3, 1, 1, 11), ("q4_k", 5, 65, 8, 11),
    ("q4_k", 900, 14336, 1, 12), ("q4_k", 123, 14336, 2, 12), ("q4_k", 40, 20480, 1, 12),
]


@pytest.mark.parametrize("fmt,rows,K,batch,seed", SMALL)
def test_gemv_matches_oracle(qk, orc, fmt, rows, K, batch, seed):
    wq = synth.weights(fmt, rows, K, seed=seed)
    x = synth.activations(batch, K, seed=seed)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert_close(y, yr, s, f"{fmt} {rows}x{K} b{batch}")


@pytest.mark.parametrize("fmt,K", [("q8_0", 4096), ("q4_k", 512), ("q4_k", 4096)])
@pytest.mark.parametrize("batch", [1, 2, 3])
def test_gemv_bit_exact_when_sums_are_exact(qk, orc, fmt, K, batch):
    """Power-of-two d/dmin and |x| <= 2: every product and partial sum is a
    multiple of 2^-4 below 2^20, so fp32 sums are exact in any order."""
    rows = 300
    if fmt == "q4_k" and K > 512:
        K = 512
    wq = synth.pow2_scaled_blocks(synth.weights(fmt, rows, K, seed=21), fmt, (-4, -3, -2, -1), 21)
    x = synth.small_int_activations(batch, K, seed=21, lo=-2, hi=2)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert np.all(s < 2.0 ** 20)
    assert np.array_equal(y, yr.astype(np.float32))


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_row_ranges_equal_fused_call(qk, fmt):
    """Row ranges 4096/1024/1024 of a fused qkv tensor give the same bits as one call."""
    K0 = 4096 if fmt == "q4_k" else 896
    plans = [qk.debug_gemv_plan(fmt, n, K0, 1) for n in (6144, 4096, 1024)]
    assert len({(p["SW"], p["nkc"], p["cpl"]) for p in plans}) == 1   # the row's cut depends on K only
    K = 4096 if fmt == "q4_k" else 896
    wq = synth.weights(fmt, 6144, K, seed=3)
    x = synth.activations(1, K, seed=3)
    wd = torch.from_numpy(wq).cuda()
    xd = torch.from_numpy(x).cuda()
    fn = qk.qmatvec_q8_0 if fmt == "q8_0" else qk.qmatvec_q4_k
    fused = fn(wd, 0, 6144, K, xd)
    parts = torch.full((1, 6144), float("nan"), device="cuda")
    for off, n in ((0, 4096), (4096, 1024), (5120, 1024)):
        fn(wd, off, n, K, xd, y=parts[:, off:], ldy=6144)
    torch.cuda.synchronize()
    assert torch.equal(fused, parts)


def test_expert_row_offsets(qk, orc):
    """3-D expert tensor [E][rows_e][K]: expert e is row_offset = e*rows_e."""
    E, rows_e, K = 6, 200, 1024
    wq = synth.weights("q4_k", E * rows_e, K, seed=4)
    x = synth.activations(2, K, seed=4)
    wd = torch.from_numpy(wq).cuda()
    xd = torch.from_numpy(x).cuda()
    for e in (0, 3, 5):
        y = qk.qmatvec_q4_k(wd, e * rows_e, rows_e, K, xd).cpu().numpy()
        yr, s = orc.gemv("q4_k", wq, K, x, rows=np.arange(e * rows_e, (e + 1) * rows_e))
        assert_close(y, yr, s, f"expert {e}")


def test_ldy_writes_only_the_range(qk, orc):
    fmt, rows, K, B, ldy = "q8_0", 500, 576, 3, 777
    wq = synth.weights(fmt, rows, K, seed=13)
    x = synth.activations(B, K, seed=13)
    y = torch.full((B, ldy), -7.0, device="cuda")
    gpu_gemv(qk, fmt, wq, 0, rows, K, x, y=y, ldy=ldy)
    yh = y.cpu().numpy()
    assert np.all(yh[:, rows:] == -7.0)
    yr, s = orc.gemv(fmt, wq, K, x)
    assert_close(yh[:, :rows], yr, s, "ldy")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_nonfinite_scales_propagate(qk, orc, fmt):
    rows, K = 64, 512
    wq = synth.weights(fmt, rows, K, seed=14)
    rec = wq.view(synth.BLOCK[fmt][2]).reshape(rows, -1)
    rec["d"][5, 0] = np.float16(np.nan)
    rec["d"][9, 1] = np.float16(np.inf)
    x = synth.activations(1, K, seed=14)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert np.isnan(y[0, 5]) and np.isnan(yr[0, 5])
    assert not np.isfinite(y[0, 9]) and not np.isfinite(yr[0, 9])
    keep = np.isfinite(yr[0])
    assert_close(y[:, keep], yr[:, keep], s[:, keep], "finite rows")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q6_k"])
@pytest.mark.parametrize("batch", [1, 2])
def test_nonfinite_activations_propagate(qk, orc, fmt, batch):
    """A NaN (or an infinity) in x makes every output of its batch row non-finite, as in the oracle."""
    rows, K = 48, 768
    wq = synth.weights(fmt, rows, K, seed=16)
    x = synth.activations(batch, K, seed=16)
    x[0, 37] = np.nan
    if batch > 1:
        x[1, 300] = np.inf
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert np.all(np.isnan(yr[0])) and np.all(np.isnan(y[0]))
    if batch > 1:
        assert not np.any(np.isfinite(yr[1])) and not np.any(np.isfinite(y[1]))


@pytest.mark.parametrize("fmt,K,batch", [("q4_k", 14336, 8), ("q4_k", 14336, 4), ("q6_k", 14336, 5),
                                         ("q8_0", 30000, 3), ("q4_k", 40960, 2)])
def test_batch_split_when_activations_do_not_fit(qk, orc, fmt, K, batch):
    """Batches whose activations exceed shared memory run as several launches of fewer rows."""
    rows = 37
    wq = synth.weights(fmt, rows, K, seed=17)
    x = synth.activations(batch, K, seed=17)
    with pytest.raises(qk.QKError):
        qk.debug_gemv_plan(fmt, rows, K, batch)          # the whole batch does not fit
    bmax = next(b for b in range(batch, 0, -1) if _fits(qk, fmt, rows, K, b))
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert_close(y, yr, s, f"split {fmt} K={K} B={batch}")
    # the launches are as even as possible; each part gives the bits of a call of its size
    parts = -(-batch // bmax)
    b0 = 0
    for p in range(parts):
        nb = (batch - b0) // (parts - p)
        yp = gpu_gemv(qk, fmt, wq, 0, rows, K, x[b0:b0 + nb]).cpu().numpy()
        assert np.array_equal(yp, y[b0:b0 + nb])
        b0 += nb


def _fits(qk, fmt, rows, K, b):
    try:
        qk.debug_gemv_plan(fmt, rows, K, b)
        return True
    except qk.QKError:
        return False


def test_too_large_is_rejected_before_launch(qk):
    """One activation row of K = 57344 (229 KB) does not fit in shared memory."""
    K, B = 14336 * 4, 8
    w = torch.zeros(qk.row_bytes("q4_k", K), dtype=torch.uint8, device="cuda")
    x = torch.zeros((B, K), device="cuda")
    y = torch.full((B, 1), 5.0, device="cuda")
    with pytest.raises(qk.QKError) as ei:
        qk.qmatvec_q4_k(w, 0, 1, K, x, y=y, ldy=1)
    assert ei.value.status == 8
    assert torch.all(y == 5.0)


@pytest.mark.parametrize("fmt,rows,K,nkc", [("q4_k", 2000, 4096, 1), ("q4_k", 4096, 14336, 2), ("q8_0", 900, 896, 1)])
def test_bounded_wait_times_out_and_context_survives(qk, orc, fmt, rows, K, nkc):
    """An item whose copy is never issued makes its warp's wait run out: the
    launch records QK_ERR_TIMEOUT and later launches work normally.  (The
    K = 14336 case splits rows into K chunks, one copy per row.)"""
    assert qk.debug_gemv_plan(fmt, rows, K, 1)["nkc"] == nkc
    wq = synth.weights(fmt, rows, K, seed=15)
    x = synth.activations(1, K, seed=15)
    assert qk.device_error() == 0
    old = qk.set_wait_limit_ns(20_000_000)
    qk.debug_skip_item(0)
    try:
        gpu_gemv(qk, fmt, wq, 0, rows, K, x)
        assert qk.device_error() == 6
    finally:
        qk.debug_skip_item(-1)
        qk.set_wait_limit_ns(old)
    assert qk.device_error() == 0
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert_close(y, yr, s, "after timeout")


# ---------------------------------------------------------------- full-size configurations
#
# Every output element is compared; the oracle runs on all host cores over
# row bands (the same code per output as the serial oracle).

LLAMA8B = [("attn_qkv", 6144, 4096), ("attn_output", 4096, 4096), ("ffn_gate_up", 28672, 4096),
           ("ffn_down", 4096, 14336)]


@pytest.mark.parametrize("name,rows,K", LLAMA8B)
def test_llama8b_layer_set_full(qk, orc, name, rows, K):
    """Full-size Llama-8B-shaped Q4_K tensors, batch 1, every row."""
    seed = 2
    wq = synth.weights("q4_k", rows, K, seed=seed, stream0=10 * LLAMA8B.index((name, rows, K)))
    x = synth.activations(1, K, seed=seed)
    y = gpu_gemv(qk, "q4_k", wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv_threaded("q4_k", wq, K, x, np.arange(rows), orc.host_cores())
    assert_close(y, yr, s, name)


@pytest.mark.parametrize("batch", [1, 8])
def test_lm_head_q8_0_full(qk, orc, batch):
    """Q8_0 lm_head 151936 x 896 (Qwen2.5-0.5B vocab), batch 1 and 8, every row."""
    rows, K, seed = 151936, 896, 3
    wq = synth.weights("q8_0", rows, K, seed=seed)
    x = synth.activations(batch, K, seed=seed)
    y = gpu_gemv(qk, "q8_0", wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv_threaded("q8_0", wq, K, x, np.arange(rows), orc.host_cores())
    assert_close(y, yr, s, f"lm_head b{batch}")


@pytest.mark.parametrize("fmt,rows,K,batch", [("q8_0", 576, 576, 1), ("q4_k", 4864, 896, 1),
                                               ("q4_k", 896, 4864, 1), ("q4_k", 28672, 4096, 4)])
def test_other_configs_full(qk, orc, fmt, rows, K, batch):
    """The SmolLM q-proj, the Qwen ffn_up and its transpose, and Llama-8B gate+up at batch 4."""
    seed = {576: 0, 4864: 1, 896: 1, 28672: 2}[rows]
    wq = synth.weights(fmt, rows, K, seed=seed)
    x = synth.activations(batch, K, seed=seed)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv_threaded(fmt, wq, K, x, np.arange(rows), orc.host_cores())
    assert_close(y, yr, s, f"{fmt} {rows}x{K} b{batch}")


def test_programmatic_launch_chain(qk, orc):
    """With programmatic dependent launch on, a chain whose every input is the
    previous call's output still sees each output complete."""
    K = 4096
    ws = [synth.weights("q4_k", K, K, seed=30 + i) for i in range(4)]
    x0 = synth.activations(1, K, seed=30)
    wd = [torch.from_numpy(w).cuda() for w in ws]
    old = qk.set_programmatic_launch(True)
    try:
        xs = [torch.from_numpy(x0).cuda()]
        for i in range(4):
            xs.append(qk.qmatvec_q4_k(wd[i], 0, K, K, xs[-1]))
        torch.cuda.synchronize()
    finally:
        qk.set_programmatic_launch(old)
    x = x0
    for i in range(4):
        got = xs[i + 1].cpu().numpy()
        yr, s = orc.gemv("q4_k", ws[i], K, x.astype(np.float32))
        # each stage is checked against the oracle fed with the GPU's own input
        assert_close(got, yr, s, f"stage {i}")
        x = xs[i + 1].cpu().numpy()


def test_binding_refuses_wrong_tensors_before_launch(qk):
    """Tensors too small for the call, of the wrong dtype or layout are refused
    by the binding with ValueError; nothing is launched and y is untouched."""
    K, rows = 512, 8
    rb = qk.row_bytes("q4_k", K)
    w = torch.zeros(rb * rows, dtype=torch.uint8, device="cuda")
    x = torch.zeros((2, K), device="cuda")
    y = torch.full((2, rows), 7.0, device="cuda")
    with pytest.raises(ValueError, match="w holds"):
        qk.qmatvec_q4_k(w, 1, rows, K, x, y=y)                        # rows 1..8 of an 8-row tensor
    with pytest.raises(ValueError, match="float32"):
        qk.qmatvec_q4_k(w, 0, rows, K, x.double(), y=y)
    with pytest.raises(ValueError, match=r"\[n\]\[512\]"):
        qk.qmatvec_q4_k(w, 0, rows, K, x[:, :256], y=y)
    with pytest.raises(ValueError, match="too small"):
        qk.qmatvec_q4_k(w, 0, rows, K, x, y=y[:, :4])
    with pytest.raises(ValueError, match="apart"):
        qk.qmatvec_q4_k(w, 0, rows, K, x, y=y, ldy=rows + 1)           # y's rows are 8 apart, not 9
    with pytest.raises(ValueError, match="int32"):
        qk.qmatvec_experts("q4_k", w, 2, rows // 2, K, x, 1, torch.zeros(2, dtype=torch.int64, device="cuda"))
    with pytest.raises(ValueError, match="reads row"):
        qk.qmatvec_experts("q4_k", w, 2, rows // 2, K, x, 1, torch.zeros(3, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


SPLIT = [("q4_k", 1, 14336), ("q4_k", 31, 14336), ("q4_k", 33, 20480), ("q4_k", 896, 4864),
         ("q8_0", 576, 20000), ("q8_0", 1, 8192), ("q6_k", 31, 14336), ("q6_k", 33, 8192)]


@pytest.mark.parametrize("fmt,rows,K", SPLIT)
@pytest.mark.parametrize("batch", [1, 3])
def test_split_k_over_warps_matches_oracle_and_unsplit_bits(qk, orc, fmt, rows, K, batch):
    """Calls with few rows a CTA share each row's K chunks among warps; the
    result equals the oracle and, bit for bit, the same rows of a call whose
    CTAs split K over a different number of warps (or not at all)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    smem = getattr(torch.cuda.get_device_properties(0), "shared_memory_per_block_optin", 232448)
    bb = batch                                      # the batch rows of one launch (the host splits larger ones)
    while qk.debug_gemv_plan_for(fmt, rows, K, bb, sms, smem) is None:
        bb -= 1
    p = qk.debug_gemv_plan_for(fmt, rows, K, bb, sms, smem)
    if p["kw"] == 1:
        pytest.skip(f"{fmt} {rows}x{K}: batch {bb} leaves no room to split")
    # the same rows in a larger call, split differently or not at all
    big = next(n for n in (4000, 16000) if qk.debug_gemv_plan_for(fmt, n, K, bb, sms, smem)["kw"] != p["kw"])
    wq = synth.weights(fmt, big, K, seed=18)
    x = synth.activations(batch, K, seed=18)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x, rows=np.arange(rows))
    assert_close(y, yr, s, f"split {fmt} {rows}x{K} b{batch}")
    y_big = gpu_gemv(qk, fmt, wq, 0, big, K, x).cpu().numpy()
    assert np.array_equal(y, y_big[:, :rows])
