"""Batch-1 GEMV parity on activations of wide dynamic range.

The batch-1 kernels hold x per 32-column group as integers that share one
binary exponent.  A shared exponent loses the small values of a group that
also holds a much larger one, so these inputs are built to break it: one
value per group 2^20 or 2^30 times the others (with the weights at those
columns set to zero in half of the rows, so that sum|w*x| does not hide the
error), tiny values, outlier channels 100 to 1000 times the rest, and fp32
subnormals.  Every case is checked element by element against the f64
oracle at the fp32 tolerance |y - y_ref| <= 1e-5 * sum|w*x| + 1e-6, for
Q8_0, Q4_K and Q6_K, and through the SwiGLU and expert forms.

Two large values in one group (both 2^20 times the rest) fall outside what
the encoding keeps exact: the other values of the group then carry an error
of at most 2^-20 times the group's second largest magnitude.  Those rows are
checked against that stated bound, the rows whose weights are random against
the plain tolerance.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth
from tests.test_gemv import REL, ABS, assert_close, gpu_gemv
from tests.test_swiglu import assert_swiglu_close

pytestmark = pytest.mark.gpu

FMTS = ["q8_0", "q4_k", "q6_k"]
EXACT_KINDS = ["group_outlier_2p20", "group_outlier_2p30", "group_tiny_2m30", "outlier_channels",
               "subnormal", "mixed_subnormal"]


def zero_weights_at(fmt, wq, K, rows, cols, row_sel):
    """Copy of the tensor whose weights W[r][c] are 0 for c in cols and r in row_sel.

    Q8_0: the quant is 0.  Q4_K: dmin is 0 in the rows' super-blocks and the
    nibble is 0.  Q6_K: the 6-bit quant is 32.  (Byte positions as in the
    block layouts stated in include/qk.h.)
    """
    out = wq.copy()
    rec = out.view(synth.BLOCK[fmt][2]).reshape(rows, -1)
    for r in row_sel:
        for c in cols:
            if fmt == "q8_0":
                rec["qs"][r, c // 32, c % 32] = 0
            elif fmt == "q4_k":
                b, j, i = c // 256, (c % 256) // 32, c % 32
                rec["dmin"][r, :] = 0
                byte = 32 * (j // 2) + i
                keep = 0xF0 if j % 2 == 0 else 0x0F
                rec["qs"][r, b, byte] &= keep
            else:
                b, cc = c // 256, c % 256
                n, cc = cc // 128, cc % 128
                t, l = cc // 32, cc % 32
                qi = 64 * n + l + 32 * (t % 2)
                if t < 2:
                    rec["ql"][r, b, qi] &= 0xF0            # low 4 bits 0
                else:
                    rec["ql"][r, b, qi] &= 0x0F
                hi = 32 * n + l
                keep2 = np.uint8(~(3 << (2 * t)) & 0xFF)
                rec["qh"][r, b, hi] = (rec["qh"][r, b, hi] & keep2) | np.uint8(2 << (2 * t))
    return out


def _case(fmt, kind, rows=256, K=1024, seed=70):
    x, cols = synth.wide_range_activations(1, K, seed=seed, kind=kind)
    wq = synth.weights(fmt, rows, K, seed=seed)
    zrows = np.arange(0, rows, 2)
    if cols[0].size:
        wq = zero_weights_at(fmt, wq, K, rows, cols[0], zrows)
    return wq, x, cols[0], zrows


@pytest.mark.parametrize("kind", EXACT_KINDS)
@pytest.mark.parametrize("fmt", FMTS)
def test_wide_range_activations_match_oracle(qk, orc, fmt, kind):
    rows, K = 256, 1024
    wq, x, cols, zrows = _case(fmt, kind, rows, K)
    if cols.size:
        W = orc.decode(fmt, wq, K, rows=zrows)
        assert np.all(W[:, cols] == 0.0)                     # the large values meet zero weights
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert_close(y, yr, s, f"{fmt} {kind}")


@pytest.mark.parametrize("fmt", FMTS)
def test_constructed_group_outlier_one_group(qk, orc, fmt):
    """One 32-column group {2^20, 31 x 0.3} against a zero weight at the 2^20."""
    rows, K = 64, 32 if fmt == "q8_0" else 256
    x = np.full((1, K), 0.3, np.float32)
    x[0, 0] = 2.0 ** 20
    wq = zero_weights_at(fmt, synth.weights(fmt, rows, K, seed=71), K, rows, [0], range(rows))
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert_close(y, yr, s, f"{fmt} constructed")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("K", [300, 4096, 14336])
def test_outlier_channels_shapes(qk, orc, fmt, K):
    """Outlier channels at the Llama-8B widths and a ragged K (the wide and K-chunked kernel forms)."""
    rows = 700
    wq, x, cols, zrows = _case(fmt, "outlier_channels", rows, K, seed=72)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy()
    yr, s = orc.gemv(fmt, wq, K, x)
    assert_close(y, yr, s, f"{fmt} K={K}")


def _group_bound(fmt, orc, wq, K, rows, x):
    """2^-20 * sum over 32-column groups of (second largest |x| of the group) * sum|w| of the group."""
    W = orc.decode(fmt, wq, K, rows=np.arange(rows))
    ng = (K + 31) // 32
    xa = np.zeros(ng * 32)
    xa[:K] = np.abs(x[0].astype(np.float64))
    a2 = np.sort(xa.reshape(ng, 32), axis=1)[:, -2]
    Wa = np.zeros((rows, ng * 32))
    Wa[:, :K] = np.abs(W)
    return 2.0 ** -20 * (Wa.reshape(rows, ng, 32).sum(axis=2) * a2[None, :]).sum(axis=1)


def factorised_magnitude(fmt, orc, wq, K, rows, x):
    """sum over c of the magnitudes of the two terms a weight is computed from,
    times |x[c]|: Q4_K |d*sc*q| + |dmin*m|, Q6_K |d*scale*q| + |32*d*scale|,
    Q8_0 |w| (the oracle decodes copies with one term removed)."""
    rec_dtype = synth.BLOCK[fmt][2]
    ax = np.abs(x[0].astype(np.float64))
    W = orc.decode(fmt, wq, K, rows=np.arange(rows))
    if fmt == "q8_0":
        return np.abs(W) @ ax
    if fmt == "q4_k":
        a = wq.copy()
        a.view(rec_dtype)["dmin"] = 0
        A = orc.decode(fmt, a, K, rows=np.arange(rows))            # d*sc*q
        return (np.abs(A) + np.abs(W - A)) @ ax
    z = wq.copy()
    z.view(rec_dtype)["ql"] = 0
    z.view(rec_dtype)["qh"] = 0
    W0 = orc.decode(fmt, z, K, rows=np.arange(rows))               # -32*d*scale
    return (np.abs(W - W0) + np.abs(W0)) @ ax


@pytest.mark.parametrize("fmt", FMTS)
def test_two_large_values_per_group(qk, orc, fmt):
    """Both large values of a group meet zero weights in half of the rows: those rows are
    checked against the stated bound (the fp32 tolerance on the factorised magnitudes plus
    2^-20 of each group's second largest |x| times the group's sum|w|)."""
    rows, K = 256, 1024
    wq, x, cols, zrows = _case(fmt, "two_large_per_group", rows, K, seed=73)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy().astype(np.float64)
    yr, s = orc.gemv(fmt, wq, K, x)
    other = np.setdiff1d(np.arange(rows), zrows)
    assert_close(y[:, other], yr[:, other], s[:, other], f"{fmt} random weights")
    bound = REL * factorised_magnitude(fmt, orc, wq, K, rows, x) + ABS + _group_bound(fmt, orc, wq, K, rows, x)
    assert np.all(np.abs(y[0] - yr[0]) <= bound)


@pytest.mark.parametrize("fmt", ["q4_k", "q6_k"])
@pytest.mark.parametrize("batch", [1, 2])
def test_cancelling_weight_terms_meet_the_factorised_bound(qk, orc, fmt, batch):
    """Weights whose two terms cancel (Q4_K d*sc*q = dmin*m, Q6_K q = 32) are near
    zero while each term is not: the kernels sum the terms separately, so these rows
    are held to the fp32 tolerance on the sum of the terms' magnitudes."""
    rows, K = 128, 1024
    wq = synth.weights(fmt, rows, K, seed=77)
    rec = wq.view(synth.BLOCK[fmt][2]).reshape(rows, -1)
    if fmt == "q4_k":
        # d = dmin, every scale and min 1, every nibble 1: w = d*1*1 - d*1 = 0 in row 0..63
        rec["dmin"][:64] = rec["d"][:64]
        rec["scales"][:64, :, :8] = 0x01                       # sc = m = 1 for sub-blocks 0..3
        rec["scales"][:64, :, 8:] = 0x11                       # and 4..7
        rec["qs"][:64] = 0x11
    else:
        # q = 32 (low 4 bits 0, high 2 bits 2) in rows 0..63
        rec["ql"][:64] = 0x00
        rec["qh"][:64] = 0xAA
    x = synth.activations(batch, K, seed=77)
    y = gpu_gemv(qk, fmt, wq, 0, rows, K, x).cpu().numpy().astype(np.float64)
    yr, s = orc.gemv(fmt, wq, K, x)
    W = orc.decode(fmt, wq, K, rows=np.arange(64))
    assert np.all(W == 0.0)
    for b in range(batch):
        bound = REL * factorised_magnitude(fmt, orc, wq, K, rows, x[b:b + 1]) + ABS
        assert np.all(np.abs(y[b] - yr[b]) <= bound), f"{fmt} batch row {b}"
    assert_close(y[:, 64:], yr[:, 64:], s[:, 64:], f"{fmt} random rows")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("kind", ["group_outlier_2p20", "outlier_channels"])
def test_wide_range_swiglu_b1(qk, orc, fmt, kind):
    F, K = 200, 1024
    x, cols = synth.wide_range_activations(1, K, seed=74, kind=kind)
    wq = zero_weights_at(fmt, synth.weights(fmt, 2 * F, K, seed=74), K, 2 * F, cols[0],
                         np.concatenate([np.arange(0, F, 2), F + np.arange(1, F, 2)]))
    wd = torch.from_numpy(wq).cuda()
    h = qk.qmatvec_swiglu(fmt, wd, 0, F, F, K, torch.from_numpy(x).cuda()).cpu().numpy()
    ref = orc.swiglu(fmt, wq, K, x, np.arange(F), np.arange(F, 2 * F))
    assert_swiglu_close(h, ref, f"{fmt} swiglu {kind}")


@pytest.mark.parametrize("fmt", FMTS)
def test_wide_range_experts_b1(qk, orc, fmt):
    E, rows, K, xk = 4, 128, 1024, 4
    x, cols = synth.wide_range_activations(1, K, seed=75, kind="group_outlier_2p30")
    wq = zero_weights_at(fmt, synth.weights(fmt, E * rows, K, seed=75), K, E * rows, cols[0],
                         np.arange(0, E * rows, 3))
    ids = np.array([3, 0, 2, 3], np.int32)
    y = qk.qmatvec_experts(fmt, torch.from_numpy(wq).cuda(), E, rows, K, torch.from_numpy(x).cuda(), xk,
                           torch.from_numpy(ids).cuda()).cpu().numpy()
    yr, s = orc.experts(fmt, wq, E, rows, K, x, xk, ids)
    assert_close(y, yr, s, f"{fmt} experts")


@pytest.mark.parametrize("fmt", FMTS)
def test_outlier_rows_ranges_equal_fused_call(qk, fmt):
    """Row-range calls give the bits of one call with outliers in x too."""
    rows, K = 3000, 4096
    x, _ = synth.wide_range_activations(1, K, seed=76, kind="outlier_channels")
    wd = torch.from_numpy(synth.weights(fmt, rows, K, seed=76)).cuda()
    xd = torch.from_numpy(x).cuda()
    fn = {"q8_0": qk.qmatvec_q8_0, "q4_k": qk.qmatvec_q4_k, "q6_k": qk.qmatvec_q6_k}[fmt]
    whole = fn(wd, 0, rows, K, xd)
    parts = torch.full((1, rows), float("nan"), device="cuda")
    for off, n in ((0, 2000), (2000, 999), (2999, 1)):
        fn(wd, off, n, K, xd, y=parts[:, off:], ldy=rows)
    torch.cuda.synchronize()
    assert torch.equal(whole, parts)
