"""Pins of the CPU oracle against facts fixed outside the oracle itself.

* fp16 / bf16 conversions against numpy's and torch's own conversions;
* the block-layout reading against hand-derived single-field probes
  (tests/golden/*_probes.txt);
* the dot product against unit-vector probes, all-zero and constant-block
  closed forms, exact integer arithmetic and a BLAS matmul;
* the encoders against their error bounds and nearest-value property;
* the bf16 GEMM reference against torch's bf16 rounding and against the
  exact reference on bf16-exact inputs;
* the SwiGLU product against known values of silu, its odd-part identity
  silu(z) - silu(-z) = z, and its limits;
* the expert matvec against experts whose rows reveal their own index.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth
from tests import golden_probes

FMTS = ["q8_0", "q4_k", "q6_k"]


# ------------------------------------------------------------ scalar codecs

def test_fp16_decode_every_pattern(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.fp16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_fp16_encode_matches_numpy(orc):
    rng = np.random.default_rng(0)
    mags = np.ldexp(rng.uniform(1.0, 2.0, 4000), rng.integers(-30, 18, 4000))
    vals = mags * rng.choice([-1.0, 1.0], 4000)
    # exact ties: midpoints between adjacent fp16 values (normal and subnormal)
    h = rng.integers(1, 0x7BFF, 2000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    vals = np.concatenate([vals, (lo + hi) / 2, [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9,
                                                 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26]])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.f64_to_fp16(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_round_matches_torch(orc):
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    u[:3000] = (u[:3000] & 0xFFFF0000) | 0x8000          # exact ties
    u[3000:4000] = (u[3000:4000] & 0xFFFF0000) | 0x7FFF
    f = u.view(np.float32)
    keep = ~np.isnan(f)
    f = f[keep]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16(v) for v in f], dtype=np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([orc.bf16_to_f64(int(b)) for b in got[:500]])
    ref_back = torch.from_numpy(ref[:500].view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    assert np.array_equal(back, ref_back)


# ------------------------------------------------------------ layout probes

@pytest.mark.parametrize("fmt", FMTS)
def test_layout_probes(orc, fmt):
    probes = golden_probes.load(fmt)
    assert len(probes) >= 6
    for name, K, raw, exp in probes:
        got = orc.decode(fmt, raw, K)[0]
        assert np.array_equal(got, exp), (name, np.nonzero(got != exp)[0][:8])


# ------------------------------------------------------------ dot product

@pytest.mark.parametrize("fmt,rows,K", [("q8_0", 3, 96), ("q4_k", 3, 512), ("q4_k", 2, 300),
                                        ("q8_0", 2, 40), ("q6_k", 3, 512), ("q6_k", 2, 300)])
def test_unit_vectors_recover_matrix(orc, fmt, rows, K):
    """x = e_c gives y[r] = W[r][c]: the dot indexes W row-major, column fastest."""
    wq = synth.weights(fmt, rows, K, seed=11)
    W = orc.decode(fmt, wq, K)
    eye = np.eye(K, dtype=np.float32)
    y, s = orc.gemv(fmt, wq, K, eye)
    assert np.array_equal(y, W.T)
    assert np.array_equal(s, np.abs(W.T))


@pytest.mark.parametrize("fmt", FMTS)
def test_all_zero_blocks(orc, fmt):
    K = 512
    wq = np.zeros(4 * synth.row_bytes(fmt, K), np.uint8)
    y, s = orc.gemv(fmt, wq, K, synth.activations(3, K, seed=2))
    assert np.all(y == 0.0) and np.all(s == 0.0)


@pytest.mark.parametrize("fmt,w_const,n_blocks", [("q8_0", 3.0, 7), ("q4_k", 2.5, 3), ("q6_k", 2.5, 3)])
def test_constant_block_closed_form(orc, fmt, w_const, n_blocks):
    """A row of identical constant blocks and x = v gives y = K * w * v exactly."""
    name, K0, raw, exp = [p for p in golden_probes.load(fmt) if p[0] == "constant_block"][0]
    assert np.all(exp == w_const)
    K = K0 * n_blocks
    wq = np.tile(raw, 2 * n_blocks)                      # 2 rows
    for v in (1.0, -0.75, 3.0):
        x = np.full((1, K), v, np.float32)
        y, s = orc.gemv(fmt, wq, K, x)
        assert np.all(y == K * w_const * v)
        assert np.all(s == K * abs(w_const * v))


@pytest.mark.parametrize("fmt", FMTS)
def test_exact_integer_dot(orc, fmt):
    """Power-of-two scales and small-integer x: every product and partial sum
    is exact in f64, so the oracle equals the exact rational dot."""
    rows, K, B = 3, 512, 2
    wq = synth.pow2_scaled_blocks(synth.weights(fmt, rows, K, seed=5), fmt, (-4, -3, -2, -1, 0), 5)
    x = synth.small_int_activations(B, K, seed=5)
    W = orc.decode(fmt, wq, K)
    y, _ = orc.gemv(fmt, wq, K, x)
    for b in range(B):
        for r in range(rows):
            exact = sum(Fraction(float(W[r, c])) * Fraction(float(x[b, c])) for c in range(K))
            assert Fraction(float(y[b, r])) == exact


@pytest.mark.parametrize("fmt,rows,K,B", [("q8_0", 17, 576, 3), ("q4_k", 9, 896, 2), ("q6_k", 9, 896, 2),
                                          ("q4_k", 5, 4096, 1)])
def test_dot_matches_blas(orc, fmt, rows, K, B):
    wq = synth.weights(fmt, rows, K, seed=3)
    x = synth.activations(B, K, seed=3)
    W = orc.decode(fmt, wq, K)
    y, s = orc.gemv(fmt, wq, K, x)
    ref = x.astype(np.float64) @ W.T
    sref = np.abs(x.astype(np.float64)) @ np.abs(W.T)
    assert np.all(np.abs(y - ref) <= 1e-13 * sref)
    assert np.allclose(s, sref, rtol=1e-13, atol=0)


def test_row_subset_equals_slice(orc):
    fmt, K = "q4_k", 512
    wq = synth.weights(fmt, 40, K, seed=9)
    x = synth.activations(2, K, seed=9)
    yall, _ = orc.gemv(fmt, wq, K, x)
    rows = [39, 0, 17, 17, 5]
    ysub, _ = orc.gemv(fmt, wq, K, x, rows=rows)
    assert np.array_equal(ysub, yall[:, rows])


def test_threaded_equals_serial(orc):
    fmt, K = "q8_0", 896
    wq = synth.weights(fmt, 301, K, seed=4)
    x = synth.activations(2, K, seed=4)
    y1, s1 = orc.gemv(fmt, wq, K, x)
    y2, s2 = orc.gemv_threaded(fmt, wq, K, x, np.arange(301), threads=4)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


# ------------------------------------------------------------ encoders

def test_q8_0_roundtrip_nearest(orc):
    rng = np.random.default_rng(7)
    K = 96
    w = rng.normal(0, 0.02, (6, K)) * rng.choice([1, 10, 0.01], (6, 1))
    w[5, :32] = 0.0                                       # all-zero block
    # tiny weights: d rounds to the fp16 subnormal 2^-24 and |w/d| > 127 clamps
    w[4] = rng.uniform(-1.0, 1.0, K) * 127 * 1.3 * 2.0 ** -24
    raw = orc.quantise("q8_0", w)
    wh = orc.decode("q8_0", raw, K)
    rec = raw.view(synth.Q8_0_DTYPE)
    d = rec["d"].astype(np.float64).reshape(6, -1)
    assert np.all(d[5, 0] == 0.0) and np.all(wh[5, :32] == 0.0)
    for r in range(6):
        for c in range(K):
            dd = d[r, c // 32]
            cands = dd * np.arange(-127, 128)
            best = np.min(np.abs(cands - w[r, c]))
            assert abs(wh[r, c] - w[r, c]) == best      # nearest representable value
    # error bound |w - w_hat| <= d/2 wherever no clamping happened
    dd = np.repeat(d, 32, axis=1)[:, :K]
    unclamped = np.abs(w) <= 127.5 * dd
    assert np.all((np.abs(wh - w) <= 0.5 * dd)[unclamped])
    assert not unclamped[4].all() and np.all(np.abs(wh[4]) <= 127 * dd[4])


def test_q4_k_roundtrip_bound(orc):
    rng = np.random.default_rng(8)
    K = 512
    w = rng.normal(0, 0.03, (5, K)) + rng.normal(0, 0.01, (5, 1))
    raw = orc.quantise("q4_k", w)
    wh = orc.decode("q4_k", raw, K)
    rec = raw.view(synth.Q4_K_DTYPE).reshape(5, -1)
    d = rec["d"].astype(np.float64)
    dmin = rec["dmin"].astype(np.float64)
    # grid step d*sc_j <= 63 d (half-step error 31.5 d); the grid's ends miss
    # [lo, hi] by at most 15 d/2 (rounding sc_j) plus dmin/2 (rounding m_j)
    bound = np.repeat(39.0 * d + 0.5 * dmin, 256, axis=1)
    assert np.all(np.abs(wh - w) <= bound)
    # 4-bit steps of about (6 sigma)/15 give an rms error near step/sqrt(12)
    assert np.sqrt(np.mean((wh - w) ** 2)) < 0.15 * np.std(w)


def test_q4_k_unit_scales_reduce_to_plain_nibbles(orc):
    """dmin = 0 and every 6-bit scale 1: a Q4_K super-block is d times its 4-bit
    quants, sub-block 2c in the low nibbles of qs[32c..32c+31] and 2c+1 in the
    high nibbles, whatever the (unused) mins hold."""
    rng = np.random.default_rng(21)
    nb = 6
    rec = np.zeros(nb, dtype=synth.Q4_K_DTYPE)
    rec["d"] = rng.uniform(0.01, 2.0, nb).astype(np.float16)
    rec["dmin"] = 0.0
    sc = np.zeros((nb, 12), np.uint8)
    sc[:, 0:4] = 1                                          # sc of sub-blocks 0..3, top bits 0
    sc[:, 4:8] = rng.integers(0, 256, (nb, 4))              # mins of 0..3 and top bits of mins 4..7
    sc[:, 8:12] = 1 | (rng.integers(0, 16, (nb, 4)) << 4)   # sc of 4..7 = 1, mins of 4..7 above
    rec["scales"] = sc
    rec["qs"] = rng.integers(0, 256, (nb, 128))
    W = orc.decode("q4_k", rec.view(np.uint8).reshape(-1), 3 * 256)     # 2 rows of 3 super-blocks
    qs = rec["qs"].reshape(nb, 4, 32).astype(np.float64)
    expect = np.empty((nb, 256))
    for c in range(4):
        expect[:, 64 * c:64 * c + 32] = np.mod(qs[:, c], 16)
        expect[:, 64 * c + 32:64 * c + 64] = np.floor(qs[:, c] / 16)
    expect *= rec["d"].astype(np.float64)[:, None]
    assert np.array_equal(W.reshape(nb, 256), expect)


def test_q8_0_requantise_reproduces_the_bytes(orc):
    """A Q8_0 block whose largest |q| is 127 re-encodes to exactly its own
    bytes: amax/127 gives back d and w/d gives back every q."""
    K = 320
    rec = synth.weights("q8_0", 5, K, seed=22).view(synth.Q8_0_DTYPE).copy()
    rec["d"] = np.where(rec["d"] == 0, np.float16(1.0), rec["d"])
    rec["qs"][:, 7] = np.where(np.arange(len(rec)) % 2 == 0, 127, -127)
    raw = rec.view(np.uint8).reshape(-1)
    back = orc.quantise("q8_0", orc.decode("q8_0", raw, K))
    assert np.array_equal(back, raw)


def test_q4_k_bytes_per_weight_give_the_page_intensity(orc):
    """144 bytes per 256 weights is 0.5625 B a weight; 2 flop a weight over
    that is the ~3.55 flop/B the nx_f32_llm_v4.nx source gives for Q4 (3.556
    cut to two decimals), and a second row starts 144 bytes later."""
    assert orc.row_bytes("q4_k", 256) == 144
    assert orc.row_bytes("q4_k", 4096) / 4096 == 0.5625
    assert int(2 / 0.5625 * 100) == 355
    raw = synth.weights("q4_k", 2, 256, seed=23)
    both = orc.decode("q4_k", raw, 256)
    assert np.array_equal(both[1], orc.decode("q4_k", raw[144:], 256)[0])
    assert not np.array_equal(both[0], both[1])


def test_q4_k_requantise_is_fixed_point_for_probes(orc):
    """Decoding the hand-derived constant block, re-encoding and decoding again
    gives the same weights (the encoder reproduces exactly representable rows)."""
    name, K, raw, exp = [p for p in golden_probes.load("q4_k") if p[0] == "constant_block"][0]
    wh = orc.decode("q4_k", orc.quantise("q4_k", exp[None, :]), K)
    assert np.allclose(wh[0], exp, rtol=2e-3)


# ------------------------------------------------------------ bf16 GEMM reference

def test_gemm_bf16_reference_matches_torch_rounding(orc):
    fmt, rows, K, M = "q4_k", 6, 512, 5
    wq = synth.weights(fmt, rows, K, seed=12)
    x = synth.activations(M, K, seed=12)
    W = orc.decode(fmt, wq, K)
    y2, s2 = orc.gemm_bf16(fmt, wq, K, x)
    Wb = torch.from_numpy(W).float().bfloat16().double()
    xb = torch.from_numpy(x).bfloat16().double()
    ref = (xb @ Wb.T).numpy()
    sref = (xb.abs() @ Wb.abs().T).numpy()
    assert np.all(np.abs(y2 - ref) <= 1e-13 * sref)
    # and it differs from the exact reference by at most two bf16 roundings
    y1, s1 = orc.gemv(fmt, wq, K, x)
    assert np.all(np.abs(y2 - y1) <= 2 * 2.0 ** -8 * s1)


def test_gemm_bf16_reference_exact_on_bf16_inputs(orc):
    """Weights and activations already representable in bf16: both references agree."""
    names = ("constant_block", "chunk2_low_nibble_scale_high_bits", "min_subblock7_high_bits",
             "full_formula_subblock6")
    probes = {p[0]: p for p in golden_probes.load("q4_k")}
    K = 256
    wq = np.concatenate([probes[n][2] for n in names])
    W = np.stack([probes[n][3] for n in names])
    exact_bf16 = torch.from_numpy(W).float().bfloat16().double().numpy() == W
    x = synth.small_int_activations(4, K, seed=1, lo=-3, hi=3)
    y1, _ = orc.gemv("q4_k", wq, K, x)
    y2, _ = orc.gemm_bf16("q4_k", wq, K, x)
    rows_exact = exact_bf16.all(axis=1)
    assert rows_exact[:3].all() and not rows_exact[3]     # 981 needs 10 significant bits
    assert np.array_equal(y1[:, :3], y2[:, :3])
    assert not np.array_equal(y1[:, 3], y2[:, 3])


# ------------------------------------------------------------ SwiGLU

def _unit_rows_q8_0(n_rows: int) -> np.ndarray:
    """Q8_0 rows of one block (K = 32), row i = the unit vector e_i (d = 1, q_i = 1)."""
    rec = np.zeros(n_rows, dtype=synth.Q8_0_DTYPE)
    rec["d"] = np.float16(1.0)
    for i in range(n_rows):
        rec["qs"][i, i] = 1
    return rec.view(np.uint8).copy()


def _swiglu_of(orc, z: float, v: float) -> float:
    """h for gate value z and up value v: gate row e_0, up row e_1, x = (z, v, 0...)."""
    wq = _unit_rows_q8_0(2)
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = z, v
    h, g, u, sg, su = orc.swiglu("q8_0", wq, 32, x, [0], [1])
    assert g[0, 0] == np.float32(z) and u[0, 0] == np.float32(v)
    return float(h[0, 0])


def test_swiglu_known_values(orc):
    """silu(ln 3) = (3/4) ln 3; silu(0) = 0; silu(z) -> z for large z and -> 0 for very negative z."""
    ln3 = float(np.float32(np.log(3.0)))
    assert abs(_swiglu_of(orc, ln3, 2.0) - 2.0 * 0.75 * 1.0986122886681098) < 3e-7
    assert _swiglu_of(orc, 0.0, 5.0) == 0.0
    assert abs(_swiglu_of(orc, 40.0, 1.5) - 60.0) < 1e-12
    assert abs(_swiglu_of(orc, -50.0, 3.0)) < 1e-18           # the gate, not the up value, goes through silu


@pytest.mark.parametrize("z", [0.3, 1.75, 5.5, 12.0])
def test_swiglu_odd_part_identity(orc, z):
    """sigma(z) + sigma(-z) = 1 makes silu(z) - silu(-z) = z."""
    assert abs((_swiglu_of(orc, z, 1.0) - _swiglu_of(orc, -z, 1.0)) - np.float32(z)) < 1e-14 * (1 + z)


def test_swiglu_uses_the_given_rows(orc):
    """h[b][p] pairs gate row gate_rows[p] with up row up_rows[p], for every batch row."""
    wq = _unit_rows_q8_0(4)
    x = synth.activations(3, 32, seed=9)
    h, g, u, _, _ = orc.swiglu("q8_0", wq, 32, x, [2, 0], [1, 3])
    assert np.array_equal(g, x[:, [2, 0]].astype(np.float64))
    assert np.array_equal(u, x[:, [1, 3]].astype(np.float64))
    assert np.all(np.abs(h) <= np.abs(g * u) + 1e-300)       # |silu(z)| <= |z|


# ------------------------------------------------------------ experts

def _tagged_experts_q8_0(n_experts: int, rows: int) -> np.ndarray:
    """Q8_0 expert tensor [E][rows][32]: row r of expert e is (e + 1) * e_r."""
    rec = np.zeros(n_experts * rows, dtype=synth.Q8_0_DTYPE)
    for e in range(n_experts):
        for r in range(rows):
            rec["d"][e * rows + r] = np.float16(e + 1)
            rec["qs"][e * rows + r, r] = 1
    return rec.view(np.uint8).copy()


@pytest.mark.parametrize("xk", [1, 2, 3])
def test_experts_select_expert_and_input_row(orc, xk):
    """y[a][r] = (expid[a] + 1) * x[a // xk][r]: the expert, its rows and the input row are the stated ones."""
    E, rows, n = 5, 7, 6
    wq = _tagged_experts_q8_0(E, rows)
    ids = np.array([3, 0, 4, 4, 1, 2], np.int32)
    x = synth.small_int_activations((n + xk - 1) // xk, 32, seed=3)
    y, s = orc.experts("q8_0", wq, E, rows, 32, x, xk, ids)
    for a in range(n):
        assert np.array_equal(y[a], (ids[a] + 1) * x[a // xk, :rows].astype(np.float64))


def test_swiglu_gemm_reference_on_bf16_exact_inputs(orc):
    """Weights and activations exact in bf16: the bf16 GEMM form of SwiGLU equals
    the exact one, and a unit-vector gate/up pair gives silu(x0) * x1."""
    wq = _unit_rows_q8_0(4)
    x = np.zeros((3, 32), np.float32)
    x[:, 0] = [0.5, -2.0, 3.0]          # bf16-exact values
    x[:, 1] = [1.0, 0.25, -1.5]
    h, g, u, _, _ = orc.swiglu_gemm_bf16("q8_0", wq, 32, x, [0], [1])
    he, _, _, _, _ = orc.swiglu("q8_0", wq, 32, x, [0], [1])
    assert np.array_equal(h, he)
    assert np.array_equal(g[:, 0], x[:, 0].astype(np.float64)) and np.array_equal(u[:, 0], x[:, 1].astype(np.float64))
    assert abs(h[0, 0] - 0.5 / (1 + np.exp(-0.5)) * 1.0) < 1e-15


def test_swiglu_gemm_reference_rounds_to_bf16(orc):
    """A gate value that bf16 cannot hold is rounded before silu: x0 = 1 + 2^-9
    is bf16 1.0 (ties to even), so g = 1 exactly."""
    wq = _unit_rows_q8_0(2)
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 1.0 + 2.0 ** -9, 1.0
    h, g, u, _, _ = orc.swiglu_gemm_bf16("q8_0", wq, 32, x, [0], [1])
    assert g[0, 0] == 1.0
    assert abs(h[0, 0] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15
