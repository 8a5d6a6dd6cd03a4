"""GPU parity of the fused gate/up GEMV with the SwiGLU product against the oracle.

h = silu(g) * u with g, u the gate and up matvecs.  The kernel computes g and
u like the plain GEMV, each within e_g = 1e-5 * S_g + 1e-6 (S = sum|w*x|), so

  |h - h_ref| <= 1.1 * e_g * |u| + (|silu(g)| + 1.1 * e_g) * e_u + 2e-6 * |h_ref|

because |silu'| <= 1.0998 everywhere (the first two terms carry the matvec
errors through silu(g) * u), and the fp32 evaluation of silu (CUDA's expf,
its fast division: within 2 ulp) and of the product adds a few units in the
last place of h, covered by the relative term.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth

pytestmark = pytest.mark.gpu


def silu(z):
    with np.errstate(over="ignore"):          # e^-z = inf for very negative z gives silu = -0
        return z / (1.0 + np.exp(-z))


def assert_swiglu_close(h, ref, what=""):
    hr, g, u, sg, su = ref
    h = np.asarray(h, dtype=np.float64)
    eg = 1e-5 * sg + 1e-6
    eu = 1e-5 * su + 1e-6
    tol = 1.1 * eg * np.abs(u) + (np.abs(silu(g)) + 1.1 * eg) * eu + 2e-6 * np.abs(hr)
    bad = ~(np.abs(h - hr) <= tol)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {i}: "
                             f"gpu {h[i]!r} oracle {hr[i]!r} g {g[i]!r} u {u[i]!r} tol {tol[i]!r}")


def run(qk, fmt, wq, gate_off, up_off, F, K, x, h=None, ldh=0):
    wd = torch.from_numpy(np.ascontiguousarray(wq)).cuda()
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = qk.qmatvec_swiglu(fmt, wd, gate_off, up_off, F, K, xd, h=h, ldh=ldh)
    torch.cuda.synchronize()
    return out


CASES = [
    # fmt, F, K, batch, seed  (fused tensor: gate rows 0..F-1, up rows F..2F-1)
    ("q8_0", 300, 896, 1, 20), ("q8_0", 300, 896, 2, 20), ("q8_0", 300, 896, 3, 20),
    ("q8_0", 37, 2080, 8, 21), ("q8_0", 129, 4096, 1, 22),
    ("q4_k", 256, 1024, 1, 23), ("q4_k", 256, 1024, 2, 23), ("q4_k", 256, 1024, 4, 23),
    ("q4_k", 100, 1024, 5, 23), ("q4_k", 100, 1024, 8, 23),
    ("q4_k", 1000, 4096, 1, 24), ("q4_k", 61, 300, 3, 25),          # ragged F and K
    ("q4_k", 150, 14336, 1, 26), ("q4_k", 77, 14336, 2, 26),        # rows cut into K chunks
    ("q4_k", 1, 256, 1, 27), ("q4_k", 3, 33, 6, 27),
]


@pytest.mark.parametrize("fmt,F,K,batch,seed", CASES)
def test_swiglu_matches_oracle(qk, orc, fmt, F, K, batch, seed):
    wq = synth.weights(fmt, 2 * F, K, seed=seed)
    x = synth.activations(batch, K, seed=seed)
    h = run(qk, fmt, wq, 0, F, F, K, x).cpu().numpy()
    ref = orc.swiglu(fmt, wq, K, x, np.arange(F), np.arange(F, 2 * F))
    assert_swiglu_close(h, ref, f"{fmt} F={F} K={K} B={batch}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_swiglu_offsets_and_ldh(qk, orc, fmt):
    """Up rows before the gate rows, a gap between them, and ldh > F."""
    K, F, B = 512, 90, 2
    wq = synth.weights(fmt, 300, K, seed=28)
    x = synth.activations(B, K, seed=28)
    gate, up, ldh = 200, 7, 131
    hbuf = torch.full((B, ldh), 7.0, device="cuda")
    run(qk, fmt, wq, gate, up, F, K, x, h=hbuf, ldh=ldh)
    h = hbuf.cpu().numpy()
    ref = orc.swiglu(fmt, wq, K, x, np.arange(gate, gate + F), np.arange(up, up + F))
    assert_swiglu_close(h[:, :F], ref, "offsets")
    assert np.all(h[:, F:] == 7.0)


def test_swiglu_row_ranges_equal_one_call(qk):
    """Output rows computed in parts give the same bits as one call."""
    K, F = 4096, 2000
    wd = torch.from_numpy(synth.weights("q4_k", 2 * F, K, seed=29)).cuda()
    xd = torch.from_numpy(synth.activations(1, K, seed=29)).cuda()
    whole = qk.qmatvec_swiglu("q4_k", wd, 0, F, F, K, xd)
    parts = torch.full((1, F), float("nan"), device="cuda")
    for off, n in ((0, 1500), (1500, 400), (1900, 100)):
        qk.qmatvec_swiglu("q4_k", wd, off, F + off, n, K, xd, h=parts[:, off:], ldh=F)
    torch.cuda.synchronize()
    assert torch.equal(whole, parts)


def test_swiglu_llama8b_ffn_full(qk, orc):
    """Llama-8B ffn gate+up (one fused 28672 x 4096 tensor), batch 1, every output."""
    K, F = 4096, 14336
    wq = synth.weights("q4_k", 2 * F, K, seed=2, stream0=20)
    x = synth.activations(1, K, seed=2)
    h = run(qk, "q4_k", wq, 0, F, F, K, x).cpu().numpy()
    idx = np.arange(F)
    ref = orc.swiglu("q4_k", wq, K, x, idx, idx + F)
    assert_swiglu_close(h, ref, "llama8b ffn")


def test_swiglu_rejects_bad_arguments(qk):
    w = torch.zeros(qk.row_bytes("q4_k", 256) * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 256), device="cuda")
    lib = qk.load()
    h = torch.zeros((1, 2), device="cuda")
    assert lib.qmatvec_swiglu_q4_k(w.data_ptr(), 0, -1, 2, 256, x.data_ptr(), 1, h.data_ptr(), 0, 0) == 2
    assert lib.qmatvec_swiglu_q4_k(w.data_ptr(), 0, 2, 2, 256, x.data_ptr(), 9, h.data_ptr(), 0, 0) == 4
    assert lib.qmatvec_swiglu_q4_k(0, 0, 2, 2, 256, x.data_ptr(), 1, h.data_ptr(), 0, 0) == 1
