"""GPU parity of the batched expert GEMV against the oracle.

y[a][r] = sum_c W[expert_ids[a]*rows + r][c] x[a // xk][c]; tolerance as the
plain GEMV: |y - y_ref| <= 1e-5 * sum|w*x| + 1e-6.
"""
import numpy as np
import pytest
import torch

from quantised_gguf_weight_gb300 import synth
from tests.test_gemv import assert_close

pytestmark = pytest.mark.gpu


def run(qk, fmt, wq, E, rows, K, x, xk, ids, y=None, ldy=0):
    wd = torch.from_numpy(np.ascontiguousarray(wq)).cuda()
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    idd = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    out = qk.qmatvec_experts(fmt, wd, E, rows, K, xd, xk, idd, y=y, ldy=ldy)
    torch.cuda.synchronize()
    return out


CASES = [
    # fmt, E, rows, K, xk, n_assign, seed
    ("q8_0", 8, 200, 1024, 8, 8, 30), ("q8_0", 6, 333, 896, 2, 6, 31), ("q8_0", 4, 64, 2080, 1, 5, 32),
    ("q4_k", 8, 200, 1024, 8, 8, 33), ("q4_k", 16, 768, 2048, 4, 16, 34), ("q4_k", 5, 77, 300, 3, 7, 35),
    ("q4_k", 3, 40, 14336, 1, 3, 36), ("q4_k", 2, 1, 256, 1, 2, 37),
]


@pytest.mark.parametrize("fmt,E,rows,K,xk,n,seed", CASES)
def test_experts_match_oracle(qk, orc, fmt, E, rows, K, xk, n, seed):
    wq = synth.weights(fmt, E * rows, K, seed=seed)
    x = synth.activations((n + xk - 1) // xk, K, seed=seed)
    ids = synth.randint(seed, 40, n, 0, E - 1).astype(np.int32)
    ids[0] = E - 1                                   # the last expert is used
    y = run(qk, fmt, wq, E, rows, K, x, xk, ids).cpu().numpy()
    yr, s = orc.experts(fmt, wq, E, rows, K, x, xk, ids)
    assert_close(y, yr, s, f"{fmt} E={E} rows={rows} K={K} xk={xk} n={n}")


def test_experts_equal_plain_row_offset_calls(qk):
    """Each assignment gives the same bits as the plain GEMV on row_offset = e*rows."""
    E, rows, K, xk, n = 6, 300, 2048, 3, 6
    wq = synth.weights("q4_k", E * rows, K, seed=38)
    x = synth.activations(2, K, seed=38)
    ids = np.array([5, 0, 2, 2, 4, 1], np.int32)
    y = run(qk, "q4_k", wq, E, rows, K, x, xk, ids)
    wd = torch.from_numpy(wq).cuda()
    xd = torch.from_numpy(x).cuda()
    for a in range(n):
        ya = qk.qmatvec_q4_k(wd, int(ids[a]) * rows, rows, K, xd[a // xk:a // xk + 1])
        assert torch.equal(y[a:a + 1], ya), a


def test_experts_bad_id_is_reported_and_not_read(qk, orc):
    E, rows, K, xk = 4, 100, 512, 1
    wq = synth.weights("q8_0", E * rows, K, seed=39)
    x = synth.activations(3, K, seed=39)
    ids = np.array([1, 4, 2], np.int32)              # 4 is out of range
    assert qk.device_error() == 0
    y = run(qk, "q8_0", wq, E, rows, K, x, xk, ids).cpu().numpy()
    assert qk.device_error() == 9
    assert qk.device_error() == 0
    assert np.all(np.isnan(y[1]))
    yr, s = orc.experts("q8_0", wq, E, rows, K, x[[0, 2]], 1, ids[[0, 2]])
    assert_close(y[[0, 2]], yr, s, "valid assignments")


def test_experts_ldy(qk, orc):
    E, rows, K, xk, n, ldy = 3, 50, 512, 1, 3, 71
    wq = synth.weights("q4_k", E * rows, K, seed=41)
    x = synth.activations(n, K, seed=41)
    ids = np.array([2, 2, 0], np.int32)
    ybuf = torch.full((n, ldy), 3.0, device="cuda")
    run(qk, "q4_k", wq, E, rows, K, x, xk, ids, y=ybuf, ldy=ldy)
    y = ybuf.cpu().numpy()
    yr, s = orc.experts("q4_k", wq, E, rows, K, x, xk, ids)
    assert_close(y[:, :rows], yr, s, "ldy")
    assert np.all(y[:, rows:] == 3.0)


def test_experts_moe_layer_full(qk, orc):
    """A MoE FFN's fused gate+up experts: 128 experts x 1536 rows x 2048, one token, top 8."""
    E, rows, K, xk = 128, 1536, 2048, 8
    wq = synth.weights("q4_k", E * rows, K, seed=42)
    x = synth.activations(1, K, seed=42)
    ids = np.array([3, 17, 64, 127, 90, 5, 33, 0], np.int32)
    y = run(qk, "q4_k", wq, E, rows, K, x, xk, ids).cpu().numpy()
    yr, s = orc.experts("q4_k", wq, E, rows, K, x, xk, ids)
    assert_close(y, yr, s, "moe top 8, every row")
