"""Host-side checks of the GEMV launch planner (no GPU: an explicit device of
152 SMs and 227 KB of shared memory per block, the GB300 figures)."""
import pytest

from quantised_gguf_weight_gb300 import qk

SMS, SMEM = 152, 232448
UNIT = {"q8_0": 32, "q4_k": 256, "q6_k": 128}       # columns of a lane unit
ROWS = [1, 7, 100, 1000, 4096, 28672, 151936]
KS = [32, 33, 256, 300, 896, 1024, 4096, 5120, 14336, 20000]


def plan(fmt, rows, K, batch, **kw):
    return qk.debug_gemv_plan_for(fmt, rows, K, batch, SMS, SMEM, **kw)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q6_k"])
@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_row_decomposition_depends_on_K_only(fmt, batch):
    """SW, cpl and nkc fix the order of a row's additions: equal for every row count."""
    for K in KS:
        shapes = {(p["SW"], p["cpl"], p["nkc"], p["R"]) for rows in ROWS if (p := plan(fmt, rows, K, batch))}
        assert len(shapes) <= 1, (fmt, K, batch, shapes)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q6_k"])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_plan_covers_the_row_and_fits(fmt, batch):
    for K in KS:
        for rows in ROWS:
            p = plan(fmt, rows, K, batch)
            if p is None:
                continue
            lu = -(-K // UNIT[fmt])
            assert p["LU"] == lu
            assert p["SW"] * p["cpl"] * p["nkc"] >= lu                  # every lane unit has a lane
            assert p["SW"] * p["cpl"] * (p["nkc"] - 1) < lu             # no empty trailing chunk
            assert 32 % p["SW"] == 0 and p["rows_w"] == (32 // p["SW"]) * p["R"]
            assert 1 <= p["nw"] <= ((15 if p["wide"] else 11) if batch == 1 else 8) and p["m"] >= 1
            assert not p["wide"] or batch == 1
            assert p["wide"] or fmt != "q6_k" or batch != 1
            assert p["stages"] == p["nw"] * p["m"] <= 32
            assert p["off_stage"] + p["stages"] * p["stage_bytes"] == p["smem"] <= SMEM
            assert p["grid"] == min(SMS, rows)
            assert p["stage_bytes"] % 128 == 0


def test_activations_that_do_not_fit_have_no_plan():
    # Llama-8B ffn_down: batch 3 fits, batch 4 does not (the host splits it)
    assert plan("q4_k", 4096, 14336, 3) is not None
    assert plan("q4_k", 4096, 14336, 4) is None
    # one row of K = 57344 does not fit at all
    assert plan("q4_k", 16, 57344, 1) is None
    assert plan("q8_0", 16, 49152, 1) is None
    assert plan("q8_0", 16, 40960, 1) is not None


def test_pair_and_expert_modes():
    p = plan("q4_k", 14336, 4096, 1, pair=True)
    assert p is not None and p["R"] % 2 == 0
    q = plan("q4_k", 1536, 2048, 1, n_assign=8)
    assert q["cpa"] == SMS // 8 and q["grid"] == 8 * q["cpa"]
    r = plan("q4_k", 1536, 2048, 1, n_assign=400)
    assert r["cpa"] == 1 and r["grid"] == 400


def test_wide_form_for_calls_with_many_items():
    """Q4_K batch 1: more items a CTA than 11 warps -> the 16-warp form."""
    assert plan("q4_k", 6144, 4096, 1)["wide"] == 0          # 11 items a CTA (qkv)
    assert plan("q4_k", 4096, 4096, 1)["wide"] == 0          # 7 (attn_output)
    assert plan("q4_k", 28672, 4096, 1)["wide"] == 1         # 48 (gate+up)
    assert plan("q4_k", 4096, 14336, 1)["wide"] == 1         # 28 (ffn_down, 2 chunks a row)
    assert plan("q4_k", 28672, 4096, 2)["wide"] == 0


def test_split_k_over_warps_for_few_row_groups():
    """A CTA with fewer row groups than warps shares each group's K chunks
    among kw warps (their sums are added in chunk order, so the row's cut and
    its bits stay those of the unsplit plan)."""
    p = plan("q4_k", 896, 4864, 1)                 # Qwen ffn_down: 6 rows a CTA, 3 chunks a row
    assert p["nkc"] == 3 and p["kw"] == 3 and p["nw"] == 3
    p = plan("q4_k", 1, 14336, 1)                  # one row, two chunks
    assert p["nkc"] == 2 and p["kw"] == 2 and p["nw"] == 2 and p["grid"] == 1
    p = plan("q8_0", 33, 20000, 1)
    assert p["kw"] > 1 and p["nw"] == p["kw"]
    assert plan("q4_k", 28672, 4096, 1)["kw"] == 1    # whole rows: nothing to split
    assert plan("q4_k", 4096, 14336, 1)["kw"] == 1    # 28 row groups a CTA fill the warps
    for fmt in ("q8_0", "q4_k", "q6_k"):
        for K in KS:
            for rows in ROWS:
                for batch in (1, 2, 8):
                    q = plan(fmt, rows, K, batch)
                    if q is None:
                        continue
                    assert 1 <= q["kw"] <= max(1, q["nkc"])
                    assert q["kw"] == 1 or (q["nkc"] > 1 and q["nw"] % q["kw"] == 0)


# ---------------------------------------------------------------- tensor-core form (batch 2..8)

def tc_plan(fmt, rows, K):
    return qk.debug_gemv_tc_plan_for(fmt, rows, K, SMS, SMEM)


def test_tensor_core_form_depends_on_format_and_K_only():
    """Q8_0 takes it for K a multiple of 128 that fits, Q4_K for any K that
    fits, Q6_K never; the plan is the same for every row count but the grid
    (K split over CTA pairs: one pair a row at most, 76 pairs on 152 SMs)."""
    for fmt in ("q8_0", "q4_k", "q6_k"):
        for K in KS + [128, 640, 2048, 4864]:
            plans = [tc_plan(fmt, rows, K) for rows in ROWS]
            taken = {p is not None for p in plans}
            assert len(taken) == 1, (fmt, K)
            if fmt == "q6_k" or (fmt == "q8_0" and K % 128):
                assert not taken.pop(), (fmt, K)
            if plans[0] is not None:
                same = {tuple(v for k, v in p.items() if k != "grid") for p in plans}
                assert len(same) == 1, (fmt, K)
                assert [p["grid"] for p in plans] == [2 * min(r, SMS // 2) if p["ks"] else min(r, SMS)
                                                      for r, p in zip(ROWS, plans)]
    # the configurations that use it
    assert tc_plan("q8_0", 151936, 896) is not None        # Q8_0 lm_head
    assert tc_plan("q4_k", 28672, 4096) is not None        # Llama-8B gate+up
    assert tc_plan("q4_k", 4096, 14336) is None            # its activations do not fit
    assert tc_plan("q8_0", 4096, 14336) is None
    # K split over CTA pairs from 8 items a tile when their number is even
    # (each CTA then holds half of x): the activations and two stages fit
    assert tc_plan("q8_0", 1000, 896)["ks"] == 0
    assert tc_plan("q8_0", 1000, 4096)["ks"] == 1
    assert tc_plan("q8_0", 1000, 4224) is None              # 17 items: not split, does not fit
    assert tc_plan("q8_0", 1000, 7168)["ks"] == 1           # split: up to 7168
    assert tc_plan("q8_0", 1000, 7680) is None
    assert tc_plan("q4_k", 1000, 4864)["ks"] == 0           # Q4_K, 19 items: not split, up to 4864
    assert tc_plan("q4_k", 1000, 8704)["ks"] == 1           # split: up to 8704
    assert tc_plan("q4_k", 1000, 8960) is None


@pytest.mark.parametrize("fmt,K", [("q8_0", 128), ("q8_0", 896), ("q8_0", 4096), ("q4_k", 256), ("q4_k", 300),
                                   ("q4_k", 4096), ("q4_k", 4864)])
def test_tensor_core_plan_layout(fmt, K):
    """Groups and items cover the padded K, the B operand (32 bytes a column
    of the CTA's part of K, 1024-byte aligned) and the tables precede at
    least two stages, and all of it fits in the block's shared memory."""
    p = tc_plan(fmt, 1000, K)
    Kp = -(-K // 256) * 256 if fmt == "q4_k" else K
    assert p["G"] * 32 == Kp
    assert p["NC"] == -(-Kp // 256)
    assert p["ks"] == (1 if p["NC"] % 2 == 0 and p["NC"] >= 8 else 0)
    assert p["off_bop"] % 1024 == 0
    assert p["off_bop"] + 32 * (Kp // 2 if p["ks"] else Kp) <= p["off_stage"]
    assert p["off_stage"] % 128 == 0
    assert p["row_stride"] % 16 == 0 and (p["row_stride"] // 16) % 2 == 1    # conflict-free row reads
    # Q4_K: one box of 128 rows x 144 bytes; Q8_0: four of 64 rows x 144 bytes
    assert p["stage_bytes"] == 128 * 144 if fmt == "q4_k" else 4 * 64 * 144
    assert 2 <= p["NS"] <= 8
    assert p["smem"] == p["off_stage"] + p["NS"] * p["stage_bytes"] + 1024 <= SMEM
