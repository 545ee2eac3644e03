"""The per-step summary of the verify timeline tool, on a synthetic stamp array whose intervals
are known: every CTA's steps advance by a fixed period and each role's stamp sits at a fixed
offset within the step, so every median the tool prints is one of those offsets."""

import numpy as np

from paged_kv_gqa_attn_gb300 import timeline as tl


def _stamps(fp8, period=2000, steps=20, ctas=3):
    a = np.zeros((ctas, tl.ST_STEPS, tl.ST_SLOTS))
    off = {tl.ST_KCOPY: -3000, tl.ST_VCOPY: -2500, tl.ST_VLANDED: -900, tl.ST_CONVV: -400,
           tl.ST_CONVK: -450, tl.ST_QK: -300, tl.ST_S: 0, tl.ST_P0: 1500, tl.ST_P1: 1600, tl.ST_PV: 1900}
    for c in range(ctas):
        base = 100000 + 7777 * c
        for k in range(steps):
            for slot, o in off.items():
                if not fp8 and slot in (tl.ST_VLANDED, tl.ST_CONVV, tl.ST_CONVK):
                    continue
                a[c, k, slot] = base + k * period + o
    return a


def test_step_summary_bf16():
    s, n = tl.step_summary(_stamps(False), fp8=False)
    assert n == 3 * (20 - 3)
    assert s["period_pv"] == 2000
    assert s["softmax_busy"] == 1600          # S seen -> the later warp's P
    assert s["softmax_wait_s"] == 400         # previous P (1600) -> this S (2000)
    assert s["p_skew"] == 100
    assert s["qk_to_s"] == 300
    assert s["pv2_to_qk"] == 2 * 2000 - 1900 - 300
    assert s["kcopy_to_qk"] == 2700
    assert s["vcopy_to_pv"] == 4400
    assert s["handoff_to_pv"] == 300          # PV (1900) after the later P (1600)
    assert "vcopy_to_landed" not in s


def test_step_summary_e4m3():
    s, _ = tl.step_summary(_stamps(True), fp8=True)
    assert s["vcopy_to_landed"] == 1600
    assert s["landed_to_converted"] == 500
    assert s["handoff_to_pv"] == 300          # the later of P (1600) and V converted (-400)
