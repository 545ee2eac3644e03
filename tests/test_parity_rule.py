"""The parity rule the GPU tests apply (oracle/parity.py), pinned on the CPU: the half-ulp it
allows where a bf16 output cannot meet the flat bar is the actual bf16 rounding error (torch's
round-to-nearest-even conversion), the bar is flat below |ref| = 4, planted errors on either side
of the bound pass or fail as they must, and every check is logged.  Also the rule by which the
bench times a workload cold (copies of its inputs rotated so that each call reads HBM)."""

import json
import math

import numpy as np
import pytest
import torch

from oracle import parity
import bench


def test_half_ulp_matches_bf16_rounding():
    g = torch.Generator().manual_seed(3)
    # fp32 values (the kernels round fp32 results to bf16 once; torch takes a float64 through
    # float32 first, which could round twice)
    x = ((torch.rand(200000, generator=g, dtype=torch.float64) * 2 - 1) * torch.exp2(
        torch.randint(-20, 20, (200000,), generator=g).double())).float().double()
    err = (x.float().to(torch.bfloat16).double() - x).abs().numpy()
    hu = parity.half_ulp_bf16(x.numpy())
    assert np.all(err <= hu * (1 + 1e-12))
    # the bound is reached: rounding errors come within 1 % of half an ulp
    assert np.any(err >= 0.99 * hu)


@pytest.mark.parametrize("x,expect", [(1.5, 2.0 ** -8), (3.0, 2.0 ** -7), (-5.0, 2.0 ** -6), (0.3, 2.0 ** -10)])
def test_half_ulp_values(x, expect):
    assert parity.half_ulp_bf16(x) == expect


def test_bound_is_flat_where_bf16_can_meet_it():
    ref = np.array([0.0, 0.5, -1.9, 3.99, 4.0, -6.0, 20.0])
    b = parity.element_bound(ref, fp8=False)
    assert np.all(b[:4] == parity.BF16_MAX)
    hu = parity.half_ulp_bf16(ref[4:])
    assert np.allclose(b[4:], hu + parity.RELAXED_EXTRA)
    bf = parity.element_bound(np.array([1.0, 15.9, 16.0]), fp8=True)
    assert bf[0] == parity.FP8_MAX and bf[1] == parity.FP8_MAX and bf[2] > parity.FP8_MAX


def test_check_accepts_and_rejects_planted_errors(monkeypatch, tmp_path):
    log = tmp_path / "parity.jsonl"
    monkeypatch.setenv("PA_PARITY_LOG", str(log))
    ref = np.linspace(-3.0, 3.0, 1000)
    ok = ref.copy()
    ok[::100] += 0.0099
    mx, mean, relaxed = parity.check(ok, ref, fp8=False, label="inside")
    assert relaxed == 0 and mx == pytest.approx(0.0099)
    bad = ref.copy()
    bad[500] += 0.0101  # one element past the flat bar at |ref| < 4
    with pytest.raises(AssertionError):
        parity.check(bad, ref, fp8=False, label="outside")
    big = np.array([5.0, -6.0, 7.5])
    # half an ulp at [4, 8) is 2^-6: 0.0165 is allowed there (bound 0.0176), 0.018 is not
    parity.check(big + 0.0165, big, fp8=False, label="relaxed", mean_bar=False)
    with pytest.raises(AssertionError):
        parity.check(big + 0.018, big, fp8=False, label="relaxed-bad", mean_bar=False)
    with pytest.raises(AssertionError):  # the bf16 mean bar
        parity.check(ref + 0.002, ref, fp8=False, label="mean")
    parity.check(ref + 0.04, ref, fp8=True, label="fp8")  # E4M3: 5e-2, no mean bar
    recs = [json.loads(l) for l in log.read_text().splitlines()]
    assert [r["label"] for r in recs] == ["inside", "outside", "relaxed", "relaxed-bad", "mean", "fp8"]
    assert recs[0]["worst_margin"] == pytest.approx(parity.BF16_MAX - 0.0099)
    assert recs[1]["worst_margin"] < 0 and recs[2]["relaxed_elements"] == 3


@pytest.mark.parametrize("mb,copies", [(0.063, 8), (176, 4), (175, 4), (300, 4), (405, 4), (406, 1), (538, 1), (3000, 1)])
def test_cold_rotation(mb, copies):
    alg = int(mb * 1e6)
    n = bench.pool_rotation(alg)
    assert n == copies
    if n > 1 and alg > 1e6:
        # the other copies' reads between two turns of one copy exceed 2x the L2
        assert (n - 1) * alg > 2 * bench.L2_BYTES
    assert math.isfinite(n)
