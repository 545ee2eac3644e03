"""Failure detection on the GPU without a fault: a bounded kernel wait that runs out, and a
context longer than the host-side bound.  Each reaches the host as a status from
check_device_errors() while the context stays usable (the next call computes correct results)."""

import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
import paged_kv_gqa_attn_gb300 as pa
from paged_kv_gqa_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _parity(p, out):
    ref = oracle.attention_problem(p)
    got = out.float().cpu().double().numpy()
    label = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    parity.check(got, ref, p.kv_dtype == W.KV_FP8_E4M3, label=label)


@pytest.mark.parametrize("helper", [0, 1, 2])
def test_wait_timeout_is_reported_and_context_stays_usable(helper):
    pa.check_device_errors()
    elapsed = pa.selftest_wait(helper, 4096)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_TIMEOUT
    assert int(elapsed.item()) > 0
    assert pa.check_device_errors() == pa.PA_OK  # reading the word clears it
    # the same context still runs a decode and a verify call correctly
    for q_len in (1, 5):
        p = W.make_problem([300, 77], 8, 2, 128, q_len=q_len, seed=950 + q_len, device="cuda")
        out = pa.run_problem(p)
        assert pa.check_device_errors() == pa.PA_OK
        _parity(p, out)


@pytest.mark.parametrize("helper,short_polls,limit,probes_per_iteration", [
    (0, 1 << 8, pa.PA_WAIT_LIMIT, 1),    # suspending polls: microseconds each
    (2, 1 << 14, pa.PA_SPIN_LIMIT, 3),   # probe loops: an issuer iteration probes up to 3 barriers
])
def test_full_wait_limit_ends_within_seconds(helper, short_polls, limit, probes_per_iteration):
    pa.check_device_errors()
    short = int(pa.selftest_wait(helper, short_polls).item())
    long = int(pa.selftest_wait(helper, short_polls * 16).item())
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_TIMEOUT
    assert long > short > 0
    per_poll = long / (short_polls * 16)
    full_s = per_poll * probes_per_iteration * limit / 1e9
    print(f"helper {helper}: {per_poll:.1f} ns per poll; full limit ~ {full_s:.2f} s")
    # a wait that can never complete gives up after about a second, not minutes
    assert full_s < 5.0


@pytest.mark.parametrize("q_len", [1, 5])
def test_context_above_the_bound_is_clamped_and_flagged(q_len):
    # context_lens says 300 tokens but the caller's bound is 160: the kernels attend to the first
    # 160 (the grid and scratch were sized for that) and flag the call
    p = W.make_problem([300, 120], 8, 2, 128, q_len=q_len, seed=960 + q_len, device="cuda")
    pa.check_device_errors()
    out = pa.run_problem(p, max_context_len=160)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    clamped = dataclasses.replace(p, context_lens=torch.clamp(p.context_lens, max=160))
    _parity(clamped, out)
