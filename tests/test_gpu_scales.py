"""E4M3 caches whose per-(block, kv head) scales are not what the append step would produce --
negative, zero, subnormal and four times larger -- through every attention route (decode on the
warp-level kernel and on the tcgen05 kernel, verify, verify beyond 64 rows per kv head, chunked
prefill), against the oracle, which decodes each stored code times its page's scale as the
definition says (study book ch.10, section 10.8.2: one scale per (block, kv head)).  Steps whose
scales are all positive and normal take the kernels' raw-score paths; these cases drive the
others, and the steps that mix both."""

import os

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
import paged_kv_gqa_attn_gb300 as pa
from paged_kv_gqa_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _label():
    return os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]


def _odd_scales(k_scale, v_scale, seed):
    """In place: an eighth of each scale table negated, an eighth zero, an eighth subnormal
    (1e-40), an eighth multiplied by 4; the rest as stored."""
    g = torch.Generator().manual_seed(seed)
    for t in (k_scale, v_scale):
        f = t.view(-1)
        n = f.numel()
        sel = torch.randperm(n, generator=g)
        q = max(1, n // 8)
        f[sel[:q]] *= -1.0
        f[sel[q:2 * q]] = 0.0
        f[sel[2 * q:3 * q]] = 1e-40
        f[sel[3 * q:4 * q]] *= 4.0


@pytest.mark.parametrize("lens,hq,hkv,d,q_len", [
    ([100, 1500, 37, 3000], 32, 8, 128, 1),    # decode, groups of 4 (warp-level kernel)
    ([100, 1500, 37, 3000], 16, 8, 64, 1),     # decode, groups of 2, d 64
    ([700, 2100, 19], 6, 2, 128, 1),           # decode, groups of 3 (tcgen05 kernel)
    ([509, 2009, 1300], 32, 8, 128, 9),        # verify, 36 rows per kv head
    ([509, 2009], 16, 4, 64, 5),               # verify, d 64
    ([509, 2009, 1300], 64, 8, 128, 9),        # verify, 72 rows per kv head (split prefill kernel)
])
def test_attention_odd_scales(lens, hq, hkv, d, q_len):
    p = W.make_problem(lens, hq, hkv, d, q_len=q_len, kv_dtype=W.KV_FP8_E4M3, seed=sum(lens) + d)
    _odd_scales(p.k_scale, p.v_scale, seed=len(lens) + q_len)
    out = pa.run_problem(p.to("cuda"))
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    ref = oracle.attention_problem(p)
    parity.check(out.float().cpu().double().numpy(), ref, True, label=_label())


@pytest.mark.parametrize("d", [128, 64])
def test_prefill_odd_scales(d):
    p = W.make_varlen_problem([0, 300, 1200, 64], [200, 150, 77, 129], 8, 2, d, seed=11 + d,
                              kv_dtype=W.KV_FP8_E4M3)
    _odd_scales(p.k_scale, p.v_scale, seed=d)
    g = p.to("cuda")
    out = pa.prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens, g.query_start_loc, g.scale,
                     k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    ref = oracle.attention_varlen_problem(p)
    parity.check(out.float().cpu().double().numpy(), ref, True, label=_label())


@pytest.mark.parametrize("tiny", [2e-38, 1e-30])
def test_prefill_tiny_normal_v_scales(tiny):
    """Half the V scales tiny but normal (a page's weights times its scale then fall below the
    smallest normal float): the row sum still counts every token's weight, as the oracle does."""
    p = W.make_varlen_problem([0, 1300, 2100], [200, 160, 130], 8, 2, 128, seed=23,
                              kv_dtype=W.KV_FP8_E4M3)
    g = torch.Generator().manual_seed(5)
    f = p.v_scale.view(-1)
    f[torch.randperm(f.numel(), generator=g)[: f.numel() // 2]] = tiny
    d = p.to("cuda")
    out = pa.prefill(d.q, d.k_cache, d.v_cache, d.block_table, d.context_lens, d.query_start_loc, d.scale,
                     k_scale=d.k_scale, v_scale=d.v_scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    ref = oracle.attention_varlen_problem(p)
    parity.check(out.float().cpu().double().numpy(), ref, True, label=_label())
