"""Pin the packed-row (varlen) oracle to torch's scaled_dot_product_attention in float64 on K/V
gathered through the block table (E4M3 pages decoded by torch's float8 type times their scale):
each sequence's q_len_b rows with the causal limit L - q_len_b + i + 1 (chunked prefill, decode
and verify rows in one batch)."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_attn_gb300 import workloads as W


def _page(cache, scale, pb):
    """One page [Hkv, bs, d] as float64: bf16 values, or E4M3 codes (torch's float8 decode) times
    the page's per-kv-head scale."""
    if scale is None:
        return cache[pb].double()
    return cache[pb].view(torch.float8_e4m3fn).double() * scale[pb].double()[:, None, None]


def _sdpa_reference(p):
    out = torch.zeros(p.q.shape, dtype=torch.float64)
    qsl = p.query_start_loc.tolist()
    G = p.num_q_heads // p.num_kv_heads
    for b in range(p.num_seqs):
        L = int(p.context_lens[b])
        ql = qsl[b + 1] - qsl[b]
        if ql == 0:
            continue
        pages = [int(x) for x in p.block_table[b, : (L + 15) // 16]]
        k = torch.cat([_page(p.k_cache, p.k_scale, pb) for pb in pages], dim=1)[:, :L]  # [Hkv, L, d]
        v = torch.cat([_page(p.v_cache, p.v_scale, pb) for pb in pages], dim=1)[:, :L]
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        q = p.q[qsl[b]:qsl[b + 1]].double().transpose(0, 1)  # [Hq, ql, d]
        i = torch.arange(ql)[:, None]
        j = torch.arange(L)[None, :]
        mask = j < (L - ql + i + 1)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=p.scale)
        out[qsl[b]:qsl[b + 1]] = o.transpose(0, 1)
    return out.numpy()


@pytest.mark.parametrize("prior,qls,hq,hkv,d", [
    ([0, 100, 5, 300, 16], [37, 64, 1, 9, 128], 8, 2, 64),
    ([0, 0, 47], [1, 20, 33], 4, 4, 32),
    ([250, 3], [0, 70], 16, 2, 64),
])
def test_varlen_oracle_matches_sdpa(prior, qls, hq, hkv, d):
    p = W.make_varlen_problem(prior, qls, hq, hkv, d, seed=sum(qls))
    got = oracle.attention_varlen_problem(p)
    ref = _sdpa_reference(p)
    assert np.abs(got - ref).max() <= 1e-12


@pytest.mark.parametrize("prior,qls,hq,hkv,d", [
    ([0, 100, 5, 300], [37, 64, 1, 9], 8, 2, 64),
    ([250, 3], [0, 70], 16, 2, 128),
])
def test_varlen_oracle_matches_sdpa_fp8(prior, qls, hq, hkv, d):
    # E4M3 caches: the same rows over K/V decoded from the stored codes and scales
    p = W.make_varlen_problem(prior, qls, hq, hkv, d, seed=7 + sum(qls), kv_dtype=W.KV_FP8_E4M3)
    got = oracle.attention_varlen_problem(p)
    ref = _sdpa_reference(p)
    assert np.abs(got - ref).max() <= 1e-12


def test_varlen_oracle_row_selection():
    p = W.make_varlen_problem([10, 200], [40, 30], 8, 2, 64, seed=9)
    full = oracle.attention_varlen_problem(p)
    rows = [0, 39, 40, 55, 69]
    part = oracle.attention_varlen_problem(p, rows=rows)
    assert np.array_equal(part[rows], full[rows])
    others = np.setdiff1d(np.arange(70), rows)
    assert np.all(part[others] == 0)
