"""GPU parity for paged prefill over packed variable-length rows (paged_attn_prefill) against the
fp64 oracle: chunked-prefill chunks, piggybacked decode and verify rows, every GQA group size,
head_dim 64 and 128, ragged tiles and tails; at the full chunked-prefill shape on sampled rows
(tile boundaries, first and last rows of every chunk)."""

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


def _run(p, **kw):
    g = p.to("cuda")
    out = pa.prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens, g.query_start_loc,
                     g.scale, k_scale=g.k_scale, v_scale=g.v_scale, **kw)
    torch.cuda.synchronize()
    return out


def _check(p, rows=None, expect=pa.PA_OK, **kw):
    out = _run(p, **kw)
    assert pa.check_device_errors() == expect
    ref = oracle.attention_varlen_problem(p, rows=rows)
    got = out.float().cpu().double().numpy()
    if rows is not None:
        got, ref = got[rows], ref[rows]
    parity.check(got, ref, p.kv_dtype == W.KV_FP8_E4M3, label=_label())
    return out


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (8, 2, 64), (4, 4, 128), (16, 8, 64), (16, 2, 128)])
def test_prefill_mixed_batch(hq, hkv, d):
    # chunks with and without prior context, a decode row, a verify-sized run, ragged tiles
    p = W.make_varlen_problem([0, 100, 5, 300, 16, 1000, 77], [37, 64, 1, 9, 128, 200, 3], hq, hkv, d,
                              seed=hq * 7 + d, tail_fill="nan")
    _check(p)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (8, 2, 64), (4, 4, 128), (16, 8, 64), (16, 2, 128)])
def test_prefill_mixed_batch_fp8(hq, hkv, d):
    # E4M3 caches: pages converted to f16 in shared memory, per-(block, kv head) scales
    p = W.make_varlen_problem([0, 100, 5, 300, 16, 1000, 77], [37, 64, 1, 9, 128, 200, 3], hq, hkv, d,
                              seed=hq * 7 + d + 1, tail_fill="nan", kv_dtype=W.KV_FP8_E4M3)
    _check(p)


def test_prefill_full_chunk_workload_sampled_fp8():
    p = W.chunked_prefill_workload(decodes=16, kv_dtype=W.KV_FP8_E4M3)
    _check(p, rows=_sample_rows(p, seed=1))


def test_prefill_long_prior_and_empty_sequences():
    p = W.make_varlen_problem([3000, 0, 50, 0], [0, 0, 300, 1], 8, 2, 128, seed=21, tail_fill="nan")
    _check(p)


def test_prefill_context_shorter_than_rows_is_flagged():
    p = W.make_varlen_problem([40], [20], 8, 2, 128, seed=22)
    p.context_lens = torch.tensor([10], dtype=torch.int32)  # rows 0..9 see nothing
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    o = out.float().cpu().numpy()
    assert np.all(o[:10] == 0)
    ref = oracle.attention_varlen_problem(p, rows=list(range(10, 20)))[10:20]
    parity.check(o[10:20], ref, False, label=_label())


def test_prefill_bad_query_start_loc_is_flagged():
    p = W.make_varlen_problem([10, 10], [5, 5], 8, 2, 64, seed=23)
    p.query_start_loc = torch.tensor([0, 5, 99], dtype=torch.int32)  # past total_q
    g = p.to("cuda")
    out = torch.zeros_like(g.q)
    pa.prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens, g.query_start_loc, g.scale,
               max_q_len=5, out=out)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    assert torch.all(out[5:] == 0)


def test_prefill_rows_match_decode_and_verify_kernels():
    # one-row sequences = the decode kernel; K+1-row sequences = the verify kernel (same inputs)
    dec = W.make_config("llama8b_decode", device="cuda")
    qsl = torch.arange(dec.num_seqs + 1, dtype=torch.int32, device="cuda")
    a = pa.prefill(dec.q[:, 0].contiguous(), dec.k_cache, dec.v_cache, dec.block_table, dec.context_lens,
                   qsl, dec.scale, max_q_len=1)
    b = pa.run_problem(dec)
    assert (a.float() - b[:, 0].float()).abs().max().item() <= 2e-2
    ver = W.make_config("spec_verify_k8", device="cuda")
    qsl = torch.arange(0, ver.num_seqs * 9 + 1, 9, dtype=torch.int32, device="cuda")
    a = pa.prefill(ver.q.reshape(-1, 32, 128), ver.k_cache, ver.v_cache, ver.block_table, ver.context_lens,
                   qsl, ver.scale, max_q_len=9)
    b = pa.run_problem(ver)
    assert (a.float() - b.reshape(-1, 32, 128).float()).abs().max().item() <= 2e-2
    assert pa.check_device_errors() == pa.PA_OK


def _sample_rows(p, per_seq=24, seed=0):
    rng = np.random.default_rng(seed)
    qsl = p.query_start_loc.cpu().tolist()
    rows = []
    for b in range(p.num_seqs):
        n = qsl[b + 1] - qsl[b]
        if n == 0:
            continue
        pick = {0, n - 1, min(31, n - 1), min(32, n - 1)}
        pick |= set(rng.integers(0, n, size=min(per_seq, n)).tolist())
        rows += [qsl[b] + i for i in sorted(pick)]
    return rows


def test_prefill_full_chunk_workload_sampled():
    p = W.chunked_prefill_workload(decodes=16)
    _check(p, rows=_sample_rows(p))


def test_prefill_deterministic():
    p = W.make_varlen_problem([500, 30], [300, 100], 32, 8, 128, seed=24).to("cuda")
    a = pa.prefill(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, p.query_start_loc, p.scale)
    b = pa.prefill(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, p.query_start_loc, p.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
