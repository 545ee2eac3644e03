"""GPU parity at the size limits: batches past the 1024-sequence scan width of the verify planner,
thousands of sequences for decode, append and acceptance, a prefill batch of hundreds of packed
sequences, and the largest vocabulary the acceptance kernel takes (2^21)."""

import os

import numpy as np
import pytest
import torch

import oracle
from oracle import append as OA
from oracle import parity
from oracle import spec_accept as SA
import paged_kv_gqa_attn_gb300 as pa
from paged_kv_gqa_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _close(out, ref, seqs=None):
    g = out.float().cpu().double().numpy()
    if seqs is not None:
        g, ref = g[seqs], ref[seqs]
    label = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    parity.check(g, ref, False, label=label)


def _lens(n, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def test_verify_batch_past_planner_scan_width():
    lens = _lens(1500, 9, 200, 1)
    p = W.make_problem(lens, 8, 2, 64, q_len=9, seed=301, device="cuda")
    out = pa.run_problem(p)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    seqs = [0, 1, 511, 1023, 1024, 1025, 1300, 1499]
    _close(out, oracle.attention_problem(p, seqs=seqs), seqs)


def test_decode_batch_of_1500():
    lens = _lens(1500, 1, 300, 2)
    p = W.make_problem(lens, 8, 2, 128, seed=302, device="cuda")
    out = pa.run_problem(p)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    seqs = [0, 7, 1023, 1024, 1499]
    _close(out, oracle.attention_problem(p, seqs=seqs), seqs)


def test_prefill_300_packed_sequences():
    g = torch.Generator().manual_seed(3)
    prior = torch.randint(0, 400, (300,), generator=g).tolist()
    qls = torch.randint(0, 70, (300,), generator=g).tolist()
    p = W.make_varlen_problem(prior, qls, 8, 2, 64, seed=303)
    gp = p.to("cuda")
    out = pa.prefill(gp.q, gp.k_cache, gp.v_cache, gp.block_table, gp.context_lens, gp.query_start_loc,
                     gp.scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    rows = list(range(0, int(p.q.shape[0]), 97)) + [int(p.q.shape[0]) - 1]
    _close(out, oracle.attention_varlen_problem(p, rows=rows), rows)


def test_append_5000_sequences():
    lens = _lens(5000, 1, 40, 4)
    p = W.make_problem(lens, 2, 1, 64, seed=304)
    g = torch.Generator().manual_seed(4)
    kn = torch.randn(5000, 1, 1, 64, generator=g).to(torch.bfloat16)
    vn = torch.randn(5000, 1, 1, 64, generator=g).to(torch.bfloat16)
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.append_kv(kn.cuda(), vn.cuda(), kc, vc, p.block_table.cuda(), p.context_lens.cuda())
    assert pa.check_device_errors() == pa.PA_OK
    rk, rv = OA.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens, n_new=1, block_size=16)
    assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), rk)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy().view(np.uint16), rv)


def _accept_check(a):
    ga = a.to("cuda")
    n, t = pa.spec_accept(ga.p, ga.q, ga.draft, ga.u_accept, ga.u_sample)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    rn, rt = SA.accept_batch(a.p.numpy(), a.q.numpy(), a.draft.numpy(), a.u_accept.numpy(),
                             a.u_sample.numpy().view(np.uint32))
    assert np.array_equal(n.cpu().numpy(), rn) and np.array_equal(t.cpu().numpy(), rt)


def test_accept_largest_vocabulary():
    _accept_check(W.make_accept_problem(2, 2, 1 << 21, seed=305))


def test_accept_3000_rounds_31_drafts():
    _accept_check(W.make_accept_problem(3000, 31, 64, seed=306))
