"""The entry points inside CUDA graphs: after one eager call (which sets up the per-device state,
the kernels' shared-memory limits and the scratch pool), decode, verify, tree verify, prefill,
append and acceptance are captured into one graph and replayed; the replay reproduces the eager
results bit for bit, including on new inputs copied into the captured buffers."""

import numpy as np
import pytest
import torch

import paged_kv_gqa_attn_gb300 as pa
from paged_kv_gqa_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def test_everything_in_one_graph():
    dec = W.make_problem([40, 700, 2100], 32, 8, 128, seed=401, device="cuda")
    ver = W.make_problem([40, 700, 2100], 32, 8, 128, q_len=9, seed=402, device="cuda")
    masks = W.random_tree_masks(3, 9, seed=3).to("cuda")
    pf = W.make_varlen_problem([0, 300, 50], [100, 1, 9], 32, 8, 128, seed=403).to("cuda")
    ap = W.make_problem([20, 33], 8, 2, 128, seed=404, device="cuda")
    g = torch.Generator().manual_seed(404)
    kn = torch.randn(2, 3, 2, 128, generator=g).to(torch.bfloat16).cuda()
    vn = torch.randn(2, 3, 2, 128, generator=g).to(torch.bfloat16).cuda()
    acc = W.make_accept_problem(4, 4, 5000, seed=405).to("cuda")
    mx_dec, mx_ver = int(dec.context_lens.max()), int(ver.context_lens.max())
    outs = {
        "dec": torch.empty_like(dec.q), "ver": torch.empty_like(ver.q), "tree": torch.empty_like(ver.q),
        "pf": torch.empty_like(pf.q), "n": torch.empty(4, dtype=torch.int32, device="cuda"),
        "tok": torch.empty(4, 5, dtype=torch.int32, device="cuda"),
    }
    kc0, vc0 = ap.k_cache.clone(), ap.v_cache.clone()

    def work(stream):
        pa.decode(dec.q, dec.k_cache, dec.v_cache, dec.block_table, dec.context_lens, dec.scale,
                  out=outs["dec"], max_context_len=mx_dec, stream=stream)
        pa.verify(ver.q, ver.k_cache, ver.v_cache, ver.block_table, ver.context_lens, ver.scale,
                  out=outs["ver"], max_context_len=mx_ver, stream=stream)
        pa.tree_verify(ver.q, ver.k_cache, ver.v_cache, ver.block_table, ver.context_lens, masks, ver.scale,
                       out=outs["tree"], max_context_len=mx_ver, stream=stream)
        pa.prefill(pf.q, pf.k_cache, pf.v_cache, pf.block_table, pf.context_lens, pf.query_start_loc,
                   pf.scale, max_q_len=100, out=outs["pf"], stream=stream)
        ap.k_cache.copy_(kc0)
        ap.v_cache.copy_(vc0)
        pa.append_kv(kn, vn, ap.k_cache, ap.v_cache, ap.block_table, ap.context_lens, stream=stream)
        pa.spec_accept(acc.p, acc.q, acc.draft, acc.u_accept, acc.u_sample, out_tokens=outs["tok"],
                       num_accepted=outs["n"], stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        work(s)  # eager: sets up state, smem limits, the pool
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in outs.items()}
    eager["kc"], eager["vc"] = ap.k_cache.clone(), ap.v_cache.clone()
    for v in outs.values():
        v.zero_()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        work(s)
    graph.replay()
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    for k in outs:
        assert torch.equal(_bits(outs[k]), _bits(eager[k])), k
    assert torch.equal(_bits(ap.k_cache), _bits(eager["kc"])) and torch.equal(_bits(ap.v_cache), _bits(eager["vc"]))

    # new inputs in the captured buffers: the replay follows them
    dec.q.copy_(torch.randn_like(dec.q.float()).to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    ref = pa.decode(dec.q, dec.k_cache, dec.v_cache, dec.block_table, dec.context_lens, dec.scale,
                    max_context_len=mx_dec)
    torch.cuda.synchronize()
    assert torch.equal(_bits(outs["dec"]), _bits(ref))
    assert not torch.equal(_bits(outs["dec"]), _bits(eager["dec"]))
