"""GPU parity for the KV append (paged_attn_append_kv) against the append oracle: bit-exact caches
and scales, for bf16 and fp8 pools, appends that stay in one block, cross a block boundary or fill
whole blocks; then attention over the appended cache against the attention oracle."""

import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import append as OA
from oracle import parity
import paged_kv_gqa_attn_gb300 as pa
from paged_kv_gqa_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _label():
    return os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]


def _new_rows(B, n_new, Hkv, d, seed, mag=1.0):
    g = torch.Generator().manual_seed(seed)
    k = (torch.randn(B, n_new, Hkv, d, generator=g) * mag).to(torch.bfloat16)
    v = (torch.randn(B, n_new, Hkv, d, generator=g) * mag).to(torch.bfloat16)
    return k, v


def _gpu(p):
    return p.to("cuda")


def _append_both(p, kn, vn, n_new):
    """Run the kernel on a GPU copy and the oracle on the CPU copy; return both results."""
    g = _gpu(p)
    kc, vc = g.k_cache.clone(), g.v_cache.clone()
    ks = g.k_scale.clone() if g.k_scale is not None else None
    vs = g.v_scale.clone() if g.v_scale is not None else None
    pa.append_kv(kn.cuda(), vn.cuda(), kc, vc, g.block_table, g.context_lens, k_scale=ks, v_scale=vs)
    assert pa.check_device_errors() == pa.PA_OK
    fp8 = p.kv_dtype == W.KV_FP8_E4M3
    ref = OA.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens, n_new=n_new,
                       block_size=p.block_size, fp8=fp8, k_scale=p.k_scale, v_scale=p.v_scale)
    got = (kc, vc, ks, vs) if fp8 else (kc, vc)
    return got, ref


def _bits(t):
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    return t.numpy()


def _assert_equal(got, ref):
    for i, (a, b) in enumerate(zip(got, ref)):
        b = np.asarray(b)
        a = _bits(a)
        if b.dtype == np.float32:
            b = b.view(np.uint32)
        assert a.shape == b.shape, i
        bad = np.argwhere(a != b)
        assert bad.size == 0, (i, len(bad), bad[:4].tolist())


@pytest.mark.parametrize("lens,n_new,Hkv,d", [
    ([20, 33, 16, 1], 1, 2, 128),
    ([37, 64, 18, 5, 100], 5, 4, 128),
    ([40, 32, 17], 16, 2, 64),
    ([300, 7], 3, 8, 64),
])
def test_append_bf16_bit_exact(lens, n_new, Hkv, d):
    p = W.make_problem(lens, Hkv * 2, Hkv, d, seed=61 + n_new)
    kn, vn = _new_rows(len(lens), n_new, Hkv, d, seed=7)
    got, ref = _append_both(p, kn, vn, n_new)
    _assert_equal(got, ref)


@pytest.mark.parametrize("lens,n_new,Hkv,d,mag", [
    ([20, 33, 16, 2], 1, 2, 128, 1.0),
    ([37, 64, 18, 5, 100], 5, 4, 128, 3.0),     # new tokens usually raise amax: old codes re-encoded
    ([40, 32, 17], 9, 2, 64, 1.0),
    ([300, 48, 31], 3, 8, 64, 1e-3),            # small new tokens: scale and old codes kept
    ([16, 32], 16, 2, 128, 1.0),                # whole fresh blocks
])
def test_append_fp8_bit_exact(lens, n_new, Hkv, d, mag):
    p = W.make_problem(lens, Hkv * 2, Hkv, d, seed=71 + n_new, kv_dtype=W.KV_FP8_E4M3)
    kn, vn = _new_rows(len(lens), n_new, Hkv, d, seed=8, mag=mag)
    got, ref = _append_both(p, kn, vn, n_new)
    _assert_equal(got, ref)


def test_append_then_decode_bf16_restores_cache():
    # write NaN over the last token of every sequence, append the original rows back: the pool is
    # bit-identical to the original and decode matches the oracle
    p = W.make_config("tiny", device="cuda")
    B, Hkv, d = p.num_seqs, p.num_kv_heads, p.head_dim
    orig_k, orig_v = p.k_cache.clone(), p.v_cache.clone()
    kn = torch.empty(B, 1, Hkv, d, dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    for b in range(B):
        j = int(p.context_lens[b]) - 1
        pb = int(p.block_table[b, j // 16])
        kn[b, 0] = p.k_cache[pb, :, j % 16]
        vn[b, 0] = p.v_cache[pb, :, j % 16]
        p.k_cache[pb, :, j % 16] = float("nan")
        p.v_cache[pb, :, j % 16] = float("nan")
    pa.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens)
    assert pa.check_device_errors() == pa.PA_OK
    assert torch.equal(p.k_cache.view(torch.int16), orig_k.view(torch.int16))
    assert torch.equal(p.v_cache.view(torch.int16), orig_v.view(torch.int16))
    out = pa.run_problem(p)
    ref = oracle.attention_problem(p.to("cpu"))
    parity.check(out.float().cpu().double().numpy(), ref, False, label=_label())


def test_append_then_decode_fp8_matches_oracle():
    p = W.make_problem([70, 33, 16, 129], 8, 2, 128, seed=81, kv_dtype=W.KV_FP8_E4M3)
    kn, vn = _new_rows(4, 1, 2, 128, seed=9, mag=2.0)
    g = _gpu(p)
    pa.append_kv(kn.cuda(), vn.cuda(), g.k_cache, g.v_cache, g.block_table, g.context_lens,
                 k_scale=g.k_scale, v_scale=g.v_scale)
    out = pa.run_problem(g)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    kc, vc, ks, vs = OA.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                                  n_new=1, block_size=16, fp8=True, k_scale=p.k_scale,
                                  v_scale=p.v_scale)
    cpu = dataclasses.replace(p, k_cache=torch.from_numpy(kc), v_cache=torch.from_numpy(vc),
                              k_scale=torch.from_numpy(ks), v_scale=torch.from_numpy(vs))
    ref = oracle.attention_problem(cpu)
    parity.check(out.float().cpu().double().numpy(), ref, True, label=_label())


def test_append_then_verify_chain():
    # the verify form appends its K+1 rows, then attends: same as the oracle over the new cache
    p = W.make_problem([50, 17, 96], 8, 2, 128, q_len=5, seed=82)
    kn, vn = _new_rows(3, 5, 2, 128, seed=10)
    g = _gpu(p)
    pa.append_kv(kn.cuda(), vn.cuda(), g.k_cache, g.v_cache, g.block_table, g.context_lens)
    out = pa.run_problem(g)
    torch.cuda.synchronize()
    kc, vc = OA.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens, n_new=5,
                          block_size=16)
    cpu = dataclasses.replace(p, k_cache=torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16),
                              v_cache=torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16))
    ref = oracle.attention_problem(cpu)
    parity.check(out.float().cpu().double().numpy(), ref, False, label=_label())


def test_append_short_context_is_flagged_and_skipped():
    p = W.make_problem([20, 3], 4, 2, 64, seed=83).to("cuda")
    before = p.k_cache.clone()
    kn, vn = _new_rows(2, 4, 2, 64, seed=11)
    cl = p.context_lens.clone()
    cl[0] = 4  # sequence 1 keeps length 3 < n_new
    pa.append_kv(kn.cuda(), vn.cuda(), p.k_cache, p.v_cache, p.block_table, cl)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    pb = int(p.block_table[1, 0])
    assert torch.equal(p.k_cache[pb].view(torch.int16), before[pb].view(torch.int16))
