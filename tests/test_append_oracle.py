"""Pins for the KV-append oracle (no GPU): the E4M3 encoder against torch's float8 cast and the
OCP definition, the bf16 path as plain indexing, and the fp8 scale policy."""

import numpy as np
import pytest
import torch

import oracle
from oracle import append as OA
from paged_kv_gqa_attn_gb300 import workloads as W


def test_e4m3_decode_matches_torch():
    codes = np.arange(256)
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([OA.e4m3_decode(int(c)) for c in codes])
    assert np.all((np.isnan(got) & np.isnan(ref)) | (got == ref))


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(1)
    x = torch.cat([
        torch.randn(4000, generator=g) * 100,
        torch.randn(2000, generator=g) * 1e-2,
        torch.randn(2000, generator=g) * 1e-3,
    ]).clamp(-463.9, 463.9).float()
    # exact code values and the midpoints between neighbours (ties)
    vals = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).float()
    vals = vals[torch.isfinite(vals)].unique()
    mids = ((vals[1:].double() + vals[:-1].double()) / 2).float()
    x = torch.cat([x, vals, mids])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([OA.e4m3_encode(float(v)) for v in x.numpy()], dtype=np.uint8)
    zero = (x == 0).numpy()  # signed zeros may differ in sign bit only
    assert np.array_equal(got[~zero], ref[~zero])


def test_e4m3_encode_saturates():
    for v in [448.0, 464.0, 480.0, 1e6, float(np.finfo(np.float32).max)]:
        assert OA.e4m3_encode(v) == 0x7E
        assert OA.e4m3_encode(-v) == 0xFE
    assert OA.e4m3_encode(float("nan")) == 0x7F


def _new_tokens(B, n_new, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, n_new, Hkv, d, generator=g).to(torch.bfloat16),
            torch.randn(B, n_new, Hkv, d, generator=g).to(torch.bfloat16))


def test_bf16_append_is_a_scatter():
    p = W.make_problem([20, 33, 16], 4, 2, 32, seed=41)
    n_new = 3
    kn, vn = _new_tokens(3, n_new, 2, 32, 5)
    kc, vc = OA.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                          n_new=n_new, block_size=16)
    kc = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    for b in range(3):
        L = int(p.context_lens[b])
        for t in range(n_new):
            j = L - n_new + t
            pb = int(p.block_table[b, j // 16])
            assert torch.equal(kc[pb, :, j % 16], kn[b, t])
    # nothing else moved
    touched = torch.zeros_like(p.k_cache, dtype=torch.bool)
    for b in range(3):
        L = int(p.context_lens[b])
        for j in range(L - n_new, L):
            touched[int(p.block_table[b, j // 16]), :, j % 16] = True
    assert torch.equal(kc[~touched], p.k_cache[~touched])


def test_fp8_append_scale_is_block_amax_over_448():
    p = W.make_problem([20, 16, 40], 4, 2, 32, seed=42, kv_dtype=W.KV_FP8_E4M3)
    n_new = 5
    kn, vn = _new_tokens(3, n_new, 2, 32, 6)
    kc, vc, ks, vs = OA.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                                  n_new=n_new, block_size=16, fp8=True, k_scale=p.k_scale,
                                  v_scale=p.v_scale)
    for b in range(3):
        L = int(p.context_lens[b])
        for blk in range((L - n_new) // 16, (L - 1) // 16 + 1):
            pb = int(p.block_table[b, blk])
            n_valid = min(L - blk * 16, 16)
            for g in range(2):
                vals = np.array([[OA.e4m3_decode(int(x)) for x in row] for row in kc[pb, g, :n_valid]])
                # after the append the largest code in the block is the largest E4M3 value (448)
                assert np.abs(vals).max() == 448.0
                # every new token decodes back within half an E4M3 step of its input
                for sl in range(max(L - n_new - blk * 16, 0), n_valid):
                    t = blk * 16 + sl - (L - n_new)
                    x = kn[b, t, g].float().numpy()
                    y = vals[sl] * ks[pb, g]
                    assert np.all(np.abs(x - y) <= np.abs(x) * 2 ** -4 + ks[pb, g] * 2 ** -9 + 1e-7)


def test_fp8_append_small_values_keep_old_bytes():
    # new values below the block's amax: the scale and the old codes do not change.  The cache
    # holds 18 tokens (block 1: slots 0, 1); the append brings the context to 20.
    p = W.make_problem([18], 2, 1, 32, seed=43, kv_dtype=W.KV_FP8_E4M3)
    p.context_lens = torch.tensor([20], dtype=torch.int32)
    n_new = 2
    kn = torch.full((1, n_new, 1, 32), 1e-3).to(torch.bfloat16)
    vn = kn.clone()
    before = p.k_cache.clone()
    kc, vc, ks, vs = OA.append_kv(kn, vn, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                                  n_new=n_new, block_size=16, fp8=True, k_scale=p.k_scale,
                                  v_scale=p.v_scale)
    pb = int(p.block_table[0, 1])  # tokens 16..19: old 16, 17 and new 18, 19
    # (448 s) / 448 in fp32 may land one ulp from s; the old codes do not move either way
    assert abs(ks[pb, 0] - p.k_scale[pb, 0].item()) <= 2 ** -22 * p.k_scale[pb, 0].item()
    assert np.array_equal(kc[pb, 0, :2], before[pb, 0, :2].numpy())
