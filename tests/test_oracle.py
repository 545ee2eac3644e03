"""Pins for the fp64 CPU oracle (no GPU).

The oracle is trusted only because these tests tie it to things other than itself:
  * exact decoders checked against torch's own bf16 / float8_e4m3fn conversions (all codes);
  * the special case that reduces to a library routine: paged attention gathered through the
    block table equals torch's scaled_dot_product_attention (float64) on the dense tensors,
    for decode and for the causal verify form, for several GQA shapes;
  * closed forms: one visible token returns its V, two tokens give sigmoid weights, identical
    keys or a zero scale give the mean of V;
  * invariants of the method: physical page order is irrelevant, GQA equals MHA with the KV
    heads repeated, verify row i equals decode with the context cut after that row, sequences
    sharing physical blocks equal unshared copies, outputs lie in the convex hull of the V rows;
  * tree masks: the chain mask is the causal verify, a random tree matches SDPA with the same
    visibility, and the rows on one branch equal a causal verify of that branch laid out alone.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_attn_gb300 import workloads as W


def _dense_sdpa(p: W.PagedAttnProblem):
    """torch SDPA (float64) on K/V gathered contiguous through the block table."""
    fp8 = p.kv_dtype == W.KV_FP8_E4M3
    if fp8:
        kc = p.k_cache.view(torch.float8_e4m3fn).double() * p.k_scale.double()[:, :, None, None]
        vc = p.v_cache.view(torch.float8_e4m3fn).double() * p.v_scale.double()[:, :, None, None]
    else:
        kc, vc = p.k_cache.double(), p.v_cache.double()
    G = p.num_q_heads // p.num_kv_heads
    out = torch.zeros(p.num_seqs, p.q_len, p.num_q_heads, p.head_dim, dtype=torch.float64)
    for b in range(p.num_seqs):
        L = int(p.context_lens[b])
        if L == 0:
            continue
        n = W.blocks_for(L, p.block_size)
        ids = p.block_table[b, :n].long()
        k = kc[ids].permute(1, 0, 2, 3).reshape(p.num_kv_heads, n * p.block_size, p.head_dim)[:, :L]
        v = vc[ids].permute(1, 0, 2, 3).reshape(p.num_kv_heads, n * p.block_size, p.head_dim)[:, :L]
        k = k.repeat_interleave(G, dim=0)[None]
        v = v.repeat_interleave(G, dim=0)[None]
        q = p.q[b].double().permute(1, 0, 2)[None]  # [1, Hq, q_len, d]
        pos_q = torch.arange(L - p.q_len, L)[:, None]
        mask = torch.arange(L)[None, :] <= pos_q
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=p.scale)
        out[b] = o[0].permute(1, 0, 2)
    return out.numpy()


def test_bf16_decoder_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(int(c)) for c in codes[::97]])
    r = ref[::97]
    both_nan = np.isnan(got) & np.isnan(r)
    assert np.all(both_nan | (got == r))


def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    both_nan = np.isnan(got) & np.isnan(ref)
    assert np.all(both_nan | (got == ref))
    # largest finite magnitude is 448 and the smallest subnormal is 2^-9
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9


SHAPES = [
    # (Hq, Hkv, d, lens, q_len)
    (4, 2, 64, [1, 17, 33, 64], 1),
    (8, 8, 32, [5, 16, 31], 1),
    (8, 1, 64, [40, 3], 1),
    (8, 2, 128, [50, 120, 20], 1),
    (4, 2, 64, [9, 30, 47], 5),
    (8, 2, 32, [17, 64], 9),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fp8", [False, True])
def test_matches_sdpa(shape, fp8):
    Hq, Hkv, d, lens, q_len = shape
    p = W.make_problem(lens, Hq, Hkv, d, q_len=q_len, seed=7 + len(lens) + d,
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    got = oracle.attention_problem(p)
    ref = _dense_sdpa(p)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_tiny_config_matches_sdpa():
    p = W.make_config("tiny")
    assert p.num_blocks == 32 and p.block_table.shape == (4, 4)
    np.testing.assert_allclose(oracle.attention_problem(p), _dense_sdpa(p), rtol=0, atol=1e-12)


def _permute_pool(p: W.PagedAttnProblem, seed: int):
    perm = torch.randperm(p.num_blocks, generator=torch.Generator().manual_seed(seed))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(p.num_blocks)
    # new physical block perm[i] holds what old block i held
    kc = torch.empty_like(p.k_cache)
    vc = torch.empty_like(p.v_cache)
    kc[perm] = p.k_cache
    vc[perm] = p.v_cache
    bt = p.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    import dataclasses

    ks = vs = None
    if p.k_scale is not None:
        ks = torch.empty_like(p.k_scale)
        vs = torch.empty_like(p.v_scale)
        ks[perm] = p.k_scale
        vs[perm] = p.v_scale
    return dataclasses.replace(p, k_cache=kc, v_cache=vc, block_table=bt, k_scale=ks, v_scale=vs)


@pytest.mark.parametrize("fp8", [False, True])
def test_page_permutation_invariance(fp8):
    p = W.make_problem([70, 3, 48, 16], 8, 2, 64, seed=11,
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    q = _permute_pool(p, 5)
    assert not torch.equal(p.block_table, q.block_table)
    a = oracle.attention_problem(p)
    b = oracle.attention_problem(q)
    assert np.array_equal(a, b)


def test_context_of_one_returns_v():
    p = W.make_problem([1, 1, 1], 4, 2, 64, seed=3)
    out = oracle.attention_problem(p)
    for b in range(3):
        pb = int(p.block_table[b, 0])
        for h in range(4):
            v = p.v_cache[pb, h // 2, 0].double().numpy()
            assert np.array_equal(out[b, 0, h], v)


def test_context_of_one_returns_v_fp8():
    p = W.make_problem([1, 1], 4, 4, 32, seed=4, kv_dtype=W.KV_FP8_E4M3)
    out = oracle.attention_problem(p)
    for b in range(2):
        pb = int(p.block_table[b, 0])
        for h in range(4):
            raw = p.v_cache[pb, h, 0].view(torch.float8_e4m3fn).double()
            v = (raw * float(p.v_scale[pb, h])).numpy()
            np.testing.assert_allclose(out[b, 0, h], v, rtol=1e-15, atol=0)


def test_identical_keys_give_mean_of_v():
    p = W.make_problem([37, 5], 4, 2, 64, seed=8)
    for b in range(2):
        L = int(p.context_lens[b])
        for j in range(L):
            pb = int(p.block_table[b, j // 16])
            p.k_cache[pb, :, j % 16] = p.k_cache[int(p.block_table[0, 0]), :, 0]
    out = oracle.attention_problem(p)
    for b in range(2):
        L = int(p.context_lens[b])
        for h in range(4):
            vs = [p.v_cache[int(p.block_table[b, j // 16]), h // 2, j % 16].double() for j in range(L)]
            mean = torch.stack(vs).mean(0).numpy()
            np.testing.assert_allclose(out[b, 0, h], mean, rtol=0, atol=1e-13)


def test_zero_scale_gives_mean_of_v():
    p = W.make_problem([29], 2, 1, 32, seed=9, scale=0.0)
    out = oracle.attention_problem(p)
    vs = [p.v_cache[int(p.block_table[0, j // 16]), 0, j % 16].double() for j in range(29)]
    np.testing.assert_allclose(out[0, 0, 0], torch.stack(vs).mean(0).numpy(), atol=1e-13, rtol=0)


def test_two_tokens_closed_form():
    p = W.make_problem([2], 2, 1, 16, seed=10)
    out = oracle.attention_problem(p)
    pb = int(p.block_table[0, 0])
    for h in range(2):
        q = p.q[0, 0, h].double()
        k0, k1 = p.k_cache[pb, 0, 0].double(), p.k_cache[pb, 0, 1].double()
        v0, v1 = p.v_cache[pb, 0, 0].double(), p.v_cache[pb, 0, 1].double()
        s0, s1 = p.scale * float(q @ k0), p.scale * float(q @ k1)
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(out[0, 0, h], (w0 * v0 + w1 * v1).numpy(), atol=1e-14, rtol=0)


def test_gqa_equals_mha_with_repeated_kv():
    G = 4
    p = W.make_problem([45, 16, 3], 8, 2, 32, seed=12)
    gqa = oracle.attention_problem(p)
    import dataclasses

    mha = dataclasses.replace(
        p, num_kv_heads=8,
        k_cache=p.k_cache.repeat_interleave(G, dim=1).contiguous(),
        v_cache=p.v_cache.repeat_interleave(G, dim=1).contiguous())
    assert np.array_equal(gqa, oracle.attention_problem(mha))


def test_group_size_one_is_mha_per_head():
    p = W.make_problem([33], 4, 4, 32, seed=13)
    out = oracle.attention_problem(p)
    for h in range(4):
        single = W.make_problem([33], 1, 1, 32, seed=13)
        import dataclasses

        single = dataclasses.replace(
            single, q=p.q[:, :, h : h + 1].contiguous(),
            k_cache=p.k_cache[:, h : h + 1].contiguous(), v_cache=p.v_cache[:, h : h + 1].contiguous(),
            block_table=p.block_table)
        assert np.array_equal(out[:, :, h : h + 1], oracle.attention_problem(single))


@pytest.mark.parametrize("fp8", [False, True])
def test_verify_row_equals_truncated_decode(fp8):
    q_len = 5
    p = W.make_problem([40, 21, 64], 8, 2, 64, q_len=q_len, seed=14,
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    ver = oracle.attention_problem(p)
    import dataclasses

    for i in range(q_len):
        lens = p.context_lens - (q_len - 1 - i)
        dec = dataclasses.replace(p, q=p.q[:, i : i + 1].contiguous(), q_len=1, context_lens=lens)
        assert np.array_equal(ver[:, i : i + 1], oracle.attention_problem(dec))


def test_shared_blocks_equal_unshared_copies():
    # sequence 1 shares its first two physical blocks with sequence 0 (prefix sharing)
    p = W.make_problem([40, 40], 4, 2, 32, seed=15)
    import dataclasses

    shared_bt = p.block_table.clone()
    shared_bt[1, :2] = p.block_table[0, :2]
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    for j in range(2):  # give the unshared copy the same contents
        kc[p.block_table[1, j]] = kc[p.block_table[0, j]]
        vc[p.block_table[1, j]] = vc[p.block_table[0, j]]
    unshared = dataclasses.replace(p, k_cache=kc, v_cache=vc)
    shared = dataclasses.replace(p, k_cache=kc, v_cache=vc, block_table=shared_bt)
    assert np.array_equal(oracle.attention_problem(shared), oracle.attention_problem(unshared))


def test_output_in_convex_hull_of_values():
    p = W.make_problem([90, 7, 16], 4, 2, 64, seed=16)
    out = oracle.attention_problem(p)
    for b in range(3):
        L = int(p.context_lens[b])
        for h in range(4):
            vs = torch.stack([p.v_cache[int(p.block_table[b, j // 16]), h // 2, j % 16].double()
                              for j in range(L)]).numpy()
            assert np.all(out[b, 0, h] <= vs.max(0) + 1e-12)
            assert np.all(out[b, 0, h] >= vs.min(0) - 1e-12)


def test_empty_context_gives_zeros_and_tail_is_never_read():
    p = W.make_problem([0, 5, 16, 17], 4, 2, 32, seed=17, tail_fill="nan")
    out = oracle.attention_problem(p)
    assert np.all(out[0] == 0)
    assert np.all(np.isfinite(out))


def test_subset_of_sequences():
    p = W.make_problem([10, 20, 30, 40], 4, 2, 32, seed=18)
    full = oracle.attention_problem(p)
    sub = oracle.attention_problem(p, seqs=[3, 1])
    assert np.array_equal(sub[[1, 3]], full[[1, 3]])
    assert np.all(sub[[0, 2]] == 0)


def test_bad_block_id_is_an_error():
    p = W.make_problem([20], 2, 1, 16, seed=19)
    p.block_table[0, 1] = p.num_blocks
    with pytest.raises(RuntimeError):
        oracle.attention_problem(p)


# --- tree verification masks (tree attention over a tree of draft branches) ---------------------

def _sdpa_tree(p, masks):
    """torch SDPA (float64) with the visibility a tree mask defines."""
    G = p.num_q_heads // p.num_kv_heads
    kc, vc = p.k_cache.double(), p.v_cache.double()
    out = torch.zeros(p.num_seqs, p.q_len, p.num_q_heads, p.head_dim, dtype=torch.float64)
    for b in range(p.num_seqs):
        L = int(p.context_lens[b])
        n = W.blocks_for(L, p.block_size)
        ids = p.block_table[b, :n].long()
        k = kc[ids].permute(1, 0, 2, 3).reshape(p.num_kv_heads, -1, p.head_dim)[:, :L]
        v = vc[ids].permute(1, 0, 2, 3).reshape(p.num_kv_heads, -1, p.head_dim)[:, :L]
        k = k.repeat_interleave(G, dim=0)[None]
        v = v.repeat_interleave(G, dim=0)[None]
        q = p.q[b].double().permute(1, 0, 2)[None]
        first_new = L - p.q_len
        vis = torch.zeros(p.q_len, L, dtype=torch.bool)
        vis[:, :first_new] = True
        for i in range(p.q_len):
            for t in range(p.q_len):
                vis[i, first_new + t] = bool((int(masks[b, i]) >> t) & 1)
        out[b] = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=vis, scale=p.scale)[0].permute(1, 0, 2)
    return out.numpy()


def test_chain_mask_equals_causal_verify():
    p = W.make_problem([30, 70, 9], 8, 2, 32, q_len=7, seed=31)
    causal = oracle.attention_problem(p)
    chain = oracle.attention_problem(p, tree_mask=W.chain_mask(3, 7))
    assert np.array_equal(causal, chain)


@pytest.mark.parametrize("fp8", [False, True])
def test_tree_mask_matches_sdpa(fp8):
    p = W.make_problem([40, 23, 90], 8, 2, 32, q_len=9, seed=32,
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    masks = W.random_tree_masks(3, 9, seed=5)
    got = oracle.attention_problem(p, tree_mask=masks)
    if fp8:
        ref = _sdpa_tree_fp8(p, masks)
    else:
        ref = _sdpa_tree(p, masks)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def _sdpa_tree_fp8(p, masks):
    import dataclasses

    kc = p.k_cache.view(torch.float8_e4m3fn).double() * p.k_scale.double()[:, :, None, None]
    vc = p.v_cache.view(torch.float8_e4m3fn).double() * p.v_scale.double()[:, :, None, None]
    # reuse the bf16 helper on float64 copies of the dequantised pools
    q = dataclasses.replace(p, k_cache=kc, v_cache=vc)
    return _sdpa_tree(q, masks)


def test_tree_branch_equals_causal_chain():
    # rows on one branch of a tree see exactly what a causal verify of that branch sees
    Hq, Hkv, d, prior = 4, 2, 32, 37
    masks = torch.tensor([[0b1, 0b11, 0b101, 0b1011, 0b10101]], dtype=torch.int32)  # 0-1-3, 0-2-4
    p = W.make_problem([prior + 5], Hq, Hkv, d, q_len=5, seed=33)
    tree = oracle.attention_problem(p, tree_mask=masks)
    for branch in ([0, 1, 3], [0, 2, 4]):
        c = W.make_problem([prior + len(branch)], Hq, Hkv, d, q_len=len(branch), seed=34,
                           pool_factor=2.0)
        def slot(prob, j):
            return int(prob.block_table[0, j // 16]), j % 16
        for j in range(prior + len(branch)):
            src = j if j < prior else prior + branch[j - prior]
            sb, st = slot(p, src)
            db, dt = slot(c, j)
            c.k_cache[db, :, dt] = p.k_cache[sb, :, st]
            c.v_cache[db, :, dt] = p.v_cache[sb, :, st]
        c.q[0] = p.q[0, branch]
        chain = oracle.attention_problem(c)
        assert np.array_equal(chain[0], tree[0, branch])
