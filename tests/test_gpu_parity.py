"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle on the same seeded
inputs.  Tolerances (on the bf16 output vs the fp64 oracle): bf16 KV max abs 1e-2 and mean abs
1e-3; fp8 KV max abs 5e-2 (the oracle decodes the stored fp8 bytes, so this measures kernel
error, not quantisation error).  Every element is held to the flat bar, except where the oracle
value is so large that half a bf16 ulp of it already reaches the bar (|o| >= 4 for bf16, >= 16
for fp8): no bf16 output can meet the flat bar there, and those elements are allowed half an ulp
of their own value plus 2e-3 (oracle.parity).  Each check prints the observed worst and mean
error."""

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

BF16_MAX, BF16_MEAN, FP8_MAX = parity.BF16_MAX, parity.BF16_MEAN, parity.FP8_MAX


def _label():
    return os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]


def _check(got, ref, fp8, mean_bar=True):
    """The element-wise bound of oracle.parity: the flat bar wherever a bf16 value can meet it."""
    if isinstance(got, torch.Tensor):
        got = got.float().cpu().double().numpy()
    return parity.check(got, ref, fp8, label=_label(), mean_bar=mean_bar)


def _assert_parity(p, out, seqs=None):
    ref = oracle.attention_problem(p, seqs=seqs)
    g = out.float().cpu().double().numpy()
    if seqs is not None:
        g, ref = g[seqs], ref[seqs]
    return _check(g, ref, p.kv_dtype == W.KV_FP8_E4M3)


def _run(p, **kw):
    out = pa.run_problem(p, **kw)
    torch.cuda.synchronize()
    return out


@pytest.fixture(autouse=True)
def _reset_partitions():
    pa.set_max_partitions(0)
    yield
    pa.set_max_partitions(0)
    torch.cuda.synchronize()


def _clean_errors():
    pa.check_device_errors()


# --- the named workloads ------------------------------------------------------------------

def test_tiny():
    p = W.make_config("tiny", device="cuda")
    _clean_errors()
    out = _run(p)
    _assert_parity(p, out)
    assert pa.check_device_errors() == pa.PA_OK


def test_llama8b_decode_full_size():
    p = W.make_config("llama8b_decode", device="cuda")
    out = _run(p)
    _assert_parity(p, out, seqs=list(range(0, 64, 4)))
    assert torch.isfinite(out.float()).all()


def test_llama70b_decode_full_size():
    # groups of 8 query heads with a bf16 cache: decode runs the tensor-core kernel
    p = W.make_config("llama70b_decode", device="cuda")
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_OK
    _assert_parity(p, out, seqs=list(range(1, 64, 4)))
    assert torch.isfinite(out.float()).all()


def test_cb_mix_full_size():
    p = W.make_config("cb_mix", device="cuda")
    lens = p.context_lens.cpu().tolist()
    order = np.argsort(lens)
    seqs = sorted(set(order[:12].tolist() + order[-12:].tolist() + list(range(0, 256, 16))))
    out = _run(p)
    _assert_parity(p, out, seqs=seqs)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", ["spec_verify_k4", "spec_verify_k8"])
def test_spec_verify_full_size(name):
    p = W.make_config(name, device="cuda")
    out = _run(p)
    _assert_parity(p, out)


def test_long_fp8_full_size():
    p = W.make_config("long_fp8", device="cuda")
    out = _run(p)
    _assert_parity(p, out, seqs=[0, 3])
    assert torch.isfinite(out.float()).all()


# --- shapes spanning several tiles, ragged tails and every supported group / head dim ------

DECODE_SHAPES = [
    # Hq, Hkv, d, lens
    (8, 8, 128, [1, 2, 15, 16, 17, 31]),
    (8, 4, 128, [33, 64, 65, 100, 129]),
    (32, 8, 128, [1, 17, 300, 513, 1000, 2049]),
    (16, 2, 128, [5, 200, 777]),
    (4, 2, 64, [1, 17, 33, 64, 511, 1025]),
    (8, 1, 64, [7, 90, 400]),
    (8, 8, 64, [3, 48, 49]),
    (16, 2, 64, [16, 250, 600]),
]


@pytest.mark.parametrize("shape", DECODE_SHAPES)
@pytest.mark.parametrize("fp8", [False, True])
def test_decode_shapes(shape, fp8):
    Hq, Hkv, d, lens = shape
    p = W.make_problem(lens, Hq, Hkv, d, seed=100 + sum(lens) % 97 + d, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16, tail_fill="nan")
    _clean_errors()
    out = _run(p)
    _assert_parity(p, out)
    assert pa.check_device_errors() == pa.PA_OK


# groups other than 1, 2, 4, 8 (e.g. 40 / 8 = 5 and 28 / 4 = 7 query heads per kv head, or 16 and
# more) take the tensor-core verify kernel with q_len = 1
OTHER_GROUP_SHAPES = [
    # Hq, Hkv, d, lens
    (15, 5, 128, [1, 17, 300, 1000]),   # 3
    (40, 8, 128, [33, 700, 2100]),      # 5
    (28, 4, 128, [5, 1100]),            # 7
    (32, 2, 64, [16, 400]),             # 16
    (64, 2, 128, [9, 260]),             # 32
    (64, 1, 64, [3, 130]),              # 64
]


@pytest.mark.parametrize("shape", OTHER_GROUP_SHAPES)
@pytest.mark.parametrize("fp8", [False, True])
def test_decode_other_groups(shape, fp8):
    Hq, Hkv, d, lens = shape
    p = W.make_problem(lens, Hq, Hkv, d, seed=150 + Hq + d, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16, tail_fill="nan")
    _clean_errors()
    out = _run(p)
    _assert_parity(p, out)
    assert pa.check_device_errors() == pa.PA_OK


VERIFY_SHAPES = [
    # Hq, Hkv, d, lens, q_len
    (32, 8, 128, [5, 16, 17, 100, 1029], 5),
    (32, 8, 128, [9, 64, 65, 700, 2100], 9),
    (8, 8, 128, [1, 2, 40], 1),
    (8, 2, 128, [16, 33, 300], 16),
    (4, 2, 64, [3, 40, 129, 515], 3),
    (16, 4, 64, [12, 77, 1100], 12),
    (8, 1, 64, [8, 200], 8),
    (8, 1, 128, [8, 129, 1500], 8),      # G = 8 at d = 128: 64 rows, the most one tile takes
    (16, 16, 128, [16, 300, 641], 16),   # MHA (G = 1) at the largest q_len
    (4, 2, 128, [2, 2, 70], 2),          # contexts equal to q_len: no prefix at all
]


@pytest.mark.parametrize("shape", VERIFY_SHAPES)
def test_verify_shapes(shape):
    Hq, Hkv, d, lens, q_len = shape
    p = W.make_problem(lens, Hq, Hkv, d, q_len=q_len, seed=200 + sum(lens) % 89 + d, device="cuda",
                       tail_fill="nan")
    _clean_errors()
    out = pa.verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, p.scale)
    torch.cuda.synchronize()
    _assert_parity(p, out)
    assert pa.check_device_errors() == pa.PA_OK


FP8_VERIFY_SHAPES = [
    # Hq, Hkv, d, lens, q_len
    (32, 8, 128, [9, 64, 65, 700, 2100], 9),
    (32, 8, 128, [5, 16, 17, 100, 1029], 5),
    (8, 1, 128, [8, 129, 1500], 8),
    (4, 2, 64, [3, 40, 129, 515], 3),
    (16, 16, 128, [16, 300], 16),
    (8, 8, 128, [1, 2, 40, 3000], 1),
]


@pytest.mark.parametrize("shape", FP8_VERIFY_SHAPES)
def test_verify_shapes_fp8(shape):
    # E4M3 caches on the tensor-core kernel: pages converted to f16 in shared memory
    Hq, Hkv, d, lens, q_len = shape
    p = W.make_problem(lens, Hq, Hkv, d, q_len=q_len, seed=300 + sum(lens) % 89 + d, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3, tail_fill="nan")
    _clean_errors()
    out = pa.verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, p.scale,
                    k_scale=p.k_scale, v_scale=p.v_scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    _assert_parity(p, out)


def test_spec_verify_k8_fp8_full_size():
    p = W.make_config("spec_verify_k8", device="cuda", kv_dtype=W.KV_FP8_E4M3)
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_OK
    _assert_parity(p, out)


# --- E4M3 decode: per-page scales of any sign and size, and a running max that jumps late ------
# The E4M3 decode folds each page's V scale into the softmax weight as log2|scale| (and its sign)
# and refreshes the running max only when a score passes it by a margin; these cases drive both.

@pytest.mark.parametrize("d", [64, 128])
def test_fp8_decode_scales_of_any_sign(d):
    p = W.make_problem([5, 47, 300, 1200], 16, 4, d, seed=810 + d, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3, tail_fill="nan")
    g = torch.Generator().manual_seed(811)
    n = p.v_scale.numel()
    pick = torch.randint(0, 4, (n,), generator=g).view_as(p.v_scale).to(p.v_scale.device)
    vs = p.v_scale.clone()
    vs[pick == 0] *= -1.0      # negative scale: the page's values change sign
    vs[pick == 1] = 0.0        # zero scale: the page contributes weight but no value
    vs[pick == 2] *= 4.0
    ks = p.k_scale.clone()
    ks[torch.randint(0, 3, (n,), generator=g).view_as(ks).to(ks.device) == 0] *= -1.0
    q = dataclasses.replace(p, v_scale=vs, k_scale=ks)
    _clean_errors()
    out = _run(q)
    assert pa.check_device_errors() == pa.PA_OK
    _assert_parity(q, out)


@pytest.mark.parametrize("factor", [2.0 ** 12, 2.0 ** -40])
def test_fp8_decode_extreme_v_scales_scale_the_output(factor):
    # a power of two times every V scale multiplies the exact output by it, and the bf16 rounding
    # of a power-of-two multiple is the same multiple of the rounding
    p = W.make_problem([33, 700, 2100], 32, 8, 128, seed=812, device="cuda", kv_dtype=W.KV_FP8_E4M3)
    base = _run(p).float()
    big = _run(dataclasses.replace(p, v_scale=p.v_scale * factor)).float()
    ref = oracle.attention_problem(p)
    _check(big.cpu().double().numpy() / factor, ref, True)
    assert (big / factor - base).abs().max().item() <= 2e-2


@pytest.mark.parametrize("at", ["late", "early"])
def test_fp8_decode_running_max_jumps(at):
    # one page's K scale times 64 lifts its scores ~90 log2 units above the rest: the running max
    # jumps there (late: after many pages were accumulated; early: the rest sits far below it)
    lens = [900, 2000, 4100]
    p = W.make_problem(lens, 32, 8, 128, seed=813, device="cuda", kv_dtype=W.KV_FP8_E4M3)
    ks = p.k_scale.clone()
    for b, L in enumerate(lens):
        j = (L - 1) // 16 - 1 if at == "late" else 1
        ks[int(p.block_table[b, j])] *= 64.0
    q = dataclasses.replace(p, k_scale=ks)
    out = _run(q)
    _assert_parity(q, out)


@pytest.mark.parametrize("at", ["late", "early"])
@pytest.mark.parametrize("Hq", [32, 64])
def test_bf16_decode_running_max_jumps(at, Hq):
    # bf16 pages: one page's K times 64 (exact in bf16) lifts its scores far above the rest, so the
    # running max jumps there; groups of 4 carry the weights' low parts in spare columns, groups
    # of 8 in a second P.V pass
    lens = [900, 2000, 4100]
    p = W.make_problem(lens, Hq, 8, 128, seed=814, device="cuda")
    kc = p.k_cache.clone()
    for b, L in enumerate(lens):
        j = (L - 1) // 16 - 1 if at == "late" else 1
        kc[int(p.block_table[b, j])] *= 64.0
    q = dataclasses.replace(p, k_cache=kc)
    out = _run(q)
    _assert_parity(q, out)


@pytest.mark.parametrize("seed", range(12))
def test_decode_random_problems(seed):
    # seeded random decode shapes: group size, head dim, kv heads, ragged contexts (incl. 1, page
    # edges, windows of more than 32 pages per warp), KV type and a forced or automatic split
    rng = np.random.default_rng(1000 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.choice([1, 15, 16, 17, 255, 256, 257, 1000, 2111, 4100], size=B)]
    fp8 = bool(rng.integers(0, 2))
    P = int(rng.choice([0, 0, 1, 2, 5, 64]))
    p = W.make_problem(lens, G * Hkv, Hkv, d, seed=1100 + seed, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16, tail_fill="nan")
    pa.set_max_partitions(P)
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_OK
    _assert_parity(p, out)


@pytest.mark.parametrize("seed", range(10))
def test_verify_random_problems(seed):
    # seeded random verify and tree-verify shapes over both verify routes (up to 64 rows per kv
    # head: the verify kernel, bf16 or E4M3; 65-128 rows, bf16: the split prefill kernel)
    rng = np.random.default_rng(2000 + seed)
    q_len = int(rng.integers(2, 17))
    G = int(rng.choice([g for g in (1, 2, 3, 4, 5, 8, 16) if g * q_len <= 128]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 6))
    lens = [max(q_len, int(x)) for x in rng.choice([1, 16, 17, 64, 65, 257, 700, 1500, 3100], size=B)]
    fp8 = bool(rng.integers(0, 2)) and G * q_len <= 64
    tree = bool(rng.integers(0, 2))
    p = W.make_problem(lens, G * Hkv, Hkv, d, q_len=q_len, seed=2100 + seed, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16, tail_fill="nan")
    _clean_errors()
    if tree:
        masks = W.random_tree_masks(B, q_len, seed=seed).to("cuda")
        out = pa.tree_verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, masks, p.scale,
                             k_scale=p.k_scale, v_scale=p.v_scale)
        torch.cuda.synchronize()
        ref = oracle.attention_problem(p, tree_mask=masks)
        _check(out, ref, fp8)
    else:
        out = _run(p)
        _assert_parity(p, out)
    assert pa.check_device_errors() == pa.PA_OK


@pytest.mark.parametrize("P", [1, 2, 7, 64])
@pytest.mark.parametrize("form", ["decode", "verify", "fp8"])
def test_split_count_does_not_change_results(P, form):
    q_len = 5 if form == "verify" else 1
    p = W.make_problem([1, 40, 700, 1500, 2100], 32, 8, 128, q_len=q_len, seed=300, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3 if form == "fp8" else W.KV_BF16)
    pa.set_max_partitions(P)
    out = _run(p)
    _assert_parity(p, out)
    pa.set_max_partitions(1)
    one = _run(p)
    d = (out.float() - one.float()).abs().max().item()
    assert d <= 2e-2


# --- invariants ------------------------------------------------------------------------------

def _permute_pool(p, seed):
    perm = torch.randperm(p.num_blocks, generator=torch.Generator().manual_seed(seed)).to(p.k_cache.device)
    kc = torch.empty_like(p.k_cache)
    vc = torch.empty_like(p.v_cache)
    kc[perm] = p.k_cache
    vc[perm] = p.v_cache
    bt = p.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    ks = vs = None
    if p.k_scale is not None:
        ks = torch.empty_like(p.k_scale)
        vs = torch.empty_like(p.v_scale)
        ks[perm] = p.k_scale
        vs[perm] = p.v_scale
    return dataclasses.replace(p, k_cache=kc, v_cache=vc, block_table=bt, k_scale=ks, v_scale=vs)


@pytest.mark.parametrize("q_len,fp8", [(1, False), (1, True), (5, False)])
def test_page_permutation_is_bit_identical(q_len, fp8):
    p = W.make_problem([70, 3, 480, 1600], 32, 8, 128, q_len=q_len, seed=400, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    a = _run(p)
    b = _run(_permute_pool(p, 9))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_deterministic():
    p = W.make_config("cb_mix", device="cuda")
    a = _run(p)
    b = _run(p)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_verify_row_equals_truncated_decode():
    q_len = 9
    p = W.make_problem([40, 300, 1100], 32, 8, 128, q_len=q_len, seed=500, device="cuda")
    ver = _run(p).float()
    for i in range(q_len):
        lens = p.context_lens - (q_len - 1 - i)
        dec = dataclasses.replace(p, q=p.q[:, i : i + 1].contiguous(), q_len=1, context_lens=lens.contiguous())
        d = _run(dec).float()
        assert (ver[:, i : i + 1] - d).abs().max().item() <= 2e-2


def test_shared_blocks_equal_unshared():
    p = W.make_problem([600, 600], 32, 8, 128, seed=600, device="cuda")
    n_shared = 20
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    for j in range(n_shared):
        kc[p.block_table[1, j]] = kc[p.block_table[0, j]]
        vc[p.block_table[1, j]] = vc[p.block_table[0, j]]
    bt = p.block_table.clone()
    bt[1, :n_shared] = p.block_table[0, :n_shared]
    unshared = _run(dataclasses.replace(p, k_cache=kc, v_cache=vc))
    shared = _run(dataclasses.replace(p, k_cache=kc, v_cache=vc, block_table=bt))
    assert torch.equal(unshared.view(torch.int16), shared.view(torch.int16))


def test_context_of_one_returns_v():
    p = W.make_problem([1, 1, 1], 32, 8, 128, seed=700, device="cuda")
    out = _run(p).float()
    for b in range(3):
        pb = int(p.block_table[b, 0])
        for h in range(32):
            assert torch.equal(out[b, 0, h], p.v_cache[pb, h // 4, 0].float())


def _e4m3_values(codes):
    """E4M3 codes (uint8) -> float32 through torch's float8 type (exact)."""
    return codes.view(torch.float8_e4m3fn).float()


def test_context_of_one_returns_dequantized_v_fp8():
    # one visible token: the output is that token's V, E4M3 code times its page's V scale
    p = W.make_problem([1, 1, 1], 32, 8, 128, seed=703, device="cuda", kv_dtype=W.KV_FP8_E4M3)
    out = _run(p).float()
    for b in range(3):
        pb = int(p.block_table[b, 0])
        for g in range(8):
            v = (_e4m3_values(p.v_cache[pb, g, 0]) * p.v_scale[pb, g]).to(torch.bfloat16).float()
            for h in range(4):
                assert (out[b, 0, g * 4 + h] - v).abs().max().item() <= 1e-6 + 2 ** -8 * v.abs().max().item()


@pytest.mark.parametrize("fp8", [False, True])
def test_zero_scale_gives_mean_of_visible_v(fp8):
    # scale 0: every visible token weighs the same, so each row is the mean of its V rows
    p = W.make_problem([1, 17, 300], 32, 8, 128, seed=704, device="cuda", scale=0.0,
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    out = _run(p).float().cpu()
    for b, L in enumerate([1, 17, 300]):
        rows = []
        for j in range(L):
            pb = int(p.block_table[b, j // 16])
            v = p.v_cache[pb, :, j % 16]
            v = (_e4m3_values(v) * p.v_scale[pb][:, None]) if fp8 else v.float()
            rows.append(v.cpu().double())
        mean = torch.stack(rows).mean(0)  # [Hkv, d]
        ref = mean.repeat_interleave(4, dim=0)
        assert (out[b, 0].double() - ref).abs().max().item() <= (FP8_MAX if fp8 else BF16_MAX)


@pytest.mark.parametrize("fp8", [False, True])
def test_gqa_equals_mha_with_repeated_kv(fp8):
    # a group of 4 query heads over one kv head = 4 heads over 4 copies of it (groups of 1)
    p = W.make_problem([40, 700, 2100], 32, 8, 128, seed=820, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    rep = lambda t: None if t is None else t.repeat_interleave(4, dim=1).contiguous()
    mha = dataclasses.replace(p, num_kv_heads=32, k_cache=rep(p.k_cache), v_cache=rep(p.v_cache),
                              k_scale=rep(p.k_scale), v_scale=rep(p.v_scale))
    a = _run(p).float()
    b = _run(mha).float()
    assert (a - b).abs().max().item() <= 2e-2


@pytest.mark.parametrize("fp8", [False, True])
def test_output_in_hull_of_visible_v(fp8):
    # softmax weights are positive and sum to 1: each output dim lies between the smallest and the
    # largest value of that dim over the visible V rows
    lens = [3, 40, 333]
    p = W.make_problem(lens, 16, 4, 128, seed=821, device="cuda", kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    out = _run(p).float().cpu()
    tol = FP8_MAX if fp8 else BF16_MAX
    for b, L in enumerate(lens):
        rows = []
        for j in range(L):
            pb = int(p.block_table[b, j // 16])
            v = p.v_cache[pb, :, j % 16]
            v = (_e4m3_values(v) * p.v_scale[pb][:, None]) if fp8 else v.float()
            rows.append(v.cpu())
        vs = torch.stack(rows)  # [L, Hkv, d]
        lo = vs.min(0).values.repeat_interleave(4, dim=0)
        hi = vs.max(0).values.repeat_interleave(4, dim=0)
        o = out[b, 0]
        assert (o >= lo - tol).all() and (o <= hi + tol).all()


def test_identical_keys_give_mean_of_v():
    p = W.make_problem([300], 8, 2, 128, seed=701, device="cuda")
    blk0 = int(p.block_table[0, 0])
    for j in range(300):
        pb = int(p.block_table[0, j // 16])
        p.k_cache[pb, :, j % 16] = p.k_cache[blk0, :, 0]
    out = _run(p).float()
    ref = oracle.attention_problem(p)
    _check(out.cpu().double().numpy(), ref, False)


def test_output_canary_fully_written():
    p = W.make_problem([5, 900, 3000], 32, 8, 128, seed=702, device="cuda")
    out = torch.full_like(p.q, float("nan"))
    pa.run_problem(p, out=out)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


def test_non_default_stream():
    p = W.make_problem([100, 2000], 32, 8, 128, seed=703, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = pa.run_problem(p, stream=s)
    s.synchronize()
    _assert_parity(p, out)


# --- device-side error reporting (never a fault: the kernels skip what they flag) ------------

def test_out_of_range_block_id_is_flagged_not_read():
    p = W.make_problem([40, 40], 8, 2, 128, seed=800, device="cuda")
    _clean_errors()
    bt = p.block_table.clone()
    bt[1, 1] = p.num_blocks + 5
    bad = dataclasses.replace(p, block_table=bt)
    out = _run(bad)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    # the untouched sequence is still right
    ref = oracle.attention_problem(p)
    _check(out[0], ref[0], False)


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8_E4M3])
def test_verify_out_of_range_block_id_is_flagged_not_read(kv):
    # a page id past the pool and a negative one inside a verify sequence's context: flagged, the
    # pages skipped (the valid-page bits the K producer hands the softmax), the other sequences exact
    p = W.make_problem([700, 900, 300], 16, 4, 128, q_len=5, seed=805, device="cuda", kv_dtype=kv)
    _clean_errors()
    bt = p.block_table.clone()
    bt[1, 3] = p.num_blocks + 5
    bt[1, 20] = -7
    bad = dataclasses.replace(p, block_table=bt)
    out = _run(bad)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    assert torch.isfinite(out.float()).all()
    _assert_parity(p, out, seqs=[0, 2])


def test_empty_context_gives_zeros_and_is_flagged():
    p = W.make_problem([0, 20], 8, 2, 128, seed=801, device="cuda")
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    assert torch.all(out[0] == 0)
    _assert_parity(p, out, seqs=[1])


def test_verify_context_shorter_than_q_len_is_flagged():
    p = W.make_problem([3, 20], 8, 2, 128, q_len=5, seed=802, device="cuda")
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    # rows 0 and 1 of sequence 0 see no token and are zero; the others are ordinary rows
    assert torch.all(out[0, :2] == 0)
    _assert_parity(p, out)


def test_verify_long_and_short_sequences():
    # long sequences split over many CTAs next to one that fits in a single CTA's range
    p = W.make_problem([5000, 4200, 77], 32, 8, 128, q_len=5, seed=900, device="cuda")
    pa.set_max_partitions(1)
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_OK
    _assert_parity(p, out)


# --- tree verification ---------------------------------------------------------------------------

# verify with more than 64 rows per kv head (bf16): the chunked-prefill kernel split like decode
WIDE_VERIFY_SHAPES = [
    # Hq, Hkv, d, lens, q_len
    (32, 4, 128, [9, 300, 2100], 9),        # groups of 8, 8 drafts: 72 rows
    (64, 8, 128, [16, 500, 1500], 16),      # 128 rows
    (32, 2, 64, [5, 90, 700], 5),           # groups of 16: 80 rows
    (16, 1, 128, [8, 17, 1000], 8),         # 128 rows, one kv head
]


@pytest.mark.parametrize("shape", WIDE_VERIFY_SHAPES)
@pytest.mark.parametrize("fp8", [False, True])
def test_wide_verify_matches_oracle(shape, fp8):
    Hq, Hkv, d, lens, q_len = shape
    p = W.make_problem(lens, Hq, Hkv, d, q_len=q_len, seed=970 + q_len + d, device="cuda", tail_fill="nan",
                       kv_dtype=W.KV_FP8_E4M3 if fp8 else W.KV_BF16)
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_OK
    _assert_parity(p, out)


def test_wide_tree_verify_fp8_matches_oracle():
    p = W.make_problem([9, 300, 2100], 32, 4, 128, q_len=9, seed=977, device="cuda", tail_fill="nan",
                       kv_dtype=W.KV_FP8_E4M3)
    masks = W.random_tree_masks(3, 9, seed=6).to("cuda")
    _clean_errors()
    out = pa.tree_verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, masks, p.scale,
                         k_scale=p.k_scale, v_scale=p.v_scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    _check(out, oracle.attention_problem(p, tree_mask=masks), True)


# --- E4M3 caches: q of any bf16 magnitude (the f16 products scale each query row by a power of
# two first), against the oracle on the same bf16 q ------------------------------------------

def _extreme_q(p, seed):
    """A copy of p whose q has, per sequence, one row scaled by 1e5 (|q| far above the f16
    maximum), one by 1e-30 (far below f16's smallest subnormal) and a few single entries set to
    -2e5."""
    q = p.q.clone().float()
    g = torch.Generator().manual_seed(seed)
    B, QL, Hq, d = q.shape
    for b in range(B):
        i = int(torch.randint(0, QL, (1,), generator=g))
        h1, h2 = (int(x) for x in torch.randperm(Hq, generator=g)[:2])
        q[b, i, h1] *= 1e5
        q[b, QL - 1 - i, h2] *= 1e-30
        for _ in range(3):
            q[b, int(torch.randint(0, QL, (1,), generator=g)), int(torch.randint(0, Hq, (1,), generator=g)),
              int(torch.randint(0, d, (1,), generator=g))] = -2e5
    return dataclasses.replace(p, q=q.to(torch.bfloat16).contiguous())


@pytest.mark.parametrize("form", ["decode", "verify", "wide_verify", "other_group"])
def test_fp8_any_q_magnitude(form):
    shape = {"decode": (32, 8, [40, 700, 2100], 1), "verify": (32, 8, [9, 300, 2100], 9),
             "wide_verify": (32, 4, [9, 300, 2100], 9), "other_group": (40, 8, [33, 700], 1)}[form]
    Hq, Hkv, lens, q_len = shape
    p = W.make_problem(lens, Hq, Hkv, 128, q_len=q_len, seed=990, device="cuda", kv_dtype=W.KV_FP8_E4M3)
    q = _extreme_q(p, seed=991)
    _clean_errors()
    out = _run(q)
    assert pa.check_device_errors() == pa.PA_OK
    assert torch.isfinite(out.float()).all()
    _assert_parity(q, out)


def test_fp8_prefill_any_q_magnitude():
    v = W.make_varlen_problem([0, 300, 1000], [70, 9, 33], 16, 2, 128, seed=992, kv_dtype=W.KV_FP8_E4M3)
    q = v.q.clone().float()
    q[3] *= 1e5
    q[80, 5] *= 1e-30
    q[100, 7, 11] = -2e5
    v = dataclasses.replace(v, q=q.to(torch.bfloat16).contiguous())
    g = v.to("cuda")
    out = pa.prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.context_lens, g.query_start_loc, g.scale,
                     k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    assert torch.isfinite(out.float()).all()
    _check(out, oracle.attention_varlen_problem(v), True)


def test_wide_verify_context_shorter_than_q_len_is_flagged():
    # 72 rows per kv head with a 3-token context: rows 0-5 of that sequence see nothing (zeros,
    # flagged), the others are ordinary; an empty context gives zeros too
    p = W.make_problem([3, 0, 400], 32, 4, 128, q_len=9, seed=976, device="cuda")
    _clean_errors()
    out = _run(p)
    assert pa.check_device_errors() == pa.PA_ERR_DEVICE_BOUNDS
    assert torch.all(out[0, :6] == 0) and torch.all(out[1] == 0)
    _assert_parity(p, out)


def test_wide_tree_verify_matches_oracle_and_chain_is_verify():
    p = W.make_problem([9, 300, 2100], 32, 4, 128, q_len=9, seed=975, device="cuda", tail_fill="nan")
    masks = W.random_tree_masks(3, 9, seed=5).to("cuda")
    _clean_errors()
    out = pa.tree_verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, masks, p.scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    ref = oracle.attention_problem(p, tree_mask=masks)
    _check(out, ref, False)
    chain = pa.tree_verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                           W.chain_mask(3, 9, device="cuda"), p.scale)
    torch.cuda.synchronize()
    assert torch.equal(_run(p).view(torch.int16), chain.view(torch.int16))


TREE_SHAPES = [
    # Hq, Hkv, d, lens, q_len
    (32, 8, 128, [9, 64, 700, 2100], 9),
    (32, 8, 128, [16, 33, 1029], 16),
    (8, 2, 64, [5, 40, 515], 5),
    (16, 4, 128, [3, 77, 300], 3),
]


@pytest.mark.parametrize("shape", TREE_SHAPES)
def test_tree_verify_matches_oracle(shape):
    Hq, Hkv, d, lens, q_len = shape
    p = W.make_problem(lens, Hq, Hkv, d, q_len=q_len, seed=950 + q_len, device="cuda", tail_fill="nan")
    masks = W.random_tree_masks(len(lens), q_len, seed=q_len).to("cuda")
    _clean_errors()
    out = pa.tree_verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, masks, p.scale)
    torch.cuda.synchronize()
    ref = oracle.attention_problem(p, tree_mask=masks)
    _check(out, ref, False)


def test_tree_verify_fp8_matches_oracle():
    p = W.make_problem([9, 64, 700, 2100], 32, 8, 128, q_len=9, seed=958, device="cuda",
                       kv_dtype=W.KV_FP8_E4M3, tail_fill="nan")
    masks = W.random_tree_masks(4, 9, seed=3).to("cuda")
    _clean_errors()
    out = pa.tree_verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens, masks, p.scale,
                         k_scale=p.k_scale, v_scale=p.v_scale)
    torch.cuda.synchronize()
    assert pa.check_device_errors() == pa.PA_OK
    ref = oracle.attention_problem(p, tree_mask=masks)
    _check(out, ref, True)


def test_chain_tree_equals_verify_bitwise():
    p = W.make_problem([40, 700, 2100], 32, 8, 128, q_len=9, seed=960, device="cuda")
    ver = _run(p)
    chain = pa.tree_verify(p.q, p.k_cache, p.v_cache, p.block_table, p.context_lens,
                           W.chain_mask(3, 9, device="cuda"), p.scale)
    torch.cuda.synchronize()
    assert torch.equal(ver.view(torch.int16), chain.view(torch.int16))
