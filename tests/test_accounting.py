"""Pins for the workload generator and the byte accounting against the pages' printed numbers.

Every expected value is read from tests/golden/accounting_pages.txt, which cites the page and
section each number is printed in.
"""

import math
import os

import pytest
import torch

from paged_kv_gqa_attn_gb300 import accounting as A
from paged_kv_gqa_attn_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accounting_pages.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                vals[k] = float(v)
    return vals


G = _golden()
KB, MB, GB, TB = 1024, 1024 ** 2, 1e9, 1e12


def test_kv_bytes_per_token_8b_gqa():
    assert A.kv_bytes_per_token(32, 8, 128, 2) == G["kv_bytes_per_token_8b_gqa"]


def test_reservation_and_use():
    per_tok = A.kv_bytes_per_token(32, 8, 128, 2)
    assert 2048 * per_tok / MB == G["reserve_2048_tokens_mb"]
    assert 300 * per_tok / MB == pytest.approx(G["in_use_300_tokens_mb"], abs=0.05)


def test_block_waste_example():
    blocks, slots, waste = A.block_usage([50, 120, 20], 16)
    assert (blocks, slots, waste) == (G["blocks_50_120_20"], G["slots_50_120_20"], G["waste_50_120_20"])


def test_last_block_waste():
    per_tok = A.kv_bytes_per_token(32, 8, 128, 2)
    worst = max(A.blocks_needed(L, 16) * 16 - L for L in range(1, 5000))
    assert worst == 15
    assert worst * per_tok / MB == pytest.approx(G["last_block_waste_mb"], abs=0.05)


def test_step_time_model():
    Wb, K, BW = 16 * GB, 0.25 * GB, 3.3 * TB
    for B, key in [(1, "step_ms_b1"), (64, "step_ms_b64"), (240, "step_ms_b240")]:
        assert A.decode_step_time(Wb, B, K, BW) * 1e3 == pytest.approx(G[key], abs=0.05)
    ratio = A.decode_throughput(Wb, 64, K, BW) / A.decode_throughput(Wb, 1, K, BW)
    assert math.floor(ratio) == G["throughput_ratio_b64_over_b1"]
    assert BW / K == pytest.approx(G["ceiling_tok_per_s"], rel=1e-9)


def test_attention_bytes_llama8b_decode():
    # 64 sequences x 2048 tokens x 8 kv heads x 128 x (K+V) x 2 B, plus Q and O
    b = A.attention_bytes([2048] * 64, 1, 32, 8, 128, 16, 2, False)
    assert b == 64 * 2048 * 8 * 128 * 2 * 2 + 64 * 32 * 128 * 4
    # one layer's share of the per-request KV of the 8B model: 2048 x 128 KB / 32 layers
    assert (b - 64 * 32 * 128 * 4) / 64 == 2048 * G["kv_bytes_per_token_8b_gqa"] / 32


def test_block_tables_are_valid_permutations():
    for name in ["tiny", "spec_verify_k4"]:
        p = W.make_config(name)
        ids = []
        for b in range(p.num_seqs):
            n = W.blocks_for(int(p.context_lens[b]), 16)
            row = p.block_table[b]
            assert torch.all(row[:n] >= 0) and torch.all(row[:n] < p.num_blocks)
            assert torch.all(row[n:] == -1)
            ids += row[:n].tolist()
        assert len(set(ids)) == len(ids)


def test_config_shapes():
    lens, q_len = W.config_context_lens("cb_mix", W.BASE_SEED + 2)
    assert len(lens) == 256 and q_len == 1
    short = [L for L in lens if L <= 512]
    long = [L for L in lens if L >= 2048]
    assert len(short) == 128 and len(long) == 128
    assert min(short) >= 32 and max(long) <= 8192
    lens, q_len = W.config_context_lens("spec_verify_k8", W.BASE_SEED + 3)
    assert q_len == 9 and all(1024 + 9 <= L <= 4096 + 9 for L in lens)
    table, nb = W.allocate_block_tables(lens, 16, free_fraction=0.1, seed=1)
    need = sum(W.blocks_for(L, 16) for L in lens)
    assert nb == math.ceil(need / 0.9)


def test_fp8_quantizer_scale_is_amax_over_448():
    p = W.make_problem([20, 16], 4, 2, 32, kv_dtype=W.KV_FP8_E4M3, seed=3)
    vals = p.k_cache.view(torch.float8_e4m3fn).float()
    amax_codes = vals.abs().amax(dim=(2, 3))
    used = set(p.block_table[p.block_table >= 0].tolist())
    for blk in used:
        # after scaling by amax/448 the largest magnitude in each tile is exactly 448
        assert torch.all(amax_codes[blk] == 448.0)
