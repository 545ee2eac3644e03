"""Byte and block accounting for paged attention (measurement helpers, no attention arithmetic).

The decode step is bound by HBM bandwidth: each step reads every cached Key/Value byte once
(aegloslab servingai 5.3.1; studybook fde-roadmap ch.10 section 10.2.3).  The algorithmic
traffic of one attention call is therefore the KV bytes of the visible tokens, plus the fp8
scales, plus Q read and O written; block tables and lengths are excluded (far below 0.1 %).
"""

from __future__ import annotations

import math
from typing import Iterable


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elt_bytes: float) -> float:
    """K and V bytes one token adds to the cache across all layers (servingai 5.3.6)."""
    return 2.0 * num_layers * num_kv_heads * head_dim * elt_bytes


def blocks_needed(context_len: int, block_size: int) -> int:
    """Blocks a sequence occupies when blocks are handed out one at a time as it grows."""
    return (int(context_len) + block_size - 1) // block_size


def block_usage(context_lens: Iterable[int], block_size: int):
    """(blocks, slots, wasted slots) for a set of sequences (studybook section 10.12.2)."""
    lens = list(context_lens)
    blocks = sum(blocks_needed(L, block_size) for L in lens)
    slots = blocks * block_size
    return blocks, slots, slots - sum(lens)


def decode_step_time(weight_bytes: float, batch: int, kv_bytes_per_request: float,
                     bandwidth: float) -> float:
    """Bandwidth-bound decode step time (W + B*K) / BW (servingai 5.3.1)."""
    return (weight_bytes + batch * kv_bytes_per_request) / bandwidth


def decode_throughput(weight_bytes: float, batch: int, kv_bytes_per_request: float,
                      bandwidth: float) -> float:
    """Tokens per second B / t_step; tends to BW / K as B grows (servingai 5.3.1)."""
    return batch / decode_step_time(weight_bytes, batch, kv_bytes_per_request, bandwidth)


def attention_bytes(context_lens: Iterable[int], q_len: int, num_q_heads: int, num_kv_heads: int,
                    head_dim: int, block_size: int, kv_elt_bytes: float, fp8_scales: bool,
                    q_elt_bytes: int = 2, out_elt_bytes: int = 2) -> int:
    """Algorithmic bytes of one paged-attention call (every visible K/V row read once)."""
    lens = [int(L) for L in context_lens]
    B = len(lens)
    tokens = sum(lens)
    kv = 2 * tokens * num_kv_heads * head_dim * kv_elt_bytes
    scales = 0
    if fp8_scales:
        pages = sum(blocks_needed(L, block_size) for L in lens)
        scales = 2 * pages * num_kv_heads * 4
    qo = B * q_len * num_q_heads * head_dim * (q_elt_bytes + out_elt_bytes)
    return int(math.ceil(kv + scales + qo))


def attention_flops(context_lens: Iterable[int], q_len: int, num_q_heads: int, head_dim: int) -> int:
    """Useful multiply-add flops (2 per FMA) of scores and value sums under the causal mask."""
    total = 0
    for L in context_lens:
        L = int(L)
        for i in range(q_len):
            n = max(L - q_len + i + 1, 0)
            total += 2 * 2 * n * head_dim * num_q_heads
    return total


def spec_tokens_per_forward(alpha: float, gamma: int) -> float:
    """Expected tokens settled per target forward when each of gamma drafts is accepted
    independently with probability alpha: the accepted run plus the one token the target always
    adds, (1 - alpha^(gamma+1)) / (1 - alpha) (servingai 5.3.11); gamma + 1 at alpha = 1."""
    if alpha >= 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def spec_speedup(alpha: float, gamma: int, c: float) -> float:
    """Speed-up over plain decode when one draft forward costs c target forwards: a round costs
    1 + gamma * c target forwards (servingai 5.3.11-12)."""
    return spec_tokens_per_forward(alpha, gamma) / (1.0 + gamma * c)
