"""Oracle for appending new tokens' K/V to the paged cache (TEST INFRASTRUCTURE ONLY).

The decode step computes the new token's K and V and stores them in the cache for the next
steps (studybook fde-roadmap ch.10, section 10.2.2 and 10.3.2); with a paged cache the slot is
found through the block table, a block being handed out when the previous one is full
(section 10.12.2; aegloslab servingai 5.3.7).  For the verify form the q_len new tokens are
appended together.

Readings (the pages say nothing on these):
  * context_lens counts the new tokens: sequence b's n_new new tokens take positions
    [L_b - n_new, L_b), slot j % bs of physical block block_table[b][j // bs];
  * bf16 caches store the new rows unchanged;
  * fp8 caches keep one scale per (physical block, kv head) equal to amax / 448 over the
    block's valid tokens (1 when amax is 0), symmetric scale quantisation (section 10.8.2).  An
    append recomputes amax over the old tokens of the block (decoded: e4m3 * old scale, an fp32
    product) and the new ones (bf16 -> fp32); if the scale changes the old tokens are re-encoded
    as round_e4m3(value / new scale), and the new tokens always are.  All of it in fp32 (the
    precision the kernel decides in); e4m3 rounding is to nearest, ties to even, saturating at
    +-448.  Slots past the sequence's last token are left as they were.

Plain numpy, one token and one (block, head) at a time: slow and obviously correct.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(byte: int) -> float:
    """OCP E4M3: (-1)^s 2^(e-7) (1 + m/8) for e > 0, (-1)^s 2^-6 m/8 for e = 0; S.1111.111 = NaN."""
    s = (byte >> 7) & 1
    e = (byte >> 3) & 15
    m = byte & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def e4m3_encode(x: float) -> int:
    """Round x (a finite or NaN fp32 value) to E4M3: nearest, ties to even, saturating at 448."""
    if np.isnan(x):
        return 0x7F
    s = 0x80 if (x < 0 or (x == 0 and np.signbit(x))) else 0
    a = abs(float(x))
    if a >= E4M3_MAX:
        return s | 0x7E
    if a < 2.0 ** -6:  # subnormal range: quantum 2^-9
        q = np.round(a / 2.0 ** -9)  # numpy rounds halves to even; exact (power-of-two scaling)
        if q >= 8:  # rounded up into the smallest normal 2^-6
            return s | (1 << 3)
        return s | int(q)
    e = int(np.floor(np.log2(a)))
    # guard against log2 rounding at exact powers of two
    if 2.0 ** (e + 1) <= a:
        e += 1
    elif 2.0 ** e > a:
        e -= 1
    quantum = 2.0 ** (e - 3)
    q = int(np.round(a / quantum))  # in [8, 16]
    if q == 16:
        e += 1
        q = 8
    if e > 8 or (e == 8 and q > 14):  # above 448 after rounding
        return s | 0x7E
    return s | ((e + 7) << 3) | (q - 8)


def _bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def append_kv(k_new, v_new, k_cache, v_cache, block_table, context_lens, *, n_new, block_size,
              fp8=False, k_scale=None, v_scale=None):
    """Return the caches (and scales) after appending.  Inputs are numpy arrays (or tensors):
    k_new/v_new bf16 bits uint16 [B, n_new, Hkv, d]; caches uint16 (bf16) or uint8 (E4M3)
    [NB, Hkv, bs, d]; scales float32 [NB, Hkv]."""
    import oracle

    kn = oracle._np(k_new, np.uint16)
    vn = oracle._np(v_new, np.uint16)
    kc = oracle._np(k_cache, np.uint8 if fp8 else np.uint16).copy()
    vc = oracle._np(v_cache, np.uint8 if fp8 else np.uint16).copy()
    bt = oracle._np(block_table, np.int32)
    cl = oracle._np(context_lens, np.int32)
    ks = oracle._np(k_scale, np.float32).copy() if fp8 else None
    vs = oracle._np(v_scale, np.float32).copy() if fp8 else None
    B = kn.shape[0]
    Hkv = kn.shape[2]
    for b in range(B):
        L = int(cl[b])
        first = L - n_new
        if first < 0:
            raise ValueError("context shorter than the appended tokens")
        if not fp8:
            for t in range(n_new):
                j = first + t
                pb = int(bt[b, j // block_size])
                kc[pb, :, j % block_size, :] = kn[b, t]
                vc[pb, :, j % block_size, :] = vn[b, t]
            continue
        for blk in range(first // block_size, (L - 1) // block_size + 1):
            pb = int(bt[b, blk])
            lo = blk * block_size
            s_new0 = max(first - lo, 0)           # slots [0, s_new0) hold older tokens
            s_new1 = min(L - lo, block_size)      # slots [s_new0, s_new1) get new tokens
            for cache, scales, new in ((kc, ks, kn), (vc, vs, vn)):
                for g in range(Hkv):
                    old_scale = np.float32(scales[pb, g])
                    old_vals = [[np.float32(e4m3_decode(int(cache[pb, g, sl, c]))) * old_scale
                                 for c in range(cache.shape[3])] for sl in range(s_new0)]
                    new_vals = [_bf16_bits_to_f32(new[b, lo + sl - first, g]) for sl in range(s_new0, s_new1)]
                    amax = np.float32(0.0)
                    for row in old_vals:
                        for v in row:
                            amax = max(amax, np.float32(abs(v)))
                    for row in new_vals:
                        amax = max(amax, np.float32(np.max(np.abs(row))))
                    new_scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
                    if s_new0 > 0 and new_scale != old_scale:
                        for sl, row in enumerate(old_vals):
                            for c, v in enumerate(row):
                                cache[pb, g, sl, c] = e4m3_encode(np.float32(v / new_scale))
                    for k, row in enumerate(new_vals):
                        for c, v in enumerate(row):
                            cache[pb, g, s_new0 + k, c] = e4m3_encode(np.float32(np.float32(v) / new_scale))
                    scales[pb, g] = new_scale
    if fp8:
        return kc, vc, ks, vs
    return kc, vc
