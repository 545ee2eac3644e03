"""Oracle for the speculative acceptance step that follows verify (TEST INFRASTRUCTURE ONLY).

Speculative sampling (studybook fde-roadmap ch.10, section 10.6.2; aegloslab servingai 5.3.10;
sirzzang "Speculative Decoding", the verification algorithm): the draft proposed tokens
x_1..x_K with draft distributions q_1..q_K; the verify forward gave the target distributions
p_1..p_{K+1}.  Going left to right, x_i is accepted with probability min(1, p_i(x_i) / q_i(x_i))
(always when p_i(x_i) >= q_i(x_i)); at the first rejection a replacement is drawn from the
residual norm(max(0, p_i - q_i)) and the round ends; if every draft is accepted a bonus token is
drawn from p_{K+1}.  A round thus emits between 1 and K+1 tokens.

Readings (the pages leave the mechanics of the draws open):
  * the random numbers are inputs: one uniform u_i in [0, 1) (fp32) per draft position, tested
    as "accept iff p >= q or u_i < p / q" with the ratio an IEEE fp32 division; and one 32-bit
    word per round for the draw;
  * a draw from weights r(x) >= 0 (the residual, or p for the bonus) is the inverse CDF in fixed
    point: w(x) = floor(min(r(x), 1) * 2^40) as an unsigned integer, Z = sum of w,
    T = floor(Z * word / 2^32), and the token is the smallest x whose inclusive prefix sum of w
    exceeds T.  Integer sums make the choice exact and independent of summation order; the
    weights lose at most 2^-40 each, a total-variation error below V * 2^-40;
  * r = max(0, p - q) is one fp32 subtraction per entry; if the residual sums to zero (possible
    only through rounding of inputs that do not sum to 1) the draw uses p_i instead; a draft
    token outside [0, V) makes the round emit nothing (count -1).

Plain numpy, one round at a time: slow and obviously correct.
"""

from __future__ import annotations

import numpy as np

FIX_BITS = 40


def fixed_weights(r) -> np.ndarray:
    """floor(min(max(r, 0), 1) * 2^40) as uint64 for an fp32 vector r."""
    r = np.clip(np.asarray(r, dtype=np.float32), 0.0, 1.0).astype(np.float64)
    return np.floor(r * float(2 ** FIX_BITS)).astype(np.uint64)


def draw(w: np.ndarray, word: int) -> int:
    """Inverse-CDF draw from integer weights w with a 32-bit uniform word; -1 if w sums to 0."""
    w = np.asarray(w, dtype=np.uint64)
    prefix = np.cumsum(w, dtype=np.uint64)
    Z = int(prefix[-1]) if len(prefix) else 0
    if Z == 0:
        return -1
    T = (Z * (int(word) & 0xFFFFFFFF)) >> 32
    return int(np.searchsorted(prefix, np.uint64(T), side="right"))


def accept_round(p_rows, q_rows, draft, u_accept, word):
    """One sequence.  p_rows [K+1, V] and q_rows [K, V] fp32, draft [K] ints, u_accept [K] fp32,
    word a 32-bit int.  Returns (number of accepted drafts, emitted tokens list)."""
    p_rows = np.asarray(p_rows, dtype=np.float32)
    q_rows = np.asarray(q_rows, dtype=np.float32)
    K = len(draft)
    V = p_rows.shape[1]
    for i in range(K):
        x = int(draft[i])
        if x < 0 or x >= V:
            return -1, []
    for i in range(K):
        x = int(draft[i])
        p = np.float32(p_rows[i, x])
        q = np.float32(q_rows[i, x])
        if p >= q or np.float32(u_accept[i]) < np.float32(p / q):
            continue
        residual = np.maximum(p_rows[i] - q_rows[i], np.float32(0.0))  # fp32 subtraction
        w = fixed_weights(residual)
        if int(w.sum(dtype=np.uint64)) == 0:
            w = fixed_weights(p_rows[i])
        return i, [int(t) for t in draft[:i]] + [draw(w, word)]
    return K, [int(t) for t in draft] + [draw(fixed_weights(p_rows[K]), word)]


def accept_batch(p, q, draft, u_accept, words):
    """Batch form: p [B, K+1, V], q [B, K, V], draft [B, K], u_accept [B, K], words [B].
    Returns (num_accepted [B] int32, tokens [B, K+1] int32 padded with -1)."""
    p = np.asarray(p, dtype=np.float32)
    q = np.asarray(q, dtype=np.float32)
    draft = np.asarray(draft)
    B, K = draft.shape
    n_acc = np.zeros(B, dtype=np.int32)
    tokens = np.full((B, K + 1), -1, dtype=np.int32)
    for b in range(B):
        n, toks = accept_round(p[b], q[b] if K else np.zeros((0, p.shape[2]), np.float32), draft[b],
                               np.asarray(u_accept)[b] if K else [], int(np.asarray(words)[b]))
        n_acc[b] = n
        tokens[b, :len(toks)] = toks
    return n_acc, tokens
