"""Pins for the speculative-acceptance oracle (no GPU): the pages' worked numbers (20 % and 2/3
acceptance, the 75 % / 25 % residual, 7 tokens from 2 rounds at K = 3), the distribution
identity min(p, q) + max(0, p - q) = p, the expected tokens per round (1 - a^(g+1)) / (1 - a),
and greedy decoding as argmax matching."""

import numpy as np
import pytest

from oracle import spec_accept as SA
from paged_kv_gqa_attn_gb300 import accounting as A

U_GRID = (np.arange(4096, dtype=np.float64) + 0.5) / 4096          # uniforms in (0, 1)
WORDS = (np.arange(4096, dtype=np.uint64) << np.uint64(20)) + np.uint64(1 << 19)  # 32-bit words


def _accept_fraction(p_x, q_x):
    p = np.array([[p_x, 1 - p_x], [0.5, 0.5]], np.float32)
    q = np.array([[q_x, 1 - q_x]], np.float32)
    acc = [SA.accept_round(p, q, [0], [u], 0)[0] == 1 for u in U_GRID]
    return float(np.mean(acc))


def test_acceptance_probability_examples():
    # studybook 10.6.2: "Machine" q 0.6, p 0.8 -> always; "today" q 0.5, p 0.1 -> 20 %
    assert _accept_fraction(0.8, 0.6) == 1.0
    assert abs(_accept_fraction(0.1, 0.5) - 0.2) <= 1 / 4096
    # sirzzang: "States" drafted with q 0.6, target 0.4 -> 2/3
    assert abs(_accept_fraction(0.4, 0.6) - 2 / 3) <= 1 / 4096


def test_residual_example_75_25():
    # studybook table 10.6.2: residual mass 0.4 split 0.3 / 0.1 -> 75 % / 25 %; the over-drafted
    # token (p 0.1 < q 0.5) leaves the candidates
    p = np.array([[0.1, 0.6, 0.3], [1 / 3, 1 / 3, 1 / 3]], np.float32)
    q = np.array([[0.5, 0.3, 0.2]], np.float32)
    toks = [SA.accept_round(p, q, [0], [0.99], int(w))[1][-1] for w in WORDS]
    freq = np.bincount(toks, minlength=3) / len(toks)
    assert freq[0] == 0.0
    assert abs(freq[1] - 0.75) <= 2 / 4096 and abs(freq[2] - 0.25) <= 2 / 4096


def test_fixed_point_draw():
    w = np.array([1, 0, 3], np.uint64)
    toks = [SA.draw(w, int(x)) for x in WORDS]
    freq = np.bincount(toks, minlength=3) / len(toks)
    assert np.allclose(freq, [0.25, 0.0, 0.75])
    assert SA.draw(w, 0) == 0 and SA.draw(w, 0xFFFFFFFF) == 2
    assert SA.draw(np.zeros(4, np.uint64), 123) == -1
    assert SA.draw(np.array([0, 0, 5], np.uint64), 0) == 2  # zero weights are never drawn
    assert np.array_equal(SA.fixed_weights(np.float32([0.5, -1.0, 2.0, 2.0 ** -41])),
                          np.array([2 ** 39, 0, 2 ** 40, 0], np.uint64))


def _emission_distribution(p, q):
    """Exact (on the uniform grids) distribution of the token a one-draft round emits first."""
    V = len(p)
    P = np.stack([p, np.full(V, 1.0 / V)]).astype(np.float32)
    Q = q[None].astype(np.float32)
    out = np.zeros(V)
    for x in range(V):
        if q[x] == 0:
            continue
        acc = np.mean([SA.accept_round(P, Q, [x], [u], 0)[0] == 1 for u in U_GRID])
        out[x] += q[x] * acc
        if acc < 1:
            toks = [SA.accept_round(P, Q, [x], [0.999999], int(w))[1][0] for w in WORDS[::4]]
            out += q[x] * (1 - acc) * np.bincount(toks, minlength=V) / len(toks)
    return out


def test_emitted_token_follows_the_target_distribution():
    # servingai 5.3.10: accepted path min(p, q) plus rejected path max(0, p - q) sums to p
    rng = np.random.default_rng(5)
    for _ in range(3):
        p = rng.dirichlet(np.ones(6)).astype(np.float32)
        q = rng.dirichlet(np.ones(6)).astype(np.float32)
        got = _emission_distribution(p.astype(np.float64), q.astype(np.float64))
        assert np.abs(got - p).max() <= 3e-3, (got, p)


def test_emitted_distribution_monte_carlo_multi_position():
    # the first emitted token of a K = 3 round is distributed as p_1 (draws from q, random uniforms)
    rng = np.random.default_rng(6)
    V, K, N = 5, 3, 20000
    p = rng.dirichlet(np.ones(V), size=K + 1).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=K).astype(np.float32)
    first = np.zeros(V)
    for _ in range(N):
        draft = [rng.choice(V, p=q[i] / q[i].sum()) for i in range(K)]
        n, toks = SA.accept_round(p, q, draft, rng.random(K).astype(np.float32), int(rng.integers(0, 2 ** 32)))
        first[toks[0]] += 1
    first /= N
    sigma = np.sqrt(p[0] * (1 - p[0]) / N)
    assert np.all(np.abs(first - p[0]) <= 5 * sigma + 1e-3), (first, p[0])


def test_two_rounds_k3_example():
    # sirzzang: K = 3; the first speculation step accepts 2 and rejects the 3rd (3 tokens), the
    # second accepts all 3 plus the bonus (4 tokens): 7 tokens from 2 target forwards, acceptance rate 5/6
    V = 4
    p = np.full((4, V), 0.25, np.float32)
    q = np.full((3, V), 0.25, np.float32)
    p1 = p.copy()
    p1[2] = [0.0, 0.5, 0.5, 0.0]  # drafted token 0 at position 3 has p = 0 < q: rejected
    n1, t1 = SA.accept_round(p1, q, [0, 1, 0], [0.5, 0.5, 0.5], 7)
    n2, t2 = SA.accept_round(p, q, [3, 2, 1], [0.5, 0.5, 0.5], 7)
    assert (n1, len(t1)) == (2, 3) and t1[:2] == [0, 1] and t1[2] in (1, 2)
    assert (n2, len(t2)) == (3, 4) and t2[:3] == [3, 2, 1]
    assert len(t1) + len(t2) == 7 and (n1 + n2) / 6 == 5 / 6


@pytest.mark.parametrize("alpha,gamma,expected", [(0.8, 4, 3.36), (0.5, 8, 1.996), (0.9, 4, 4.095)])
def test_expected_tokens_per_round(alpha, gamma, expected):
    # servingai 5.3.11-12: with each draft accepted independently with probability alpha,
    # E[tokens per target forward] = (1 - alpha^(gamma+1)) / (1 - alpha); 3.36 at 0.8 / 4
    assert abs(A.spec_tokens_per_forward(alpha, gamma) - expected) < 6e-3
    rng = np.random.default_rng(7)
    V, N = 4, 20000
    q = np.full((gamma, V), 0.25, np.float32)
    p = np.full((gamma + 1, V), 0.25, np.float32)
    p[:gamma, 0] = np.float32(0.25 * alpha)  # drafted token 0 at every position: p/q = alpha
    p[:gamma, 1] = np.float32(0.25 + 0.25 * (1 - alpha))
    total = 0
    for _ in range(N):
        n, toks = SA.accept_round(p, q, [0] * gamma, rng.random(gamma).astype(np.float32),
                                  int(rng.integers(0, 2 ** 32)))
        total += len(toks)
    mean = total / N
    assert abs(mean - A.spec_tokens_per_forward(alpha, gamma)) <= 5 * 1.6 / np.sqrt(N)


def test_speedup_formula_pins():
    # servingai 5.3.12: alpha 0.8, c 0.1: gamma 3..7 -> 2.27, 2.40, 2.46, 2.47, 2.45; ceiling
    # 1 / (1 - alpha) = 10 at alpha 0.9
    for g, s in zip(range(3, 8), [2.27, 2.40, 2.46, 2.47, 2.45]):
        assert abs(A.spec_speedup(0.8, g, 0.1) - s) < 6e-3
    assert abs(A.spec_tokens_per_forward(0.9, 400) - 10.0) < 1e-9
    assert A.spec_tokens_per_forward(1.0, 4) == 5


def test_greedy_is_argmax_matching():
    # sirzzang: at temperature 0 the rule reduces to "accept iff the draft is the target argmax"
    rng = np.random.default_rng(8)
    V, K = 10, 6
    for trial in range(50):
        tgt = rng.integers(0, V, size=K + 1)
        draft = tgt[:K].copy()
        m = rng.integers(0, K + 1)
        if m < K:
            draft[m] = (tgt[m] + 1 + rng.integers(0, V - 1)) % V
        p = np.eye(V, dtype=np.float32)[tgt]
        q = np.eye(V, dtype=np.float32)[draft]
        n, toks = SA.accept_round(p, q, draft, rng.random(K).astype(np.float32), int(rng.integers(0, 2 ** 32)))
        assert n == m
        assert toks == [int(t) for t in draft[:m]] + [int(tgt[m])]


def test_bad_draft_token():
    p = np.full((2, 3), 1 / 3, np.float32)
    q = np.full((1, 3), 1 / 3, np.float32)
    assert SA.accept_round(p, q, [3], [0.5], 0) == (-1, [])
    n, toks = SA.accept_batch(p[None], q[None], np.array([[-1]]), np.array([[0.5]]), np.array([0]))
    assert n[0] == -1 and np.all(toks == -1)


def test_zero_drafts_is_plain_sampling():
    p = np.array([[0.25, 0.0, 0.75]], np.float32)
    toks = [SA.accept_round(p, np.zeros((0, 3), np.float32), [], [], int(w))[1][0] for w in WORDS]
    assert abs(np.mean(np.array(toks) == 2) - 0.75) <= 1 / 4096
