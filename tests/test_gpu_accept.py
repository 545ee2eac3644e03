"""GPU parity for speculative acceptance (paged_attn_spec_accept) against the acceptance oracle:
bit-exact accepted counts and emitted tokens on the same seeded distributions and uniforms, from
small ragged vocabularies to the Llama-3 vocabulary at the verify batch sizes; greedy (one-hot)
rounds; the zero-residual fallback; bad draft tokens."""

import numpy as np
import pytest
import torch

import paged_kv_gqa_attn_gb300 as pa
from oracle import spec_accept as SA
from paged_kv_gqa_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _oracle(a):
    return SA.accept_batch(a.p.cpu().numpy(), a.q.cpu().numpy(), a.draft.cpu().numpy(),
                           a.u_accept.cpu().numpy(), a.u_sample.cpu().numpy().view(np.uint32))


def _gpu(a):
    g = a.to("cuda")
    n, t = pa.spec_accept(g.p, g.q, g.draft, g.u_accept, g.u_sample)
    torch.cuda.synchronize()
    return n.cpu().numpy(), t.cpu().numpy()


def _check(a, expect_status=pa.PA_OK):
    n, t = _gpu(a)
    assert pa.check_device_errors() == expect_status
    rn, rt = _oracle(a)
    assert np.array_equal(n, rn), (n, rn)
    assert np.array_equal(t, rt), np.argwhere(t != rt)[:5]
    return n, t


@pytest.mark.parametrize("B,K,V,seed", [
    (4, 3, 1000, 1),
    (7, 5, 4099, 2),        # a ragged last chunk
    (3, 0, 5000, 3),        # no drafts: plain sampling from p
    (5, 31, 300, 4),        # the most drafts
    (6, 4, 8192, 5),        # whole chunks
    (2, 2, 1, 6),           # a one-token vocabulary
    (9, 6, 40000, 7),
])
def test_accept_matches_oracle(B, K, V, seed):
    _check(W.make_accept_problem(B, K, V, seed=seed))


@pytest.mark.parametrize("name", list(W.ACCEPT_CONFIGS))
def test_accept_full_size(name):
    n, t = _check(W.make_accept_config(name))
    K = W.ACCEPT_CONFIGS[name][1]
    assert n.min() >= 0 and n.max() <= K
    assert np.all(t[np.arange(len(n)), n] >= 0)  # every round emits its last token


def test_accept_sweeps_acceptance_rates():
    # a draft close to the target accepts most drafts; a far one few; both bit-exact
    near = W.make_accept_problem(32, 8, 2000, seed=11, draft_noise=0.05)
    far = W.make_accept_problem(32, 8, 2000, seed=12, draft_noise=4.0)
    n_near, _ = _check(near)
    n_far, _ = _check(far)
    assert n_near.mean() > n_far.mean()


def test_accept_all_when_draft_equals_target():
    a = W.make_accept_problem(8, 5, 3000, seed=13)
    a.q = a.p[:, :5].clone()
    n, t = _check(a)
    assert np.all(n == 5)


def test_greedy_rounds_are_argmax_matching():
    rng = np.random.default_rng(14)
    B, K, V = 12, 6, 777
    tgt = rng.integers(0, V, size=(B, K + 1))
    draft = tgt[:, :K].copy()
    m = rng.integers(0, K + 1, size=B)
    for b in range(B):
        if m[b] < K:
            draft[b, m[b]] = (tgt[b, m[b]] + 1) % V
    eye = np.eye(V, dtype=np.float32)
    a = W.AcceptProblem(torch.from_numpy(eye[tgt]), torch.from_numpy(eye[draft]),
                        torch.from_numpy(draft.astype(np.int32)),
                        torch.rand(B, K, generator=torch.Generator().manual_seed(1)),
                        torch.randint(-2 ** 31, 2 ** 31 - 1, (B,), dtype=torch.int32))
    n, t = _check(a)
    assert np.array_equal(n, m)
    for b in range(B):
        assert t[b, m[b]] == tgt[b, m[b]]


def test_zero_residual_falls_back_to_target():
    # p below q everywhere (inputs that do not sum to one): the residual is empty and the draw
    # uses p_i itself
    a = W.make_accept_problem(4, 3, 2048, seed=15)
    a.p = a.p * 0.5
    a.q = torch.maximum(a.q, a.p[:, :3] * 1.5)
    a.u_accept = torch.full_like(a.u_accept, 0.999)
    _check(a)


def test_bad_draft_token_flags_and_empties_the_round():
    a = W.make_accept_problem(3, 4, 1000, seed=16)
    a.draft[1, 2] = 1000
    n, t = _check(a, expect_status=pa.PA_ERR_DEVICE_BOUNDS)
    assert n[1] == -1 and np.all(t[1] == -1)
    assert n[0] >= 0 and n[2] >= 0
