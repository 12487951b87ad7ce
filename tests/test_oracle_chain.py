"""Pins for the oracle's chain verification and sampling (CPU only).

Greedy: hand examples. Rejection sampling: a hand-worked V=2 case, the exact
output distribution of the whole chain enumerated analytically on tiny
vocabularies (chi-square against the oracle's draws over many Philox
streams), the speculative-sampling theorem (every emitted position is
distributed as the target), the acceptance-rate identities sum_x min(p, q),
max_i p_i and sum_i p_i^2, the one-hot special cases, and the output invariants.
"""
import itertools

import numpy as np
import pytest
from scipy import stats


# ---- greedy -------------------------------------------------------------------------

def _onehot_logits(tokens, V, hi=5.0):
    x = np.zeros((len(tokens), V), np.float32)
    for r, t in enumerate(tokens):
        x[r, t] = hi
    return x


def test_greedy_hand_examples(orc):
    V, D = 6, 3
    x = _onehot_logits([2, 4, 1, 5], V)
    r = orc.verify_chain_greedy(x, D, np.array([[2, 4, 1]]))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [2, 4, 1, 5])
    assert r["accept_length"][0] == 4
    np.testing.assert_array_equal(r["accept_index"][0], [0, 1, 2, 3])
    r = orc.verify_chain_greedy(x, D, np.array([[3, 4, 1]]))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [2, -1, -1, -1])
    assert r["accept_length"][0] == 1
    np.testing.assert_array_equal(r["accept_index"][0], [0, -1, -1, -1])
    r = orc.verify_chain_greedy(x, D, np.array([[2, 4, 0]]))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [2, 4, 1, -1])
    # ties resolve to the lowest id: a draft naming the second of two maxima fails
    y = np.zeros((2, 4), np.float32)
    y[0, [1, 3]] = 2.0
    y[1, 0] = 1.0
    r = orc.verify_chain_greedy(y, 1, np.array([[3]]))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [1, -1])
    r = orc.verify_chain_greedy(y, 1, np.array([[1]]))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [1, 0])


def test_greedy_logprob_of_argmax(orc):
    x = np.array([[0.0, 1.0, 3.0], [2.0, 2.0, 0.0]], np.float32)
    r = orc.verify_chain_greedy(x, 1, np.array([[2]]))
    z = np.exp([0.0, 1.0, 3.0])
    assert r["logprobs"][0, 0] == pytest.approx(np.log(z[2] / z.sum()), rel=1e-14)
    # row 1 = (2, 2, 0): the bonus is the lowest argmax, token 0
    assert r["accepted_tokens"][0, 1] == 0
    assert r["logprobs"][0, 1] == pytest.approx(np.log(np.e**2 / (2 * np.e**2 + 1)), rel=1e-14)


def test_greedy_d0_is_argmax(orc):
    x = np.array([[0.0, 4.0, 1.0], [9.0, 0.0, 0.0]], np.float32)
    r = orc.verify_chain_greedy(x, 0, np.zeros((2, 0), np.int32))
    np.testing.assert_array_equal(r["accepted_tokens"][:, 0], [1, 0])
    np.testing.assert_array_equal(r["accept_length"], [1, 1])


# ---- rejection sampling: hand example --------------------------------------------------

def test_rejection_hand_example(orc):
    # V=2, p_0 = (0.25, 0.75), q_0 = (0.5, 0.5), draft x = 0.
    # u_0 = 0.6: 0.6 * 0.5 = 0.3 >= 0.25 -> reject; residual (0, 0.25) -> token 1.
    p = np.array([[0.25, 0.75], [0.9, 0.1]], np.float32)
    q = np.array([[[0.5, 0.5]]], np.float32)
    for uD in (0.01, 0.5, 0.99):
        r = orc.chain_spec_sampling(p, False, 1, np.array([[0]]), draft_probs=q,
                                    uniforms=np.array([[0.6, uD]], np.float32))
        np.testing.assert_array_equal(r["accepted_tokens"][0], [1, -1])
        assert r["accept_length"][0] == 1
    # u_0 = 0.4: 0.2 < 0.25 -> accept; bonus from p_1 = (0.9, 0.1) with u_D
    r = orc.chain_spec_sampling(p, False, 1, np.array([[0]]), draft_probs=q,
                                uniforms=np.array([[0.4, 0.85]], np.float32))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [0, 0])
    r = orc.chain_spec_sampling(p, False, 1, np.array([[0]]), draft_probs=q,
                                uniforms=np.array([[0.4, 0.95]], np.float32))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [0, 1])
    assert r["accept_length"][0] == 2
    assert r["logprobs"][0, 1] == pytest.approx(np.log(float(np.float32(0.1))), rel=1e-12)


def test_target_only_hand_example(orc):
    # target-only: accept iff u < p(x); the residual zeroes x and renormalises
    p = np.array([[0.2, 0.5, 0.3], [0.1, 0.1, 0.8]], np.float32)
    r = orc.chain_spec_sampling(p, False, 1, np.array([[1]]),
                                uniforms=np.array([[0.49, 0.9]], np.float32))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [1, 2])  # bonus: 0.9 > 0.2
    r = orc.chain_spec_sampling(p, False, 1, np.array([[1]]),
                                uniforms=np.array([[0.51, 0.3]], np.float32))
    # residual (0.2, 0, 0.3): t = 0.15 < 0.2 -> token 0
    np.testing.assert_array_equal(r["accepted_tokens"][0], [0, -1])
    r = orc.chain_spec_sampling(p, False, 1, np.array([[1]]),
                                uniforms=np.array([[0.51, 0.5]], np.float32))
    np.testing.assert_array_equal(r["accepted_tokens"][0], [2, -1])  # t = 0.25 >= 0.2


# ---- rejection sampling: exact distributions ----------------------------------------------

def _rand_dist(rng, V):
    x = rng.gamma(0.7, size=V) + 1e-3
    return (x / x.sum()).astype(np.float32)


def _chain_law(p, q):
    """Exact law of the emitted sequence for fixed per-position p_j (j=0..D) and q_j
    (j<D), drafts x_j ~ q_j independently, accept w.p. min(1, p_j(x)/q_j(x))."""
    D = len(q)
    V = len(p[0])
    law = {}

    def resid(j):
        r = np.maximum(p[j] - q[j], 0.0)
        return r / r.sum()

    def rec(j, prefix, prob):
        if j == D:
            for t in range(V):
                law[prefix + (t,)] = law.get(prefix + (t,), 0.0) + prob * p[D][t]
            return
        rj = resid(j)
        rej = 0.0
        for x in range(V):
            a = min(1.0, p[j][x] / q[j][x])
            rec(j + 1, prefix + (x,), prob * q[j][x] * a)
            rej += q[j][x] * (1.0 - a)
        for t in range(V):
            law[prefix + (t,)] = law.get(prefix + (t,), 0.0) + prob * rej * rj[t]

    rec(0, (), 1.0)
    return law


@pytest.mark.parametrize("V,D", [(2, 1), (3, 2), (5, 1), (3, 3)])
def test_rejection_full_chain_law_chi_square(orc, V, D):
    rng = np.random.default_rng(100 * V + D)
    R = D + 1
    p = [_rand_dist(rng, V).astype(np.float64) for _ in range(R)]
    q = [_rand_dist(rng, V).astype(np.float64) for _ in range(D)]
    n = 120000
    drafts = np.stack([rng.choice(V, size=n, p=q[j] / q[j].sum()) for j in range(D)], 1)
    target = np.tile(np.stack(p).astype(np.float32), (n, 1))
    qq = np.tile(np.stack(q).astype(np.float32)[None], (n, 1, 1))
    r = orc.chain_spec_sampling(target, False, D, drafts.astype(np.int32), draft_probs=qq,
                                seed=np.full(n, 77, np.int64),
                                offset=np.arange(n, dtype=np.int64), logprobs=False)
    # invariants
    L = r["accept_length"]
    assert L.min() >= 1 and L.max() <= R
    for b in range(200):
        row = r["accepted_tokens"][b]
        assert (row[L[b]:] == -1).all() and (row[:L[b]] >= 0).all()
        np.testing.assert_array_equal(row[:L[b] - 1], drafts[b, :L[b] - 1])
    # the whole emitted sequence against its exact law
    law = _chain_law(p, q)
    keys = sorted(law)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for b in range(n):
        counts[index[tuple(r["accepted_tokens"][b, :L[b]])]] += 1
    expect = np.array([law[k] for k in keys])
    expect = expect / expect.sum() * n  # the fp32 rows sum to 1 only to rounding
    assert counts[expect == 0].sum() == 0  # nothing outside the law's support
    counts, expect = counts[expect > 0], expect[expect > 0]
    keep = expect > 5
    obs, exp_ = counts[keep], expect[keep]
    if (~keep).any():
        obs, exp_ = np.append(obs, counts[~keep].sum()), np.append(exp_, expect[~keep].sum())
    chi = stats.chisquare(obs, exp_)
    assert chi.pvalue > 1e-4, chi
    # the speculative-sampling theorem: position 0 is distributed as p_0
    first = np.bincount(r["accepted_tokens"][:, 0], minlength=V)
    assert stats.chisquare(first, p[0] / p[0].sum() * n).pvalue > 1e-4


def test_rejection_acceptance_rate_is_sum_min(orc):
    rng = np.random.default_rng(11)
    V, n = 7, 100000
    p = _rand_dist(rng, V).astype(np.float64)
    q = _rand_dist(rng, V).astype(np.float64)
    drafts = rng.choice(V, size=n, p=q / q.sum()).astype(np.int32)[:, None]
    target = np.tile(np.stack([p, p]).astype(np.float32), (n, 1))
    qq = np.tile(q.astype(np.float32)[None, None], (n, 1, 1))
    r = orc.chain_spec_sampling(target, False, 1, drafts, draft_probs=qq,
                                seed=np.full(n, 5, np.int64),
                                offset=np.arange(n, dtype=np.int64), logprobs=False)
    rate = (r["accept_length"] == 2).mean()
    want = np.minimum(p, q).sum()
    assert abs(rate - want) < 4 * np.sqrt(want * (1 - want) / n)


def test_q_equal_p_accepts_everything(orc):
    rng = np.random.default_rng(12)
    V, D, n = 9, 4, 3000
    p = np.stack([_rand_dist(rng, V) for _ in range(D + 1)])
    drafts = np.stack([rng.choice(V, size=n, p=p[j].astype(np.float64) / p[j].astype(np.float64).sum())
                       for j in range(D)], 1).astype(np.int32)
    target = np.tile(p, (n, 1))
    qq = np.tile(p[:D][None], (n, 1, 1))
    r = orc.chain_spec_sampling(target, False, D, drafts, draft_probs=qq,
                                seed=np.full(n, 1, np.int64),
                                offset=np.arange(n, dtype=np.int64))
    assert (r["accept_length"] == D + 1).all()


def test_target_only_acceptance_identities(orc):
    # accept w.p. p(x): argmax drafts accept at rate max p, drafts ~ p at rate sum p^2
    rng = np.random.default_rng(13)
    V, n = 6, 100000
    p = _rand_dist(rng, V)
    p64 = p.astype(np.float64)
    target = np.tile(np.stack([p, p]), (n, 1))
    seeds, offs = np.full(n, 3, np.int64), np.arange(n, dtype=np.int64)
    am = np.full((n, 1), int(np.argmax(p)), np.int32)
    r = orc.chain_spec_sampling(target, False, 1, am, seed=seeds, offset=offs)
    rate = (r["accept_length"] == 2).mean()
    assert abs(rate - p64.max()) < 4 * np.sqrt(p64.max() * (1 - p64.max()) / n)
    d = rng.choice(V, size=n, p=p64 / p64.sum()).astype(np.int32)[:, None]
    r = orc.chain_spec_sampling(target, False, 1, d, seed=seeds, offset=offs)
    rate = (r["accept_length"] == 2).mean()
    want = (p64 ** 2).sum()
    assert abs(rate - want) < 4 * np.sqrt(want * (1 - want) / n)
    # and the first emitted token is distributed as p (residual = p with x removed)
    first = np.bincount(r["accepted_tokens"][:, 0], minlength=V)
    assert stats.chisquare(first, p64 / p64.sum() * n).pvalue > 1e-4


def test_onehot_draft_reduces_to_strict_acceptance(orc):
    # draft probs one-hot at the draft token: accept iff u < p(x), as target-only
    rng = np.random.default_rng(14)
    V, D, n = 5, 2, 4000
    p = np.stack([_rand_dist(rng, V) for _ in range(D + 1)])
    target = np.tile(p, (n, 1))
    drafts = rng.integers(0, V, size=(n, D)).astype(np.int32)
    qq = np.zeros((n, D, V), np.float32)
    for j in range(D):
        qq[np.arange(n), j, drafts[:, j]] = 1.0
    kw = dict(seed=np.full(n, 9, np.int64), offset=np.arange(n, dtype=np.int64))
    a = orc.chain_spec_sampling(target, False, D, drafts, draft_probs=qq, **kw)
    b = orc.chain_spec_sampling(target, False, D, drafts, **kw)
    np.testing.assert_array_equal(a["accepted_tokens"], b["accepted_tokens"])
    np.testing.assert_array_equal(a["accept_length"], b["accept_length"])


def test_delta0_padding_samples_the_target(orc):
    # a padding row drafts token 0 with q = delta_0: acceptance emits 0 w.p. p(0),
    # rejection samples p conditioned on a nonzero token; together they sample p
    rng = np.random.default_rng(15)
    V, n = 6, 100000
    p = _rand_dist(rng, V)
    target = np.tile(np.stack([p, p]), (n, 1))
    qq = np.zeros((n, 1, V), np.float32)
    qq[:, 0, 0] = 1.0
    r = orc.chain_spec_sampling(target, False, 1, np.zeros((n, 1), np.int32),
                                draft_probs=qq, seed=np.full(n, 4, np.int64),
                                offset=np.arange(n, dtype=np.int64))
    first = np.bincount(r["accepted_tokens"][:, 0], minlength=V)
    assert stats.chisquare(first, p.astype(np.float64) / p.astype(np.float64).sum() * n).pvalue > 1e-4


def test_logits_path_equals_probs_path_on_filtered_distribution(orc):
    # with logits + T/k/p the chain works on p'' = filter(logits); feeding p'' as
    # probabilities gives the same decisions away from the boundary
    rng = np.random.default_rng(16)
    V, D, B = 40, 3, 300
    R = D + 1
    x = (rng.standard_normal((B * R, V)) * 2).astype(np.float32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    k = rng.choice([0, 3, 10], B).astype(np.int32)
    tp = rng.choice([1.0, 0.9], B).astype(np.float32)
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    uni = rng.uniform(0.01, 0.99, (B, R)).astype(np.float32)
    a = orc.chain_spec_sampling(x, True, D, drafts, temperature=T, top_k=k, top_p=tp,
                                uniforms=uni, logprobs=False)
    pp = np.zeros((B * R, V), np.float64)
    for r in range(B * R):
        pp[r], _ = orc.filter_row(x[r], True, T=T[r // R], top_k=k[r // R], top_p=tp[r // R])
    b = orc.chain_spec_sampling(pp.astype(np.float32), False, D, drafts, uniforms=uni,
                                logprobs=False)
    ok = a["margin"] > 1e-6
    assert ok.mean() > 0.95
    np.testing.assert_array_equal(a["accepted_tokens"][ok], b["accepted_tokens"][ok])


def test_greedy_temperature_rows_are_strict(orc):
    # T = 0 with logits: p'' is one-hot, so target-only sampling = greedy verify
    rng = np.random.default_rng(17)
    V, D, B = 30, 3, 200
    x = rng.integers(-4, 4, size=(B * (D + 1), V)).astype(np.float32)
    am = x.reshape(B, D + 1, V)[:, :D].argmax(-1).astype(np.int32)
    drafts = np.where(rng.random((B, D)) < 0.7, am, rng.integers(0, V, (B, D))).astype(np.int32)
    g = orc.verify_chain_greedy(x, D, drafts)
    s = orc.chain_spec_sampling(x, True, D, drafts, temperature=np.zeros(B, np.float32),
                                seed=np.arange(B), offset=np.arange(B))
    np.testing.assert_array_equal(g["accepted_tokens"], s["accepted_tokens"])
    np.testing.assert_array_equal(g["accept_length"], s["accept_length"])
    assert np.isinf(s["margin"]).all()


# ---- Gumbel-max -----------------------------------------------------------------------------

def test_gumbel_is_a_temperature_sample(orc):
    rng = np.random.default_rng(18)
    V, n = 12, 60000
    l = (rng.standard_normal(V) * 1.5).astype(np.float32)
    l[3] = -np.inf
    for T in (0.7, 1.0, 1.6):
        x = np.tile(l, (n, 1))
        tok, _ = orc.gumbel_max_sample(x, 1, np.full(n, T, np.float32),
                                       np.full(n, 2024, np.int64), np.arange(n))
        assert (tok != 3).all()
        w = np.exp(l.astype(np.float64) / np.float64(np.float32(T)))
        w[3] = 0.0
        counts = np.bincount(tok, minlength=V)
        keep = w > 0
        assert stats.chisquare(counts[keep], (w / w.sum() * n)[keep]).pvalue > 1e-4


def test_gumbel_greedy_rows_and_rows_within_request(orc):
    x = np.array([[0.0, 5.0, 5.0], [1.0, 0.0, 0.0], [0.0, 0.0, 0.0], [0.0, 1.0, 0.0]],
                 np.float32)
    tok, marg = orc.gumbel_max_sample(x, 2, np.zeros(4, np.float32),
                                      np.array([1, 2]), np.array([0, 1]))
    np.testing.assert_array_equal(tok, [1, 0, 0, 1])
    assert np.isinf(marg).all()
    # rows of one request draw independent noise (row index n in the counter)
    n = 4000
    y = np.zeros((2 * n, 8), np.float32)
    tok, _ = orc.gumbel_max_sample(y, 2, np.ones(2 * n, np.float32),
                                   np.full(n, 5, np.int64), np.arange(n))
    assert (tok[0::2] == tok[1::2]).mean() < 0.2
