"""Pins of the oracle's ragged verification: full windows reduce to the rectangular
functions; greedy windows match a numpy restatement of the pages' count of accepted
tokens (leading draft/target matches, masked past each window); every window equals
the rectangular chain run on that request alone (packed rows, padded drafts, draft
probabilities and coins, the final coin at the window's last position); windows that do
not fit are left at accept_length 0."""
import numpy as np

import oracle
from speculative_decoding_verify_temp_gb300 import synth


def _packed(rng, B, D, V, lens):
    qo = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = (rng.standard_normal((int(qo[-1]), V)) * 2).astype(np.float32)
    return qo, x


def test_full_windows_equal_the_rectangular_calls():
    rng = np.random.default_rng(21)
    B, D, V = 7, 3, 300
    R = D + 1
    qo, x = _packed(rng, B, D, V, np.full(B, R))
    am = x.reshape(B, R, V)[:, :D].argmax(-1)
    drafts = np.where(rng.random((B, D)) < 0.7, am, rng.integers(0, V, (B, D))).astype(np.int32)
    g = oracle.verify_chain_greedy(x, D, drafts)
    gr = oracle.verify_chain_greedy_ragged(x, D, qo, drafts)
    for k in ("accepted_tokens", "accept_length", "accept_index"):
        np.testing.assert_array_equal(gr[k], g[k])
    kw = dict(temperature=rng.uniform(0.5, 1.2, B).astype(np.float32),
              top_k=rng.choice([0, 5], B).astype(np.int32), seed=synth.request_seeds(B),
              offset=np.arange(B, dtype=np.int64))
    c = oracle.chain_spec_sampling(x, True, D, drafts, **kw)
    cr = oracle.chain_spec_sampling_ragged(x, True, D, qo, drafts, **kw)
    for k in ("accepted_tokens", "accept_length", "accept_index"):
        np.testing.assert_array_equal(cr[k], c[k])


def test_greedy_windows_count_leading_matches():
    """count_accepted_ragged, restated: the target token of each packed row is its
    argmax; a request accepts 1 + the number of leading positions j < L_b - 1 whose
    draft equals the target token there; its tokens are the target tokens up to that
    count."""
    rng = np.random.default_rng(22)
    B, D, V = 40, 5, 97
    lens = rng.integers(1, D + 2, B)
    qo, x = _packed(rng, B, D, V, lens)
    tgt = x.argmax(1)
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    for b in range(B):  # make long runs of matches common
        n = int(rng.integers(0, lens[b]))
        drafts[b, :n] = tgt[qo[b]:qo[b] + n]
    r = oracle.verify_chain_greedy_ragged(x, D, qo, drafts)
    for b in range(B):
        L = int(lens[b])
        n = 0
        while n < L - 1 and drafts[b, n] == tgt[qo[b] + n]:
            n += 1
        assert r["accept_length"][b] == n + 1
        np.testing.assert_array_equal(r["accepted_tokens"][b, :n + 1], tgt[qo[b]:qo[b] + n + 1])
        assert (r["accepted_tokens"][b, n + 1:] == -1).all()
        np.testing.assert_array_equal(r["accept_index"][b, :n + 1], qo[b] + np.arange(n + 1))
        lse = np.log(np.exp(x[qo[b]:qo[b] + n + 1].astype(np.float64)).sum(1))
        np.testing.assert_allclose(r["logprobs"][b, :n + 1],
                                   x[qo[b] + np.arange(n + 1), tgt[qo[b]:qo[b] + n + 1]] - lse,
                                   rtol=1e-12)


def test_each_window_is_its_own_chain():
    rng = np.random.default_rng(23)
    B, D, V = 24, 4, 200
    R = D + 1
    lens = rng.integers(1, R + 1, B)
    qo, x = _packed(rng, B, D, V, lens)
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    q = rng.random((B * D, V)).astype(np.float32)
    q /= q.sum(1, keepdims=True)
    T = rng.uniform(0.4, 1.3, B).astype(np.float32)
    T[3] = 0.0
    k = rng.choice([0, 3, 30], B).astype(np.int32)
    p = rng.choice([1.0, 0.9], B).astype(np.float32)
    u = rng.uniform(0.01, 0.99, (B, R)).astype(np.float32)
    for use_q in (False, True):
        r = oracle.chain_spec_sampling_ragged(x, True, D, qo, drafts,
                                              draft_probs=q if use_q else None, temperature=T,
                                              top_k=k, top_p=p, uniforms=u)
        for b in range(B):
            L = int(lens[b])
            Db = L - 1
            one = oracle.chain_spec_sampling(
                x[qo[b]:qo[b] + L], True, Db, drafts[b:b + 1, :Db],
                draft_probs=q[b * D:b * D + Db] if (use_q and Db > 0) else None,
                temperature=T[b:b + 1], top_k=k[b:b + 1], top_p=p[b:b + 1],
                uniforms=u[b:b + 1, :L])
            assert r["accept_length"][b] == one["accept_length"][0]
            np.testing.assert_array_equal(r["accepted_tokens"][b, :L], one["accepted_tokens"][0])
            assert (r["accepted_tokens"][b, L:] == -1).all()
            got_idx = r["accept_index"][b, :L]
            want_idx = np.where(one["accept_index"][0] >= 0, one["accept_index"][0] + qo[b], -1)
            np.testing.assert_array_equal(got_idx, want_idx)
            assert r["margin"][b] == one["margin"][0]


def test_philox_coins_follow_the_window():
    """Without explicit coins the final draw of a window of L rows uses position L - 1 of
    the request's stream: the same as the explicit coins verify_coin(seed, offset, j)."""
    rng = np.random.default_rng(24)
    B, D, V = 10, 3, 150
    lens = rng.integers(1, D + 2, B)
    qo, x = _packed(rng, B, D, V, lens)
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    seed, off = synth.request_seeds(B), np.arange(B, dtype=np.int64) + 99
    a = oracle.chain_spec_sampling_ragged(x, True, D, qo, drafts, seed=seed, offset=off)
    u = np.array([[oracle.verify_coin(seed[b], off[b], j) for j in range(D + 1)]
                  for b in range(B)], np.float32)
    b_ = oracle.chain_spec_sampling_ragged(x, True, D, qo, drafts, uniforms=u)
    np.testing.assert_array_equal(a["accepted_tokens"], b_["accepted_tokens"])


def test_windows_that_do_not_fit_are_left_unverified():
    rng = np.random.default_rng(25)
    D, V = 2, 50
    qo = np.array([0, 2, 2, 6, 7], np.int32)  # lengths 2, 0, 4 (> D + 1), 1
    x = (rng.standard_normal((7, V))).astype(np.float32)
    drafts = rng.integers(0, V, (4, D)).astype(np.int32)
    r = oracle.verify_chain_greedy_ragged(x, D, qo, drafts)
    assert r["accept_length"][1] == 0 and r["accept_length"][2] == 0
    assert (r["accepted_tokens"][[1, 2]] == -1).all()
    assert r["accept_length"][0] >= 1 and r["accept_length"][3] == 1
    c = oracle.chain_spec_sampling_ragged(x, True, D, qo, drafts, seed=synth.request_seeds(4),
                                          offset=np.arange(4))
    assert c["accept_length"][1] == 0 and c["accept_length"][2] == 0
