"""Pins of the oracle's single-step sampler, joint filter order, min_p and relaxed
acceptance against definitions written out independently here: exact rational brute
force on dyadic probability rows, closed-form worked cases, reductions to the greedy
routine and the plain chain, and the inverse-CDF law on a grid of coins."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from speculative_decoding_verify_temp_gb300 import synth


def _order(vals):
    """Token ids in (value descending, id ascending) order."""
    return sorted(range(len(vals)), key=lambda i: (-vals[i], i))


def _kept_brute(vals, k, p, min_p, joint):
    """The kept set of a probability row, by definition, in exact rationals: the top-k
    prefix; the nucleus (rank r kept iff r == 0 or the mass before it is below top_p
    times the reference mass: the top-k mass, or the whole row's when joint), cut
    within the top-k prefix; then, of those, the tokens whose weight is at least min_p
    times the largest (the argmax always stays)."""
    w = [Fraction(float(v)) for v in vals]
    order = _order(vals)
    V = len(vals)
    nk = k if 0 < k < V else V
    topk = order[:nk]
    zref = sum(w[i] for i in (order if joint else topk))
    kept = topk
    if p < 1.0:
        P = Fraction(float(np.float32(p))) * zref
        out, S = [], Fraction(0)
        for r, i in enumerate(topk):
            if r == 0 or S < P:
                out.append(i)
                S += w[i]
            else:
                break
        kept = out
    if min_p > 0.0:
        mp = min(Fraction(float(np.float32(min_p))), Fraction(1))
        w0 = w[kept[0]]
        kept = [kept[0]] + [i for i in kept[1:] if w[i] >= mp * w0]
    return kept


def _dyadic_rows(rng, n, V):
    """Probability rows of multiples of 2^-12 (fp64 sums of them are exact), with ties."""
    rows = []
    for _ in range(n):
        c = rng.integers(0, 9, V).astype(np.float64)
        c[rng.integers(0, V)] += 1  # at least one nonzero
        rows.append((c / 4096.0).astype(np.float32))
    return rows


@pytest.mark.parametrize("joint", [False, True])
def test_filter_brute_force_all_knobs(joint):
    rng = np.random.default_rng(5 + joint)
    for vals in _dyadic_rows(rng, 60, 9):
        for k in (0, 1, 2, 4, 9):
            for p in (1.0, 0.95, 0.5, 0.3, 0.05):
                for mp in (0.0, 0.3, 0.5, 1.0):
                    got, _ = oracle.filter_row(vals, False, 1.0, k, p, min_p=mp, joint=joint)
                    kept = _kept_brute(vals, k, p, mp, joint)
                    z = sum(Fraction(float(vals[i])) for i in kept)
                    want = np.zeros(len(vals))
                    for i in kept:
                        want[i] = float(Fraction(float(vals[i])) / z)
                    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0,
                                               err_msg=f"k={k} p={p} mp={mp} {vals}")


def test_joint_worked_case():
    """p = (0.4, 0.35, 0.25), top_k = 2, top_p = 0.5. Top-k first: p' = (8/15, 7/15), and
    the first token's 8/15 already reaches 0.5: only token 0. Joint: the nucleus of p is
    {0, 1} (0.4 < 0.5, then 0.75), inside the top 2: tokens 0 and 1 at 8/15 and 7/15."""
    vals = np.array([0.4, 0.35, 0.25], np.float32)
    seq, _ = oracle.filter_row(vals, False, 1.0, 2, 0.5)
    jnt, _ = oracle.filter_row(vals, False, 1.0, 2, 0.5, joint=True)
    np.testing.assert_array_equal(seq, [1.0, 0.0, 0.0])
    w0, w1 = float(np.float32(0.4)), float(np.float32(0.35))
    np.testing.assert_allclose(jnt, [w0 / (w0 + w1), w1 / (w0 + w1), 0.0], rtol=1e-15)


def test_joint_properties_on_logits():
    """Joint keeps a superset of top-k-first, and equals it when only one knob is on."""
    rng = np.random.default_rng(11)
    for _ in range(40):
        V = int(rng.integers(2, 300))
        x = (rng.standard_normal(V) * 2).astype(np.float32)
        T = float(rng.uniform(0.3, 1.5))
        k = int(rng.choice([0, 1, 5, 50, V]))
        p = float(rng.choice([1.0, 0.95, 0.8, 0.3]))
        s, _ = oracle.filter_row(x, True, T, k, p)
        j, _ = oracle.filter_row(x, True, T, k, p, joint=True)
        assert set(np.flatnonzero(s)) <= set(np.flatnonzero(j))
        if k in (0, V) or p >= 1.0:
            np.testing.assert_array_equal(s, j)


def test_min_p_on_logits_is_a_log_ratio_threshold():
    """On logits, min_p keeps (of the top-k/top-p set) the tokens with
    (l - M) / T >= ln(min_p); the decisions off the reported margin agree with that
    test done here in numpy fp64."""
    rng = np.random.default_rng(12)
    for _ in range(60):
        V = int(rng.integers(2, 500))
        x = (rng.standard_normal(V) * 3).astype(np.float32)
        T = float(rng.uniform(0.3, 1.5))
        mp = float(rng.choice([0.01, 0.1, 0.5, 0.9]))
        got, marg = oracle.filter_row(x, True, T, 0, 1.0, min_p=mp)
        d = (x.astype(np.float64) - x.max()) / T
        want = d >= np.log(np.float32(mp))
        if marg > 1e-9:
            np.testing.assert_array_equal(got > 0, want)
        np.testing.assert_allclose(got[want].sum(), 1.0, rtol=1e-12)


def test_sample_inverse_cdf_on_a_coin_grid():
    """With coins (m + 1/2) / Mc, m < Mc, the inverse CDF in token-id order hands token i
    the coins inside its CDF interval: count_i = Mc * p_i within 1."""
    rng = np.random.default_rng(13)
    V, Mc = 40, 4000
    x = (rng.standard_normal(V) * 1.5).astype(np.float32)
    for k, p, mp, joint in [(0, 1.0, 0.0, False), (10, 0.9, 0.0, True), (10, 0.9, 0.0, False),
                            (0, 0.7, 0.05, False)]:
        p_kept, _ = oracle.filter_row(x, True, 0.8, k, p, min_p=mp, joint=joint)
        u = ((np.arange(Mc) + 0.5) / Mc).astype(np.float32)
        r = oracle.sample_from_logits(np.repeat(x[None], Mc, 0), 1,
                                      temperature=np.full(Mc, 0.8, np.float32),
                                      top_k=np.full(Mc, k, np.int32),
                                      top_p=np.full(Mc, p, np.float32),
                                      min_p=np.full(Mc, mp, np.float32), joint=joint, uniforms=u)
        cnt = np.bincount(r["tokens"], minlength=V)
        assert np.abs(cnt - Mc * p_kept).max() <= 1.0 + 1e-9
        assert (cnt[p_kept == 0] == 0).all()


def test_sample_coins_come_from_the_requests_stream():
    """Row j of request b draws with coin j of the request's verify stream; greedy rows
    take the argmax; logprobs are the temperature-1 log-softmax of the token."""
    rng = np.random.default_rng(14)
    B, n, V = 5, 3, 257
    x = (rng.standard_normal((B * n, V)) * 2).astype(np.float32)
    T = rng.uniform(0.5, 1.2, B * n).astype(np.float32)
    T[4] = 0.0
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64) * 7 + (1 << 40)
    k = rng.choice([0, 5, 50], B * n).astype(np.int32)
    p = rng.choice([1.0, 0.9], B * n).astype(np.float32)
    a = oracle.sample_from_logits(x, n, temperature=T, top_k=k, top_p=p, joint=True, seed=seed,
                                  offset=off)
    u = np.array([oracle.verify_coin(seed[r // n], off[r // n], r % n) for r in range(B * n)],
                 np.float32)
    b = oracle.sample_from_logits(x, n, temperature=T, top_k=k, top_p=p, joint=True, uniforms=u)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    assert a["tokens"][4] == int(np.argmax(x[4]))
    xd = x.astype(np.float64)
    lse = xd.max(1) + np.log(np.exp(xd - xd.max(1, keepdims=True)).sum(1))
    np.testing.assert_allclose(a["logprobs"], xd[np.arange(B * n), a["tokens"]] - lse, rtol=1e-12)


def test_sample_probs_output_is_the_kept_distribution():
    rng = np.random.default_rng(15)
    x = (rng.standard_normal((6, 120)) * 2).astype(np.float32)
    r = oracle.sample_from_logits(x, 2, temperature=np.full(6, 0.9, np.float32),
                                  top_k=np.array([0, 3, 10, 0, 120, 7], np.int32),
                                  top_p=np.array([0.9, 1.0, 0.5, 1.0, 0.99, 0.8], np.float32),
                                  min_p=np.array([0.0, 0.0, 0.0, 0.2, 0.0, 0.1], np.float32),
                                  seed=synth.request_seeds(3), offset=np.arange(3), probs=True)
    pr = r["probs"]
    np.testing.assert_allclose(pr.sum(1), 1.0, rtol=1e-12)
    assert (pr[np.arange(6), r["tokens"]] > 0).all()
    # kept probabilities keep the ratios of the temperature weights
    for i in range(6):
        kept = np.flatnonzero(pr[i])
        w = np.exp((x[i, kept].astype(np.float64) - x[i].max()) / float(np.float32(0.9)))
        np.testing.assert_allclose(pr[i, kept], w / w.sum(), rtol=1e-12)


def test_relaxed_thresholds_of_one_are_plain_rejection_sampling():
    d = synth.tiny_verify()
    kw = dict(temperature=np.full(d["B"], 0.9, np.float32), seed=synth.request_seeds(d["B"]),
              offset=np.arange(d["B"]))
    a = oracle.chain_spec_sampling(d["logits"], True, d["D"], d["draft_tokens"], **kw)
    b = oracle.chain_spec_sampling(d["logits"], True, d["D"], d["draft_tokens"], **kw,
                                   threshold_single=1.0, threshold_acc=1.0, min_p=np.zeros(d["B"]))
    for key in ("accepted_tokens", "accept_length", "accept_index"):
        np.testing.assert_array_equal(a[key], b[key])


def test_relaxed_acceptance_rate_on_a_coin_grid():
    """D = 1, target-only: over coins (m + 1/2) / Mc the draft is accepted for
    Mc * min(1, p(x) / threshold_acc) of them (all of them if p(x) >= threshold_single)."""
    rng = np.random.default_rng(16)
    V, Mc = 30, 2000
    row = (rng.standard_normal(V) * 1.2).astype(np.float32)
    x = np.repeat(np.stack([row, row])[None], Mc, 0).reshape(Mc * 2, V)
    p_row, _ = oracle.filter_row(row, True, 1.0)
    order = np.argsort(-p_row)
    u = np.stack([(np.arange(Mc) + 0.5) / Mc, np.full(Mc, 0.5)], 1).astype(np.float32)
    for tok in (order[0], order[3]):
        for ts, ta in [(1.0, 1.0), (1.0, 0.5), (1.0, 0.2), (0.05, 1.0)]:
            r = oracle.chain_spec_sampling(x, True, 1, np.full((Mc, 1), tok, np.int32),
                                           uniforms=u, threshold_single=ts, threshold_acc=ta)
            acc = (r["accept_length"] == 2).sum()
            px = p_row[tok]
            want = Mc if px >= ts else np.sum(u[:, 0].astype(np.float64) * ta < px)
            assert acc == want
            assert abs(want - (Mc if px >= ts else Mc * min(1.0, px / ta))) <= 1.0


def test_min_p_one_makes_the_chain_greedy():
    """min_p = 1 keeps only the maximum-valued tokens: with distinct logits p'' is the
    one-hot argmax, so target-only chain sampling reduces to greedy verification."""
    d = synth.greedy_verify(B=12, D=3, V=500)
    x = synth.f32_from_bf16_bits(d["logits_bits"])
    # make every row's maximum unique
    am = x.argmax(1)
    x[np.arange(x.shape[0]), am] += 1.0
    g = oracle.verify_chain_greedy(x, 3, d["draft_tokens"])
    c = oracle.chain_spec_sampling(x, True, 3, d["draft_tokens"],
                                   temperature=np.full(12, 0.7, np.float32),
                                   min_p=np.ones(12, np.float32), seed=synth.request_seeds(12),
                                   offset=np.arange(12))
    np.testing.assert_array_equal(c["accept_length"], g["accept_length"])
    np.testing.assert_array_equal(c["accepted_tokens"], g["accepted_tokens"])


def test_relaxed_thresholds_do_not_apply_with_draft_probs():
    d = synth.tiny_verify()
    q = d["draft_probs"]
    kw = dict(draft_probs=q, seed=synth.request_seeds(d["B"]), offset=np.arange(d["B"]))
    a = oracle.chain_spec_sampling(d["logits"], True, d["D"], d["draft_tokens"], **kw)
    b = oracle.chain_spec_sampling(d["logits"], True, d["D"], d["draft_tokens"], **kw,
                                   threshold_single=0.1, threshold_acc=0.1)
    np.testing.assert_array_equal(a["accept_length"], b["accept_length"])
