"""Pins for the oracle's decision margins and its logits + draft-probabilities branch
(CPU only).

Every GPU parity test excuses a request whose oracle margin is at most 1e-6, so the
margin itself must be right. Each test here places the deciding quantity a known
distance d from its edge, on inputs whose arithmetic is exact (powers of two, or a
closed form), and checks that the reported margin is that distance, in the units
the definition uses: absolute for the accept test (a probability against a
probability), relative to the total mass for a top-p cut and for the final draw,
and relative to max(1, |best score|) for the Gumbel best-minus-second gap. A cut or
a draw exactly on its edge (d = 0) must report 0, so that it is always excused.

The chain law of the logits + draft-probabilities branch (target logits filtered by
temperature and top-k, rejection against explicit q) is checked against the exact
law of the emitted sequence, enumerated from p = softmax(l / T) computed by numpy.
"""
import math

import numpy as np
import pytest
from scipy import stats

D_SMALL = 2.0 ** -20


def _chain(orc, x, D, drafts, uni, logits=True, **kw):
    x = np.asarray(x, np.float32)
    return orc.chain_spec_sampling(x, logits, D, np.asarray(drafts, np.int32),
                                   uniforms=np.asarray(uni, np.float32), logprobs=False, **kw)


# ---- the accept test --------------------------------------------------------------------

@pytest.mark.parametrize("u,accepted,want", [(0.5 + D_SMALL, False, D_SMALL),
                                             (0.5 - D_SMALL, True, D_SMALL),
                                             (0.5, False, 0.0)])
def test_accept_margin_target_only_is_u_minus_p(orc, u, accepted, want):
    # logits (0, 0) at T = 1: p(0) = 1/2 exactly. On rejection the residual (p with the
    # draft removed) has one token, and the bonus row (0, -inf) is one-hot, so neither
    # draw can flip: the request's margin is the accept test's alone.
    x = [[0.0, 0.0], [0.0, -np.inf]]
    r = _chain(orc, x, 1, [[0]], [[u, 0.3]])
    assert r["margin"][0] == want
    assert list(r["accepted_tokens"][0]) == ([0, 0] if accepted else [1, -1])


@pytest.mark.parametrize("l1,T", [(1.0, 1.0), (-0.75, 0.6), (2.5, 1.3)])
def test_accept_margin_target_only_closed_form(orc, l1, T):
    # two logits: p(0) = 1 / (1 + exp(l1 / T)) (logistic form), coin placed 1e-4 above it
    l1f, Tf = float(np.float32(l1)), float(np.float32(T))
    p0 = 1.0 / (1.0 + math.exp(l1f / Tf))
    u = float(np.float32(p0 + 1e-4))
    r = _chain(orc, [[0.0, l1], [0.0, -np.inf]], 1, [[0]], [[u, 0.3]],
               temperature=np.array([T], np.float32))
    assert r["margin"][0] == pytest.approx(abs(u - p0), rel=1e-9, abs=1e-15)
    assert r["accept_length"][0] == (2 if u < p0 else 1)


@pytest.mark.parametrize("u,accepted", [(0.5 + D_SMALL, False), (0.5 - D_SMALL, True),
                                        (0.5, False)])
def test_accept_margin_with_draft_probs_is_uq_minus_p(orc, u, accepted):
    # four equal logits: p = 1/4 each; q(x) = 1/2 so u q(x) = p(x) at u = 1/2 and the
    # margin is |u q - p| = d / 2 (not |u - p|). The rejection residual max(p - q, 0) =
    # (0, 0, 1/4, 1/4) is drawn with u_D = 1/4 (t = 1/8, halfway inside token 2: draw
    # margin 1/4), and the bonus row is one-hot.
    x = [[0.0, 0.0, 0.0, 0.0], [0.0, -np.inf, -np.inf, -np.inf]]
    q = np.array([[[0.5, 0.5, 0.0, 0.0]]], np.float32)
    r = _chain(orc, x, 1, [[0]], [[u, 0.25]], draft_probs=q)
    assert r["margin"][0] == abs(u - 0.5) / 2
    assert list(r["accepted_tokens"][0]) == ([0, 0] if accepted else [2, -1])


# ---- the top-p cut ---------------------------------------------------------------------

# sorted masses 0.5 (id 2), 0.25 (id 0), 0.125 (id 1), 0.125 (id 3): the mass before
# ranks 1, 2, 3 is 0.5, 0.75, 0.875
P4 = [0.25, 0.125, 0.5, 0.125]


@pytest.mark.parametrize("tp,kept,want", [
    (0.75 - D_SMALL, {0, 2}, D_SMALL),        # rank 2 (mass before 0.75) just dropped
    (0.5 + D_SMALL, {0, 2}, D_SMALL),         # rank 1 (mass before 0.5) just kept
    (0.75 + D_SMALL, {0, 1, 2}, D_SMALL),     # rank 2 just kept
    (0.75, {0, 2}, 0.0),                      # on the edge: dropped, and always excused
    (0.6, {0, 2}, 0.1),                       # far from both edges: 0.6 - 0.5
])
def test_top_p_margin_is_distance_to_cut(orc, tp, kept, want):
    for scale in (1.0, 0.5):  # the margin is relative to the kept mass
        p = np.array([P4], np.float32) * np.float32(scale)
        out, m = orc.topk_topp_renorm(p, top_p=np.array([tp], np.float32))
        assert {i for i in range(4) if out[0, i] > 0} == kept
        assert m[0] == pytest.approx(want, rel=1e-6, abs=1e-16)


def test_top_p_margin_is_relative_to_top_k_mass(orc):
    # top-k = 4 drops the 0.1 token: the kept mass is 1 (not the row's 1.1), so a cut
    # 2^-20 from the edge reports 2^-20
    p = np.array([P4 + [0.1]], np.float32)
    out, m = orc.topk_topp_renorm(p, top_k=np.array([4], np.int32),
                                  top_p=np.array([0.75 - D_SMALL], np.float32))
    assert {i for i in range(5) if out[0, i] > 0} == {0, 2}
    assert m[0] == pytest.approx(D_SMALL, rel=1e-6)


def test_top_p_margin_enters_the_chain(orc):
    # the same cut inside a target-only chain from logits: log2 of the masses as logits
    # at T = 1 / ln 2 give the P4 weights up to the fp32 rounding of T (a few 1e-9)
    l = [math.log2(v) + 1.0 for v in P4]
    Tln2 = np.float32(1.0 / math.log(2.0))
    x = np.array([l, [0.0, -np.inf, -np.inf, -np.inf]], np.float32)
    r = _chain(orc, x, 1, [[2]], [[0.1, 0.3]], temperature=np.array([Tln2], np.float32),
               top_p=np.array([0.75 - D_SMALL], np.float32))
    # draft 2 (p'' = 2/3) is accepted with u = 0.1; the bonus row is one-hot
    assert list(r["accepted_tokens"][0]) == [2, 0]
    assert r["margin"][0] == pytest.approx(D_SMALL, abs=1e-8)


# ---- the final draw --------------------------------------------------------------------

@pytest.mark.parametrize("uD,tok,want", [(0.375 + D_SMALL, 2, D_SMALL),
                                         (0.375 - D_SMALL, 1, D_SMALL),
                                         (0.375, 2, 0.0),
                                         (0.5, 2, 0.125)])
def test_draw_margin_is_distance_to_cdf_edge(orc, uD, tok, want):
    # bonus draw (D = 0) from P4 in token-id order: inclusive prefixes 0.25, 0.375,
    # 0.875, 1; scaling the row by 1/2 leaves the relative margin unchanged
    for scale in (1.0, 0.5):
        p = np.array([P4], np.float32) * np.float32(scale)
        r = _chain(orc, p, 0, np.zeros((1, 0)), [[uD]], logits=False)
        assert r["accepted_tokens"][0, 0] == tok
        assert r["margin"][0] == pytest.approx(want, rel=1e-6, abs=1e-16)


def test_draw_margin_on_the_residual_is_relative_to_its_mass(orc):
    # target-only rejection of draft 2 (u = 0.9 > p(2) = 0.5, an exact fp32 decision):
    # residual (0.25, 0.125, 0, 0.125), mass 1/2, prefixes 0.25, 0.375, 0.375, 0.5.
    # u_D = 1/2 + 2d puts t = 1/4 + d, i.e. d past the first edge: relative margin
    # d / (1/2) = 2d (an absolute margin would read d).
    p = np.array([P4, [1.0, 0.0, 0.0, 0.0]], np.float32)
    r = _chain(orc, p, 1, [[2]], [[0.9, 0.5 + 2 * D_SMALL]], logits=False)
    assert list(r["accepted_tokens"][0]) == [1, -1]
    assert r["margin"][0] == pytest.approx(2 * D_SMALL, rel=1e-6)


# ---- Gumbel best minus second ------------------------------------------------------------

@pytest.mark.parametrize("level,delta", [(0.5, 1e-3), (10.0, 1e-3), (0.5, 0.0)])
def test_gumbel_margin_is_best_minus_second(orc, level, delta):
    # logits placed against the oracle's own noise for this (seed, offset, row) so that
    # token 1 beats token 0 by about delta and token 2 trails by 5: the margin is the
    # top-two gap over max(1, |best|), not the gap to the third
    seed, off = 97, 3
    g = [-math.log(-math.log(float(orc.gumbel_u01(seed, off, 0, v)))) for v in range(3)]
    l = np.array([[level - g[0], level - g[1] + delta, level - 5.0 - g[2]]], np.float32)
    s = [float(l[0, v]) + g[v] for v in range(3)]  # the scores at T = 1
    tok, marg = orc.gumbel_max_sample(l, 1, np.ones(1, np.float32), np.array([seed]),
                                      np.array([off]))
    best = int(np.argmax(s))
    gap = abs(s[1] - s[0])
    assert tok[0] == best
    assert marg[0] == pytest.approx(gap / max(1.0, abs(s[best])), rel=1e-9, abs=1e-15)
    if delta == 0.0:
        assert marg[0] <= 1e-6  # a tie up to the logits' rounding is flagged
    else:
        assert marg[0] == pytest.approx(delta / max(1.0, level), rel=1e-3)


# ---- the logits + draft-probabilities branch -----------------------------------------------

def _softmax(l, T):
    z = np.asarray(l, np.float64) / np.float64(np.float32(T))
    e = np.exp(z - z.max())
    return e / e.sum()


def _topk_renorm(p, k):
    if k <= 0 or k >= len(p):
        return p
    order = sorted(range(len(p)), key=lambda i: (-p[i], i))
    out = np.zeros_like(p)
    out[order[:k]] = p[order[:k]]
    return out / out.sum()


def _chain_law(p, q):
    """Exact law of the emitted sequence: drafts x_j ~ q_j, accept w.p. min(1, p/q),
    residual norm(max(p - q, 0)) at the first rejection, bonus from p_D."""
    D, V = len(q), len(p[0])
    law = {}

    def rec(j, prefix, prob):
        if j == D:
            for t in range(V):
                law[prefix + (t,)] = law.get(prefix + (t,), 0.0) + prob * p[D][t]
            return
        r = np.maximum(p[j] - q[j], 0.0)
        r = r / r.sum()
        rej = 0.0
        for x in range(V):
            if q[j][x] == 0.0:
                continue
            a = min(1.0, p[j][x] / q[j][x])
            rec(j + 1, prefix + (x,), prob * q[j][x] * a)
            rej += q[j][x] * (1.0 - a)
        for t in range(V):
            law[prefix + (t,)] = law.get(prefix + (t,), 0.0) + prob * rej * r[t]

    rec(0, (), 1.0)
    return law


@pytest.mark.parametrize("V,D,T,k", [(3, 2, 0.8, 0), (4, 1, 1.3, 2), (3, 3, 1.0, 0)])
def test_logits_with_draft_probs_chain_law_chi_square(orc, V, D, T, k):
    rng = np.random.default_rng(1000 + 10 * V + D)
    R, n = D + 1, 100000
    lg = (rng.standard_normal((R, V)) * 1.2).astype(np.float32)
    p = [_topk_renorm(_softmax(lg[j], T), k) for j in range(R)]
    q = []
    for _ in range(D):
        w = rng.gamma(0.8, size=V) + 0.05
        q.append((w / w.sum()).astype(np.float32).astype(np.float64))
    drafts = np.stack([rng.choice(V, size=n, p=q[j] / q[j].sum()) for j in range(D)], 1)
    r = orc.chain_spec_sampling(np.tile(lg, (n, 1)), True, D, drafts.astype(np.int32),
                                draft_probs=np.tile(np.stack(q).astype(np.float32)[None],
                                                    (n, 1, 1)),
                                temperature=np.full(n, T, np.float32),
                                top_k=np.full(n, k, np.int32), seed=np.full(n, 31, np.int64),
                                offset=np.arange(n, dtype=np.int64), logprobs=False)
    L = r["accept_length"]
    assert L.min() >= 1 and L.max() <= R
    law = _chain_law(p, q)
    keys = sorted(law)
    index = {key: i for i, key in enumerate(keys)}
    counts = np.zeros(len(keys))
    for b in range(n):
        counts[index[tuple(r["accepted_tokens"][b, :L[b]])]] += 1
    expect = np.array([law[key] for key in keys])
    expect = expect / expect.sum() * n
    assert counts[expect == 0].sum() == 0
    counts, expect = counts[expect > 0], expect[expect > 0]
    keep = expect > 5
    obs, ex = counts[keep], expect[keep]
    if (~keep).any():
        obs, ex = np.append(obs, counts[~keep].sum()), np.append(ex, expect[~keep].sum())
    assert stats.chisquare(obs, ex).pvalue > 1e-4
    # the speculative-sampling theorem: position 0 is distributed as p_0
    first = np.bincount(r["accepted_tokens"][:, 0], minlength=V)
    nz = p[0] > 0
    assert (first[~nz] == 0).all()
    assert stats.chisquare(first[nz], p[0][nz] / p[0][nz].sum() * n).pvalue > 1e-4


def test_logits_with_draft_probs_hand_example(orc):
    # logits (0, ln 3) at T = 1: p = (1/4, 3/4) up to the fp32 rounding of ln 3;
    # q = (1/2, 1/2), draft 0: u q = 0.3 >= p(0) -> reject; residual (0, p1 - 1/2):
    # token 1 for every u_D. u = 0.4: 0.2 < 1/4 -> accept, bonus from row 1.
    l = np.array([[0.0, math.log(3.0)], [0.0, -np.inf]], np.float32)
    q = np.array([[[0.5, 0.5]]], np.float32)
    for uD in (0.01, 0.99):
        r = _chain(orc, l, 1, [[0]], [[0.6, uD]], draft_probs=q)
        assert list(r["accepted_tokens"][0]) == [1, -1]
    r = _chain(orc, l, 1, [[0]], [[0.4, 0.5]], draft_probs=q)
    assert list(r["accepted_tokens"][0]) == [0, 0]
    p0 = 1.0 / (1.0 + math.exp(float(l[0, 1])))
    assert r["margin"][0] == pytest.approx(abs(float(np.float32(0.4)) * 0.5 - p0), rel=1e-9)
