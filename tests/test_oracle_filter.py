"""Pins for the oracle's softmax, top-k/top-p renorm, argmax and logprobs (CPU only).

Each check rests on something outside the oracle's own code: a closed form,
a library routine doing the same textbook operation (torch in float64), a
hand-worked example, or the defining property of the set being selected.
"""
import itertools
import math

import numpy as np
import pytest
import torch


def test_argmax_lowest_index_on_ties(orc):
    assert orc.argmax(np.array([1, 3, 3, 2], np.float32)) == 1
    assert orc.argmax(np.array([-np.inf, -np.inf, 0.5], np.float32)) == 2
    x = np.random.default_rng(0).integers(-3, 3, size=(50, 17)).astype(np.float32)
    for row in x:
        assert orc.argmax(row) == int(torch.argmax(torch.from_numpy(row)))


def test_softmax_two_token_closed_form(orc):
    # p_0 = 1 / (1 + exp((l_1 - l_0) / T)): the logistic form of a 2-way softmax
    for l0, l1, T in [(0.0, 1.0, 1.0), (2.5, -1.25, 0.5), (3.0, 3.0, 2.0), (-7.0, 1.0, 1.3)]:
        p = orc.softmax_temp(np.array([[l0, l1]], np.float32),
                             np.array([T], np.float32))[0]
        want = 1.0 / (1.0 + math.exp((float(np.float32(l1)) - float(np.float32(l0)))
                                     / float(np.float32(T))))
        assert p[0] == pytest.approx(want, rel=1e-14)
        assert p[0] + p[1] == pytest.approx(1.0, abs=1e-15)


def test_softmax_matches_torch_float64(orc):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((6, 300)) * 4).astype(np.float32)
    T = np.array([1.0, 0.5, 2.0, 0.3, 1.7, 1e-4], np.float32)
    p = orc.softmax_temp(x, T)
    ref = torch.softmax(torch.from_numpy(x).double() / torch.from_numpy(T).double()[:, None],
                        dim=-1).numpy()
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)


def test_softmax_greedy_and_masked(orc):
    x = np.array([[0.1, 2.0, 2.0, -1.0], [1.0, -np.inf, 0.0, -np.inf]], np.float32)
    p = orc.softmax_temp(x, np.array([0.0, 1.0], np.float32))
    np.testing.assert_array_equal(p[0], [0, 1, 0, 0])  # one-hot at the lowest argmax
    assert p[1, 1] == 0.0 and p[1, 3] == 0.0
    assert p[1, 0] == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-14)
    # the greedy threshold: just below is one-hot, at the threshold it is not
    y = np.array([[0.0, 1e-6]], np.float32)
    assert orc.softmax_temp(y, np.array([9.9e-6], np.float32))[0, 1] == 1.0
    assert orc.softmax_temp(y, np.array([1e-5], np.float32))[0, 1] < 1.0


def test_renorm_hand_example(orc):
    # p = (0.5, 0.3, 0.2), top_p = 0.6: mass before token 1 is 0.5 < 0.6 (kept),
    # mass before token 2 is 0.8 >= 0.6 (dropped) -> (0.625, 0.375, 0)
    p = np.array([[0.5, 0.3, 0.2]], np.float32)
    out, m = orc.topk_topp_renorm(p, top_p=np.array([0.6], np.float32))
    np.testing.assert_allclose(out[0], [0.5 / 0.8, 0.3 / 0.8, 0.0], rtol=1e-7)
    # top_k = 2 alone gives the same support
    out2, _ = orc.topk_topp_renorm(p, top_k=np.array([2], np.int32))
    np.testing.assert_allclose(out2[0], out[0], rtol=1e-7)
    # top_k = 1 is the argmax; top_k >= V and top_p = 1 are the identity
    out3, _ = orc.topk_topp_renorm(p, top_k=np.array([1], np.int32))
    np.testing.assert_array_equal(out3[0], [1.0, 0.0, 0.0])
    for k in (0, 3, 7, -2):
        o, _ = orc.topk_topp_renorm(p, top_k=np.array([k], np.int32),
                                    top_p=np.array([1.0], np.float32))
        np.testing.assert_allclose(o[0], p[0] / p[0].astype(np.float64).sum(), rtol=1e-7)


def test_renorm_ties_keep_lowest_ids(orc):
    p = np.array([[0.1, 0.3, 0.2, 0.3, 0.1]], np.float32)
    out, _ = orc.topk_topp_renorm(p, top_k=np.array([1], np.int32))
    np.testing.assert_array_equal(out[0], [0, 1, 0, 0, 0])
    out, _ = orc.topk_topp_renorm(p, top_k=np.array([4], np.int32))
    assert out[0, 4] == 0.0 and out[0, 0] > 0.0


def _defining_property(vals, w, k, top_p):
    """The kept set from its definition: the k-prefix of the order, then the
    shortest prefix of it whose mass reaches top_p of the k-prefix mass."""
    V = len(vals)
    order = sorted(range(V), key=lambda i: (-float(vals[i]), i))
    kk = k if 0 < k < V else V
    pref = order[:kk]
    Zk = sum(w[i] for i in pref)
    if top_p >= 1.0:
        return set(pref)
    for n in range(1, kk + 1):
        if sum(w[i] for i in pref[:n]) >= top_p * Zk:
            return set(pref[:n])
    return set(pref)


@pytest.mark.parametrize("V", [1, 2, 3, 5, 8])
def test_renorm_brute_force_all_tie_patterns(orc, V):
    # values on a coarse grid so that every tie pattern of small rows shows up
    grid = [0.05, 0.1, 0.2, 0.4]
    rng = np.random.default_rng(V)
    rows = list(itertools.product(grid, repeat=V)) if V <= 3 else \
        [tuple(rng.choice(grid, V)) for _ in range(300)]
    for vals in rows:
        p = np.array(vals, np.float32)
        w = p.astype(np.float64)
        for k in (0, 1, 2, V):
            for tp in (1.0, 0.95, 0.5, 0.3):
                out, m = orc.topk_topp_renorm(p[None], top_k=np.array([k], np.int32),
                                              top_p=np.array([tp], np.float32))
                kept = _defining_property(p, w, k, np.float64(np.float32(tp)))
                got = {i for i in range(V) if out[0, i] > 0}
                if m >= 1e-9:  # exactly-at-threshold cuts are the boundary rule's business
                    assert got == kept, (vals, k, tp)
                Z = sum(w[i] for i in got)
                for i in got:
                    assert out[0, i] == pytest.approx(w[i] / Z, rel=1e-12)


def test_renorm_from_logits_orders_by_logit(orc):
    # with logits the order is the logit order and the weights the softmax
    x = np.array([2.0, 1.0, 2.0, 0.0, -1.0], np.float32)
    out, m = orc.filter_row(x, True, T=1.0, top_k=2)
    e = np.exp(np.array([2.0, 2.0]) - 2.0)
    np.testing.assert_allclose(out, [0.5, 0, 0.5, 0, 0], rtol=1e-14)
    out, m = orc.filter_row(x, True, T=1.0, top_p=0.5)
    # sorted masses e^0, e^0, e^-1, ...; the first token alone has mass < 0.5 Z
    # only if Z > 2: Z = 2 + e^-1 + e^-2 + e^-3 = 2.553, 0.5 Z = 1.277 > 1 -> keep two
    np.testing.assert_allclose(out[[0, 2]], [0.5, 0.5], rtol=1e-14)
    assert e.sum() == 2.0


def test_topk_exact_k_with_ties_in_logits(orc):
    x = np.array([1.0, 3.0, 3.0, 3.0, 0.0], np.float32)
    out, _ = orc.filter_row(x, True, T=0.7, top_k=2)
    assert set(np.nonzero(out)[0]) == {1, 2}


def test_logprobs_match_torch(orc):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((8, 97)) * 3).astype(np.float32)
    x[0, 5] = -np.inf
    tok = rng.integers(0, 97, size=8).astype(np.int32)
    tok[0] = 4
    tok[3] = -1
    got = orc.gather_logprobs(x, False, tok)
    ref = torch.log_softmax(torch.from_numpy(x).double(), -1).numpy()
    for r in range(8):
        want = 0.0 if tok[r] < 0 else ref[r, tok[r]]
        assert got[r] == pytest.approx(want, rel=1e-13, abs=1e-13)
    p = torch.softmax(torch.from_numpy(x).double(), -1).float().numpy()
    got = orc.gather_logprobs(p, True, tok)
    for r in range(8):
        want = 0.0 if tok[r] < 0 else math.log(float(p[r, tok[r]]))
        assert got[r] == pytest.approx(want, rel=1e-13)
