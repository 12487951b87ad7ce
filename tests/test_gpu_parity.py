"""GPU parity: every C-ABI call against the oracle on the same seeded inputs.

Sizes span several tiles, clusters of 1 to 8 CTAs and ragged tails; the workloads of
the benchmark configurations are covered at full size in test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_temp_gb300 import synth
from speculative_decoding_verify_temp_gb300 import tsverify as tv
from tests.gpu_util import TOL, BOUNDARY, compare_chain, dev, dev_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    oracle.build()
    yield
    assert tv.device_error() == 0


def _rand_logits(rng, rows, V, dtype, sigma=3.0, zipf=True):
    x = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(sigma)
    if zipf:
        x += synth.zipf_bias(V)[None, :]
    if dtype == "bf16":
        bits = synth.bf16_bits_from_f32(x)
        return dict(dtype="bf16", logits_bits=bits, logits=synth.f32_from_bf16_bits(bits))
    return dict(dtype="f32", logits=x)


# ---- greedy chain verification ------------------------------------------------------------

@pytest.mark.parametrize("B,D,V,dtype", [(4, 3, 1024, "f32"), (64, 3, 32000, "bf16"),
                                         (7, 0, 1000, "f32"), (5, 6, 129, "bf16"),
                                         (3, 2, 7, "f32"), (2, 1, 1, "f32"),
                                         (16, 4, 50007, "bf16")])
def test_greedy_verify(B, D, V, dtype):
    rng = np.random.default_rng(B * 1000 + V)
    d = _rand_logits(rng, B * (D + 1), V, dtype)
    am = d["logits"].reshape(B, D + 1, V)[:, :D].argmax(-1)
    drafts = np.where(rng.random((B, D)) < 0.7, am, rng.integers(0, V, (B, D))).astype(np.int32)
    g = tv.verify_chain_greedy(dev_logits(d), D, dev(drafts))
    ref = oracle.verify_chain_greedy(d["logits"], D, drafts)
    compare_chain(g, ref, dtype)


def test_greedy_verify_ties_neginf_and_padded_rows():
    B, D, V = 6, 3, 300
    x = np.zeros((B * (D + 1), V), np.float32)
    x[:, 250:] = -np.inf
    x[0, [5, 9]] = 3.0  # tie: the lowest id wins
    x[1, :] = -np.inf  # an all -inf row has argmax 0
    x[2, 249] = -1.0  # below the zeros: the row argmax stays at id 0
    drafts = np.array([[9, 0, 0], [0, 0, 0], [0, 1, 2], [3, 3, 3], [0, 0, 0], [1, 1, 1]], np.int32)
    ld = 320  # padded rows: ld > V, 16-byte aligned
    xp = np.full((B * (D + 1), ld), 7.0, np.float32)
    xp[:, :V] = x
    xt = torch.from_numpy(xp).cuda()[:, :V]
    g = tv.verify_chain_greedy(xt, D, dev(drafts))
    ref = oracle.verify_chain_greedy(x, D, drafts)
    compare_chain(g, ref, "f32")
    # a row stride that breaks 16-byte alignment takes the scalar path
    ld2 = 301
    xq = np.full((B * (D + 1), ld2), 7.0, np.float32)
    xq[:, :V] = x
    g = tv.verify_chain_greedy(torch.from_numpy(xq).cuda()[:, :V], D, dev(drafts))
    compare_chain(g, ref, "f32")


# ---- logprobs ------------------------------------------------------------------------------

@pytest.mark.parametrize("rows,V,dtype", [(33, 1000, "f32"), (9, 128256, "bf16"), (5, 3, "f32")])
def test_gather_logprobs(rows, V, dtype):
    rng = np.random.default_rng(rows + V)
    d = _rand_logits(rng, rows, V, dtype)
    tok = rng.integers(-1, V, rows).astype(np.int32)
    got = tv.gather_logprobs(dev_logits(d), dev(tok)).cpu().numpy()
    np.testing.assert_allclose(got, oracle.gather_logprobs(d["logits"], False, tok), **TOL[dtype])
    p = oracle.softmax_temp(d["logits"]).astype(np.float32)
    got = tv.gather_logprobs(dev(p), dev(tok), is_probs=True).cpu().numpy()
    np.testing.assert_allclose(got, oracle.gather_logprobs(p, True, tok), rtol=1e-6, atol=1e-6)


# ---- softmax -------------------------------------------------------------------------------

@pytest.mark.parametrize("rows,V,dtype", [(8, 1024, "f32"), (5, 40000, "f32"), (6, 128256, "bf16"),
                                          (3, 201088, "bf16"), (4, 151936, "f32"), (3, 17, "bf16"),
                                          (2, 300000, "f32")])
def test_softmax_temp(rows, V, dtype):
    rng = np.random.default_rng(rows * 7 + V)
    d = _rand_logits(rng, rows, V, dtype)
    T = rng.uniform(0.3, 1.5, rows).astype(np.float32)
    T[0] = 0.0  # greedy row
    got = tv.softmax_temp(dev_logits(d), dev(T)).cpu().numpy()
    ref = oracle.softmax_temp(d["logits"], T)
    np.testing.assert_allclose(got, ref, **TOL[dtype])
    np.testing.assert_allclose(got.sum(-1), 1.0, rtol=1e-5)


@pytest.mark.parametrize("V,dtype", [(1001, "bf16"), (65539, "bf16"), (40001, "f32")])
def test_softmax_temp_padded_rows(V, dtype):
    # 16-byte aligned rows (ld padded) whose vocabulary ends inside a vector: the staged
    # slices end on a ragged tail read from global memory
    rng = np.random.default_rng(V)
    rows = 5
    x = rng.standard_normal((rows, V)).astype(np.float32) * np.float32(2.0)
    if dtype == "bf16":
        x = synth.f32_from_bf16_bits(synth.bf16_bits_from_f32(x))
    T = rng.uniform(0.3, 1.5, rows).astype(np.float32)
    T[1] = 0.0
    ld = (V + 7) // 8 * 8
    full = np.zeros((rows, ld), np.float32)
    full[:, :V] = x
    t = torch.from_numpy(full).cuda()
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    got = tv.softmax_temp(t[:, :V], dev(T)).cpu().numpy()
    ref = oracle.softmax_temp(x, T)
    np.testing.assert_allclose(got, ref, **TOL[dtype])
    np.testing.assert_allclose(got.sum(-1), 1.0, rtol=1e-5)


# ---- top-k / top-p renorm --------------------------------------------------------------------

def _check_renorm(got, ref, marg, probs):
    ok = marg > BOUNDARY
    assert (~ok).sum() <= max(1, len(ok) // 50)
    np.testing.assert_array_equal(got[ok] > 0, ref[ok] > 0)
    np.testing.assert_allclose(got[ok], ref[ok], rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("rows,V", [(24, 1000), (12, 32000), (8, 151936), (10, 5)])
def test_topk_topp_renorm(rows, V):
    rng = np.random.default_rng(rows + 3 * V)
    d = _rand_logits(rng, rows, V, "f32", sigma=2.5)
    T = rng.uniform(0.5, 1.2, rows).astype(np.float32)
    p = oracle.softmax_temp(d["logits"], T).astype(np.float32)
    k = rng.choice(np.array([0, 1, 20, 50, 1000, V, -3], np.int32), rows).astype(np.int32)
    tp = rng.choice(np.array([1.0, 0.95, 0.9, 0.5, 0.0], np.float32), rows).astype(np.float32)
    got = tv.topk_topp_renorm(dev(p), dev(k), dev(tp)).cpu().numpy()
    ref, marg = oracle.topk_topp_renorm(p, k, tp)
    _check_renorm(got, ref, marg, p)
    # knobs absent: pure renormalisation
    got = tv.topk_topp_renorm(dev(p)).cpu().numpy()
    ref, marg = oracle.topk_topp_renorm(p)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


def test_renorm_ties_exact_k():
    # many equal probabilities around the k-th: exactly k survive, lowest ids first
    V = 4096
    p = np.full((3, V), 1.0 / V, np.float32)
    p[1, ::3] = 2.0 / V
    p[2, 100:200] = 5.0 / V
    p /= p.sum(-1, keepdims=True)
    k = np.array([10, 700, 150], np.int32)
    got = tv.topk_topp_renorm(dev(p), dev(k)).cpu().numpy()
    ref, _ = oracle.topk_topp_renorm(p, k)
    np.testing.assert_array_equal(got > 0, ref > 0)
    assert ((got > 0).sum(-1) == k).all()
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("V", [3000, 40000, 151936])
def test_topk_only_flat_rows(V):
    # top-k without top-p on flat rows: the k-th key is found among the elements that pass
    # the thread-maxima bound, so membership must apply that bound too
    rng = np.random.default_rng(V)
    p = oracle.softmax_temp(rng.standard_normal((6, V)).astype(np.float32)).astype(np.float32)
    k = np.array([1, 5, 17, 100, 1000, 4000], np.int32)
    got = tv.topk_topp_renorm(dev(p), dev(k)).cpu().numpy()
    ref, _ = oracle.topk_topp_renorm(p, k)
    np.testing.assert_array_equal(got > 0, ref > 0)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-7)


def test_renorm_in_place():
    rng = np.random.default_rng(9)
    p = oracle.softmax_temp(rng.standard_normal((4, 3000)).astype(np.float32)).astype(np.float32)
    t = dev(p)
    k = dev(np.array([5, 0, 100, 3000], np.int32))
    tv.topk_topp_renorm(t, k, None, out=t)
    ref, _ = oracle.topk_topp_renorm(p, np.array([5, 0, 100, 3000], np.int32))
    np.testing.assert_allclose(t.cpu().numpy(), ref, rtol=1e-5, atol=1e-7)


def _renorm_rows(rng, rows, V):
    """Probability rows of several shapes: smooth, heavy-tailed down to denormals, sparse,
    one-hot and flat."""
    kind = rng.integers(0, 5, rows)
    p = np.empty((rows, V), np.float32)
    for r in range(rows):
        if kind[r] == 0:
            x = rng.standard_normal(V).astype(np.float32) * np.float32(2.0)
        elif kind[r] == 1:
            x = rng.standard_normal(V).astype(np.float32) * np.float32(30.0)
        else:
            x = rng.standard_normal(V).astype(np.float32)
        q = oracle.softmax_temp(x[None])[0]
        if kind[r] == 2:
            q = q * (rng.random(V) < 0.1)
            q[rng.integers(0, V)] += 0.01
        elif kind[r] == 3:
            q = np.zeros(V)
            q[rng.integers(0, V)] = 1.0
        elif kind[r] == 4:
            q = np.full(V, 1.0)
        p[r] = (q / q.sum()).astype(np.float32)
    return p


@pytest.mark.parametrize("V,rows", [(1, 40), (7, 320), (4095, 320), (4097, 320), (8193, 320),
                                    (70001, 40), (262144, 12)])
def test_renorm_row_kernel_edges(V, rows):
    # vocabularies around the row kernel's 16 KB stages and its largest vocabulary, padded
    # rows (16-byte aligned, ld > V), more rows than resident CTAs, every knob kind
    rng = np.random.default_rng(V + rows)
    p = _renorm_rows(rng, rows, V)
    k = rng.choice(np.array([0, 1, 5, 300, 1024, 1025, 3000, V + 1, -3], np.int32),
                   rows).astype(np.int32)
    tp = rng.choice(np.array([1.0, 0.9, 0.5, 0.0], np.float32), rows).astype(np.float32)
    ld = (V + 3) // 4 * 4 + 4
    full = np.full((rows, ld), 7.0, np.float32)  # the padding must not be read
    full[:, :V] = p
    t = torch.from_numpy(full).cuda()
    got = tv.topk_topp_renorm(t[:, :V], dev(k), dev(tp)).cpu().numpy()
    ref, marg = oracle.topk_topp_renorm(p, k, tp)
    ok = marg > BOUNDARY
    assert ok.mean() > 0.9
    np.testing.assert_array_equal(got[ok] > 0, ref[ok] > 0)
    np.testing.assert_allclose(got[ok], ref[ok], rtol=1e-5, atol=1e-6)
    # rows near a top-p boundary still hold a valid distribution over a prefix of the order
    np.testing.assert_allclose(got.sum(-1), 1.0, rtol=1e-5)
    assert (got[p == 0] == 0).all()


# ---- chain speculative sampling: probability rows ----------------------------------------------

def test_rejection_tiny_config():
    d = synth.tiny_verify()
    B, D, V = d["B"], d["D"], d["V"]
    p = oracle.softmax_temp(d["logits"]).astype(np.float32)
    g = tv.chain_spec_sampling(dev(p), False, D, dev(d["draft_tokens"]),
                               draft_probs=dev(d["draft_probs"]), seed=dev(d["seed"]),
                               offset=dev(d["offset"]))
    ref = oracle.chain_spec_sampling(p, False, D, d["draft_tokens"], draft_probs=d["draft_probs"],
                                     seed=d["seed"], offset=d["offset"])
    compare_chain(g, ref, "f32")


@pytest.mark.parametrize("B,D,V,with_q", [(64, 3, 5000, True), (40, 7, 30011, True),
                                          (50, 4, 2048, False), (16, 1, 3, True),
                                          (8, 0, 100, False)])
def test_rejection_probs(B, D, V, with_q):
    rng = np.random.default_rng(B + D + V)
    R = D + 1
    tl = rng.standard_normal((B * R, V)).astype(np.float32) * 2.5
    p = oracle.softmax_temp(tl).astype(np.float32)
    q = oracle.softmax_temp(tl.reshape(B, R, V)[:, :D].reshape(B * D, V)
                            + rng.standard_normal((B * D, V)).astype(np.float32) * 0.7)
    q = q.astype(np.float32).reshape(B, D, V)
    src = q if with_q else p.reshape(B, R, V)[:, :D]
    src = src.astype(np.float64)
    drafts = np.array([[rng.choice(V, p=src[b, j] / src[b, j].sum())
                        for j in range(D)] for b in range(B)], np.int32).reshape(B, D)
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64) * 3
    kw = dict(draft_probs=dev(q) if with_q else None, seed=dev(seed), offset=dev(off))
    g = tv.chain_spec_sampling(dev(p), False, D, dev(drafts), **kw)
    ref = oracle.chain_spec_sampling(p, False, D, drafts, draft_probs=q if with_q else None,
                                     seed=seed, offset=off)
    compare_chain(g, ref, "f32")
    # explicit uniforms replace Philox
    uni = rng.uniform(0.0, 1.0, (B, R)).astype(np.float32)
    uni = np.clip(uni, 1e-7, 1 - 1e-7).astype(np.float32)
    g = tv.chain_spec_sampling(dev(p), False, D, dev(drafts), draft_probs=kw["draft_probs"],
                               uniforms=dev(uni))
    ref = oracle.chain_spec_sampling(p, False, D, drafts, draft_probs=q if with_q else None,
                                     uniforms=uni)
    compare_chain(g, ref, "f32")


# ---- chain speculative sampling: target-only from logits ----------------------------------------

@pytest.mark.parametrize("B,D,V,dtype", [(4, 3, 1024, "f32"), (48, 4, 32000, "bf16"),
                                         (12, 4, 128256, "bf16"), (6, 3, 201088, "bf16"),
                                         (10, 2, 40000, "f32"), (9, 0, 3000, "f32")])
def test_target_only_from_logits(B, D, V, dtype):
    rng = np.random.default_rng(B * 31 + V)
    R = D + 1
    d = _rand_logits(rng, B * R, V, dtype)
    T = rng.uniform(0.3, 1.5, B).astype(np.float32)
    T[rng.random(B) < 0.2] = 0.0
    k = rng.choice(np.array(synth.TOPK_CHOICES, np.int32), B).astype(np.int32)
    tp = rng.choice(np.array(synth.TOPP_CHOICES, np.float32), B).astype(np.float32)
    lg = d["logits"].reshape(B, R, V)[:, :D]
    am = lg.argmax(-1)
    drafts = np.where(rng.random((B, D)) < 0.6, am, rng.integers(0, V, (B, D))).astype(np.int32)
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64)
    g = tv.chain_spec_sampling(dev_logits(d), True, D, dev(drafts), temperature=dev(T),
                               top_k=dev(k), top_p=dev(tp), seed=dev(seed), offset=dev(off))
    ref = oracle.chain_spec_sampling(d["logits"], True, D, drafts, temperature=T, top_k=k,
                                     top_p=tp, seed=seed, offset=off)
    compare_chain(g, ref, dtype, max_boundary_frac=0.05)


@pytest.mark.parametrize("pad,dtype", [(8, "bf16"), (3, "bf16"), (4, "f32"), (1, "f32")])
def test_target_only_mixed_routes_and_strides(pad, dtype):
    # One launch mixes greedy requests, small and large top-k (above the split-row
    # kernel's limit: the staged kernel finishes those rows), top-p alone, knobs off and
    # rows with only a few finite logits; rows are `pad` elements longer than the
    # vocabulary, so with pad 3 (bf16) or 1 (f32) they are not 16-byte aligned.
    rng = np.random.default_rng(1000 + pad)
    B, D, V = 30, 3, 50000
    R = D + 1
    x = rng.standard_normal((B * R, V), dtype=np.float32) * np.float32(3.0)
    x += synth.zipf_bias(V)[None, :]
    x[5 * R:6 * R] = -np.inf
    x[5 * R:6 * R, 7:17] = rng.standard_normal((R, 10)).astype(np.float32)
    x[6 * R:7 * R, 1000:] = -np.inf
    if dtype == "bf16":
        x = synth.f32_from_bf16_bits(synth.bf16_bits_from_f32(x))
    T = rng.choice(np.array([0.0, 0.5, 1.3], np.float32), B)
    k = rng.choice(np.array([0, 5, 1000, 2000, V + 1], np.int32), B).astype(np.int32)
    tp = rng.choice(np.array([1.0, 0.9, 0.0], np.float32), B).astype(np.float32)
    T[5:7] = 1.0
    k[5:7] = (1000, 50)
    lg = x.reshape(B, R, V)[:, :D]
    drafts = np.where(rng.random((B, D)) < 0.6, lg.argmax(-1),
                      rng.integers(0, V, (B, D))).astype(np.int32)
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64)
    full = np.zeros((B * R, V + pad), np.float32)
    full[:, :V] = x
    t = torch.from_numpy(full).cuda()
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    g = tv.chain_spec_sampling(t[:, :V], True, D, dev(drafts), temperature=dev(T),
                               top_k=dev(k), top_p=dev(tp), seed=dev(seed), offset=dev(off),
                               logprobs=True)
    ref = oracle.chain_spec_sampling(x, True, D, drafts, temperature=T, top_k=k, top_p=tp,
                                     seed=seed, offset=off)
    compare_chain(g, ref, dtype)


@pytest.mark.parametrize("V,dtype", [(1, "f32"), (7, "bf16"), (9, "f32"), (4095, "f32"),
                                     (8191, "bf16"), (8193, "bf16"), (16385, "f32"),
                                     (24577, "bf16")])
def test_target_only_vocab_edges(V, dtype):
    # vocabularies around the row kernel's 16 KB stages, with a ragged last vector; rows are
    # padded to 16 elements so that they stay 16-byte aligned (the row kernel's route)
    rng = np.random.default_rng(V + 7)
    B, D = 12, 3
    R = D + 1
    x = rng.standard_normal((B * R, V), dtype=np.float32) * np.float32(2.0)
    if dtype == "bf16":
        x = synth.f32_from_bf16_bits(synth.bf16_bits_from_f32(x))
    T = rng.choice(np.array([0.0, 0.7, 1.3], np.float32), B).astype(np.float32)
    k = rng.choice(np.array([0, 1, 5, 300, V + 1], np.int32), B).astype(np.int32)
    tp = rng.choice(np.array([1.0, 0.9, 0.0], np.float32), B).astype(np.float32)
    lg = x.reshape(B, R, V)[:, :D]
    drafts = np.where(rng.random((B, D)) < 0.6, lg.argmax(-1),
                      rng.integers(0, V, (B, D))).astype(np.int32)
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64)
    ld = (V + 15) // 16 * 16
    full = np.zeros((B * R, ld), np.float32)
    full[:, :V] = x
    t = torch.from_numpy(full).cuda()
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    g = tv.chain_spec_sampling(t[:, :V], True, D, dev(drafts), temperature=dev(T),
                               top_k=dev(k), top_p=dev(tp), seed=dev(seed), offset=dev(off))
    ref = oracle.chain_spec_sampling(x, True, D, drafts, temperature=T, top_k=k, top_p=tp,
                                     seed=seed, offset=off)
    compare_chain(g, ref, dtype)


def test_renorm_many_short_rows():
    # more rows than the CTAs' tiered row lists hold (they then take rows in turn), and a
    # count just below that limit
    for rows in (160000, 150000):
        rng = np.random.default_rng(rows)
        V = 8
        p = rng.random((rows, V)).astype(np.float32)
        p /= p.sum(-1, keepdims=True)
        k = rng.choice(np.array([0, 1, 3, 5], np.int32), rows).astype(np.int32)
        tp = rng.choice(np.array([1.0, 0.5, 0.8], np.float32), rows).astype(np.float32)
        got = tv.topk_topp_renorm(dev(p), dev(k), dev(tp)).cpu().numpy()
        want, marg = oracle.topk_topp_renorm(p, k, tp)
        ok = marg > BOUNDARY
        assert ok.mean() > 0.99
        np.testing.assert_array_equal(got[ok] > 0, want[ok] > 0)
        np.testing.assert_allclose(got[ok], want[ok], rtol=1e-5, atol=1e-6)


def test_top_p_crossing_in_the_far_tail():
    # one dominant token and a long tail of tokens below 2^-24 of it: for top_p close to 1
    # the crossing falls among the tail's weights (the streaming histogram leaves those out
    # and hands such rows to the general path); smaller top_p keeps the head alone
    rng = np.random.default_rng(31)
    B, D, V = 4, 1, 131072
    R = D + 1
    x = (rng.standard_normal((B * R, V)) * 0.1 - 18.0).astype(np.float32)
    x[:, 5] = 0.0
    x[:, 77] = -2.0
    T = np.ones(B, np.float32)
    tp = np.array([0.999, 0.9999, 0.5, 0.99], np.float32)
    k = np.zeros(B, np.int32)
    drafts = np.full((B, D), 77, np.int32)
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64)
    g = tv.chain_spec_sampling(dev(x), True, D, dev(drafts), temperature=dev(T), top_k=dev(k),
                               top_p=dev(tp), seed=dev(seed), offset=dev(off))
    ref = oracle.chain_spec_sampling(x, True, D, drafts, temperature=T, top_k=k, top_p=tp,
                                     seed=seed, offset=off)
    compare_chain(g, ref, "f32")
    # the same rows as probabilities through the renorm call
    p = oracle.softmax_temp(x).astype(np.float32)
    tpr = np.repeat(tp, R)
    got = tv.topk_topp_renorm(dev(p), None, dev(tpr)).cpu().numpy()
    want, marg = oracle.topk_topp_renorm(p, None, tpr)
    ok = marg > BOUNDARY
    assert ok.sum() == 4  # top_p 0.5 and 0.99 keep the head alone
    np.testing.assert_array_equal(got[ok] > 0, want[ok] > 0)
    np.testing.assert_allclose(got[ok], want[ok], rtol=1e-5, atol=1e-6)
    # a crossing among near-equal tail weights is a boundary case: the kept set is still a
    # prefix of the (value desc, index asc) order, of about the oracle's size
    for r in np.flatnonzero(~ok):
        order = np.lexsort((np.arange(V), -p[r]))
        m = int((got[r] > 0).sum())
        assert (got[r][order[:m]] > 0).all()
        assert abs(m - int((want[r] > 0).sum())) <= V // 100
        np.testing.assert_allclose(got[r].sum(), 1.0, rtol=1e-5)


def test_target_only_explicit_uniforms_and_knobs_off():
    rng = np.random.default_rng(77)
    B, D, V = 40, 3, 5000
    R = D + 1
    d = _rand_logits(rng, B * R, V, "f32", sigma=1.0, zipf=False)
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    uni = rng.uniform(0.001, 0.999, (B, R)).astype(np.float32)
    g = tv.chain_spec_sampling(dev_logits(d), True, D, dev(drafts), uniforms=dev(uni))
    ref = oracle.chain_spec_sampling(d["logits"], True, D, drafts, uniforms=uni)
    compare_chain(g, ref, "f32")


def test_determinism_bitwise():
    rng = np.random.default_rng(5)
    B, D, V = 32, 4, 128256
    d = _rand_logits(rng, B * (D + 1), V, "bf16")
    T = rng.uniform(0.5, 1.2, B).astype(np.float32)
    k = rng.choice(np.array(synth.TOPK_CHOICES, np.int32), B).astype(np.int32)
    tp = rng.choice(np.array(synth.TOPP_CHOICES, np.float32), B).astype(np.float32)
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    args = (dev_logits(d), True, D, dev(drafts))
    kw = dict(temperature=dev(T), top_k=dev(k), top_p=dev(tp),
              seed=dev(synth.request_seeds(B)), offset=dev(np.arange(B)))
    a = tv.chain_spec_sampling(*args, **kw)
    b = tv.chain_spec_sampling(*args, **kw)
    for key in ("accepted_tokens", "accept_length", "logprobs"):
        assert torch.equal(a[key], b[key])


# ---- Gumbel-max ------------------------------------------------------------------------------

@pytest.mark.parametrize("B,N,V,dtype", [(4, 4, 1024, "f32"), (16, 4, 32000, "bf16"),
                                         (2, 4, 201088, "bf16"), (3, 2, 13, "f32")])
def test_gumbel(B, N, V, dtype):
    rng = np.random.default_rng(B + N + V)
    d = _rand_logits(rng, B * N, V, dtype)
    if V > 100:
        d["logits"][:, V - 50:] = -np.inf
        if dtype == "bf16":
            d["logits_bits"][:, V - 50:] = 0xFF80
    T = np.repeat(rng.uniform(0.3, 1.5, B), N).astype(np.float32)
    T[:N] = 0.0
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64)
    got = tv.gumbel_max_sample(dev_logits(d), N, dev(T), dev(seed), dev(off)).cpu().numpy()
    ref, marg = oracle.gumbel_max_sample(d["logits"], N, T, seed, off)
    ok = marg > BOUNDARY
    assert (~ok).sum() <= 1
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert (got < V - 50).all() or V <= 100


def _strided(t, ld):
    """A copy of the 2-D tensor t in rows of ld elements (the first t.shape[1] hold t)."""
    buf = torch.full((t.shape[0], ld), float("-inf"), dtype=t.dtype, device=t.device)
    buf[:, :t.shape[1]] = t
    return buf[:, :t.shape[1]]


@pytest.mark.parametrize("B,N,V,dtype,ld", [(8, 4, 8195, "bf16", 8200), (5, 3, 50001, "f32", 50004),
                                            (1, 4, 32000, "bf16", 32000),
                                            (64, 4, 4099, "f32", 4100),
                                            (3, 4, 200003, "bf16", 200008),
                                            (2, 1, 5, "bf16", 8)])
def test_gumbel_chunked(B, N, V, dtype, ld):
    """The chunked kernel (16-byte aligned rows, ragged tails, few and many chunks a row)
    against the oracle, and token for token equal to the per-split route that serves
    unaligned rows: the two compute the same scores, so every row must agree, boundary
    rows included. Rows with ties, an all -inf row and greedy rows are in the mix."""
    rng = np.random.default_rng(B * 7 + V)
    d = _rand_logits(rng, B * N, V, dtype)
    x = d["logits"]
    if V > 64:
        x[0] = np.float32(1.5)  # every logit equal
        x[1, V // 3:] = -np.inf
    if B * N > 3:
        x[3] = -np.inf
    if dtype == "bf16":
        d["logits_bits"] = synth.bf16_bits_from_f32(x)
        d["logits"] = x = synth.f32_from_bf16_bits(d["logits_bits"])
    T = np.repeat(rng.uniform(0.3, 1.5, B), N).astype(np.float32)
    if B > 1:
        T[N:2 * N] = 0.0
    seed = synth.request_seeds(B)
    off = (np.arange(B, dtype=np.int64) + (1 << 33)).astype(np.int64)
    t = dev_logits(d)
    aligned = _strided(t, ld)
    unaligned = _strided(t, ld + 1)
    args = (N, dev(T), dev(seed), dev(off))
    got = tv.gumbel_max_sample(aligned, *args).cpu().numpy()
    alt = tv.gumbel_max_sample(unaligned, *args).cpu().numpy()
    np.testing.assert_array_equal(got, alt)
    ref, marg = oracle.gumbel_max_sample(x, N, T, seed, off)
    ok = marg > BOUNDARY
    assert (~ok).sum() <= 1
    np.testing.assert_array_equal(got[ok], ref[ok])
    if B * N > 3:
        assert got[3] == 0  # no finite logit: token 0


# ---- argument validation through the ABI (no launch) --------------------------------------------

def test_invalid_arguments_raise():
    x = torch.zeros((4, 10), device="cuda")
    with pytest.raises(tv.TsError):
        tv.verify_chain_greedy(x, 65, torch.zeros((1, 65), dtype=torch.int32, device="cuda"))
    with pytest.raises(tv.TsError):
        tv.chain_spec_sampling(x, True, 1, torch.zeros((2, 1), dtype=torch.int32, device="cuda"))
    with pytest.raises(tv.TsError):
        tv.gather_logprobs(x.to(torch.bfloat16), torch.zeros(4, dtype=torch.int32, device="cuda"),
                           is_probs=True)


# ---- routes of the cluster-staged selection ------------------------------------------------

def _route_rows(V, dtype, rng):
    """Rows that send the selection down each route: ordinary, all-equal (ties swamp the
    candidate lists: general path), flat high-temperature (large nucleus), spiky."""
    x = rng.standard_normal((8, V), dtype=np.float32) * np.float32(3.0)
    x += synth.zipf_bias(V)[None, :]
    x[1] = 0.5                                   # all equal
    x[2] = rng.integers(-2, 2, V).astype(np.float32)  # few distinct values, many ties
    x[3] *= np.float32(0.05)                     # nearly flat
    x[4, 100:200] = 30.0                         # a block of equal maxima
    if dtype == "bf16":
        bits = synth.bf16_bits_from_f32(x)
        return dict(dtype="bf16", logits_bits=bits, logits=synth.f32_from_bf16_bits(bits))
    return dict(dtype="f32", logits=x)


@pytest.mark.parametrize("V,dtype", [(32000, "bf16"), (201088, "bf16"), (60000, "f32")])
@pytest.mark.parametrize("k,p,T", [(1, 1.0, 1.0), (50, 1.0, 0.7), (1000, 0.9, 1.5),
                                   (3000, 1.0, 1.0), (0, 0.95, 1.5), (0, 0.5, 0.3),
                                   (0, 0.0, 1.0), (7, 0.0, 1.0), (0, 1.0, 1.2),
                                   (64, 1.0, 1.0), (100, 0.9, 0.8), (128, 1.0, 1.3),
                                   (129, 0.95, 1.0), (500, 1.0, 0.6)])
def test_selection_routes(V, dtype, k, p, T):
    rng = np.random.default_rng(V + k + int(100 * p))
    d = _route_rows(V, dtype, rng)
    B, D = 2, 3
    R = D + 1
    drafts = rng.integers(0, V, (B, D)).astype(np.int32)
    drafts[0, :] = d["logits"][:3].argmax(-1)
    uni = rng.uniform(0.01, 0.99, (B, R)).astype(np.float32)
    kw = dict(temperature=np.full(B, T, np.float32), top_k=np.full(B, k, np.int32),
              top_p=np.full(B, p, np.float32))
    g = tv.chain_spec_sampling(dev_logits(d), True, D, dev(drafts), uniforms=dev(uni),
                               **{a: dev(b) for a, b in kw.items()})
    ref = oracle.chain_spec_sampling(d["logits"], True, D, drafts, uniforms=uni, **kw)
    compare_chain(g, ref, dtype)
    # the same rows as probabilities through the renorm call
    pr = oracle.softmax_temp(d["logits"], np.full(8, T, np.float32)).astype(np.float32)
    got = tv.topk_topp_renorm(dev(pr), dev(np.full(8, k, np.int32)),
                              dev(np.full(8, p, np.float32))).cpu().numpy()
    want, marg = oracle.topk_topp_renorm(pr, np.full(8, k, np.int32), np.full(8, p, np.float32))
    ok = marg > BOUNDARY
    np.testing.assert_array_equal(got[ok] > 0, want[ok] > 0)
    np.testing.assert_allclose(got[ok], want[ok], rtol=1e-5, atol=1e-6)


# ---- logits with explicit draft probabilities --------------------------------------------

def _draws(rng, q):
    """One draw per row of q (input preparation: the drafts are sampled from q)."""
    c = np.cumsum(q.astype(np.float64), axis=-1)
    u = rng.random(c.shape[0]) * c[:, -1]
    return np.minimum((c < u[:, None]).sum(-1), q.shape[-1] - 1).astype(np.int32)


@pytest.mark.parametrize("B,D,V,dtype", [(4, 3, 1024, "f32"), (32, 3, 50000, "bf16"),
                                         (16, 7, 151936, "f32"), (24, 2, 8195, "bf16")])
def test_logits_with_draft_probs(B, D, V, dtype):
    # the target distribution is the filtered softmax of the logits (temperature, top-k,
    # top-p); drafts are drawn from q, the softmax of noisy target logits; the accept test
    # uses q(x) and a rejected row draws from norm(max(p'' - q, 0))
    rng = np.random.default_rng(B * 7 + V)
    R = D + 1
    d = _rand_logits(rng, B * R, V, dtype, sigma=2.5, zipf=V > 2000)
    lg = d["logits"].reshape(B, R, V)[:, :D].astype(np.float64)
    noisy = lg + rng.standard_normal(lg.shape) * 0.7
    e = np.exp(noisy - noisy.max(-1, keepdims=True))
    q = (e / e.sum(-1, keepdims=True)).astype(np.float32)
    drafts = _draws(rng, q.reshape(B * D, V)).reshape(B, D)
    T = rng.choice(np.array([0.0, 0.7, 1.0, 1.3], np.float32), B)
    k = rng.choice(np.array([0, 20, 500], np.int32), B).astype(np.int32)
    tp = rng.choice(np.array([1.0, 0.9], np.float32), B).astype(np.float32)
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64)
    x = dev_logits(d)
    if V % 8:  # a ragged vocabulary in rows padded to 16-byte multiples (the kernel's route)
        ld = (V + 7) // 8 * 8
        full = torch.zeros((B * R, ld), dtype=x.dtype, device=x.device)
        full[:, :V] = x
        x = full[:, :V]
    g = tv.chain_spec_sampling(x, True, D, dev(drafts), draft_probs=dev(q),
                               temperature=dev(T), top_k=dev(k), top_p=dev(tp), seed=dev(seed),
                               offset=dev(off), logprobs=True)
    ref = oracle.chain_spec_sampling(d["logits"], True, D, drafts, draft_probs=q, temperature=T,
                                     top_k=k, top_p=tp, seed=seed, offset=off)
    compare_chain(g, ref, dtype)
    # both outcomes occur: some requests reject before their last row (the residual draw)
    alen = g["accept_length"].cpu().numpy()
    assert (alen <= D).any()


def test_logits_with_draft_probs_unaligned_rows_are_refused():
    V, D, B = 1001, 2, 3
    x = torch.zeros((B * (D + 1), V + 1), dtype=torch.bfloat16, device="cuda")[:, :V]
    q = torch.full((B * D, V), 1.0 / V, device="cuda")
    drafts = torch.zeros((B, D), dtype=torch.int32, device="cuda")
    seed = torch.zeros(B, dtype=torch.int64, device="cuda")
    with pytest.raises(tv.TsError) as e:
        tv.chain_spec_sampling(x, True, D, drafts, draft_probs=q, seed=seed, offset=seed)
    assert e.value.status == 1
