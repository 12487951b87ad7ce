"""GPU parity of ragged verification (packed target rows by qo_indptr, each request
verifying its own window) against the oracle: greedy and sampled chains, target-only and
with draft probabilities, explicit and Philox coins, windows that do not fit; full
windows against the rectangular calls; and the largest shape on every request."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_temp_gb300 import synth
from speculative_decoding_verify_temp_gb300 import tsverify as tv
from tests.gpu_util import TOL, compare_chain, dev, oracle_ragged_all

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


def _packed(rng, lens, V, dtype):
    qo = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = rng.standard_normal((int(qo[-1]), V), dtype=np.float32) * np.float32(3.0)
    x += synth.zipf_bias(V)[None, :]
    if dtype == "bf16":
        bits = synth.bf16_bits_from_f32(x)
        xf = synth.f32_from_bf16_bits(bits)
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        xf = x
        t = torch.from_numpy(x).cuda()
    return qo, xf, t


def _drafts(rng, x, qo, D, V):
    B = len(qo) - 1
    am = x.argmax(1)
    d = rng.integers(0, V, (B, D)).astype(np.int32)
    for b in range(B):
        n = min(D, int(qo[b + 1] - qo[b]) - 1)
        take = rng.random(n) < 0.7
        d[b, :n] = np.where(take, am[qo[b]:qo[b] + n], d[b, :n])
    return d


@pytest.mark.parametrize("B,D,V,dtype", [(33, 4, 32000, "bf16"), (12, 3, 5004, "f32"),
                                         (8, 0, 1000, "f32")])
def test_greedy_ragged(B, D, V, dtype):
    rng = np.random.default_rng(B * 31 + V)
    lens = rng.integers(1, D + 2, B)
    qo, x, t = _packed(rng, lens, V, dtype)
    drafts = _drafts(rng, x, qo, D, V)
    got = tv.verify_chain_greedy_ragged(t, D, dev(qo), dev(drafts))
    ref = oracle.verify_chain_greedy_ragged(x, D, qo, drafts)
    for k in ("accepted_tokens", "accept_length", "accept_index"):
        np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k])
    np.testing.assert_allclose(got["logprobs"].cpu().numpy(), ref["logprobs"], **TOL[dtype])


def test_windows_that_do_not_fit():
    rng = np.random.default_rng(9)
    D, V = 2, 4096
    qo = np.array([0, 2, 2, 6, 7], np.int32)  # lengths 2, 0, 4 (> D + 1), 1
    x = rng.standard_normal((7, V), dtype=np.float32)
    t = torch.from_numpy(x).cuda()
    drafts = rng.integers(0, V, (4, D)).astype(np.int32)
    g = tv.verify_chain_greedy_ragged(t, D, dev(qo), dev(drafts))
    ref = oracle.verify_chain_greedy_ragged(x, D, qo, drafts)
    np.testing.assert_array_equal(g["accept_length"].cpu().numpy(), ref["accept_length"])
    np.testing.assert_array_equal(g["accepted_tokens"].cpu().numpy(), ref["accepted_tokens"])
    c = tv.chain_spec_sampling(t, True, D, dev(drafts), seed=dev(synth.request_seeds(4)),
                               offset=dev(np.arange(4)), qo_indptr=dev(qo))
    cref = oracle.chain_spec_sampling_ragged(x, True, D, qo, drafts, seed=synth.request_seeds(4),
                                             offset=np.arange(4))
    np.testing.assert_array_equal(c["accept_length"].cpu().numpy(), cref["accept_length"])
    np.testing.assert_array_equal(c["accepted_tokens"].cpu().numpy()[[1, 2]], -1)


@pytest.mark.parametrize("B,D,V,dtype,use_q,coins", [(40, 4, 32000, "bf16", False, "philox"),
                                                     (24, 3, 50004, "f32", True, "philox"),
                                                     (16, 5, 8192, "bf16", True, "uniforms"),
                                                     (30, 2, 129024, "bf16", False, "uniforms")])
def test_chain_ragged(B, D, V, dtype, use_q, coins):
    rng = np.random.default_rng(B + D + V)
    R = D + 1
    lens = rng.integers(1, R + 1, B)
    qo, x, t = _packed(rng, lens, V, dtype)
    drafts = _drafts(rng, x, qo, D, V)
    T = rng.uniform(0.3, 1.5, B).astype(np.float32)
    T[rng.random(B) < 0.2] = 0.0
    k = rng.choice(np.array(synth.TOPK_CHOICES, np.int32), B).astype(np.int32)
    p = rng.choice(np.array(synth.TOPP_CHOICES, np.float32), B).astype(np.float32)
    q = None
    if use_q:
        q = rng.random((B * D, V)).astype(np.float32) ** 4
        q /= q.sum(1, keepdims=True)
    kw = dict(temperature=T, top_k=k, top_p=p)
    if coins == "philox":
        kw.update(seed=synth.request_seeds(B), offset=np.arange(B, dtype=np.int64) + 17)
    else:
        kw.update(uniforms=rng.uniform(0.001, 0.999, (B, R)).astype(np.float32))
    got = tv.chain_spec_sampling(t, True, D, dev(drafts), draft_probs=dev(q),
                                 **{kk: dev(v) for kk, v in kw.items()}, qo_indptr=dev(qo))
    ref = oracle.chain_spec_sampling_ragged(x, True, D, qo, drafts, draft_probs=q, **kw)
    compare_chain(got, ref, dtype, max_boundary_frac=0.1, row_base=qo[:-1])
    # accept_index: packed row numbers of the emitted positions
    alen = got["accept_length"].cpu().numpy()
    aidx = got["accept_index"].cpu().numpy()
    pos = np.arange(R)[None, :]
    np.testing.assert_array_equal(aidx, np.where(pos < alen[:, None], qo[:-1, None] + pos, -1))


def test_full_windows_equal_rectangular():
    rng = np.random.default_rng(3)
    B, D, V = 20, 3, 32000
    R = D + 1
    qo, x, t = _packed(rng, np.full(B, R), V, "bf16")
    drafts = _drafts(rng, x, qo, D, V)
    kw = dict(temperature=dev(rng.uniform(0.5, 1.2, B).astype(np.float32)),
              top_k=dev(rng.choice([0, 20], B).astype(np.int32)),
              seed=dev(synth.request_seeds(B)), offset=dev(np.arange(B)))
    a = tv.chain_spec_sampling(t, True, D, dev(drafts), **kw)
    b = tv.chain_spec_sampling(t, True, D, dev(drafts), **kw, qo_indptr=dev(qo))
    for k in ("accepted_tokens", "accept_length", "accept_index", "logprobs"):
        assert torch.equal(a[k], b[k]), k
    g = tv.verify_chain_greedy(t, D, dev(drafts))
    gr = tv.verify_chain_greedy_ragged(t, D, dev(qo), dev(drafts))
    for k in ("accepted_tokens", "accept_length", "accept_index", "logprobs"):
        assert torch.equal(g[k], gr[k]), k


def test_ragged_fullsize():
    """512 requests with windows of 1 to 4 rows of 201088 bf16 logits (the verify step's
    knob mix): every request against the oracle."""
    d = synth.verify_step(B=512, D=3, V=201088, real_vocab=200019)
    B, D, V = 512, 3, 201088
    rng = np.random.default_rng(512)
    lens = rng.integers(1, D + 2, B)
    qo = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    # request b's window: the first lens[b] rows of its rectangular rows
    rows = np.concatenate([np.arange(b * 4, b * 4 + lens[b]) for b in range(B)])
    bits = np.ascontiguousarray(d["logits_bits"][rows])
    t = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    kn = {k: d[k] for k in ("temperature", "top_k", "top_p", "seed", "offset")}
    got = tv.chain_spec_sampling(t, True, D, dev(d["draft_tokens"]),
                                 **{k: dev(v) for k, v in kn.items()}, qo_indptr=dev(qo))
    ref = oracle_ragged_all("chain_spec_sampling_ragged", bits, True, D, qo, args=(True,),
                            per_request=dict(kn, draft_tokens=d["draft_tokens"]))
    nb = compare_chain(got, ref, "bf16", max_boundary_frac=0.05, row_base=qo[:-1])
    print(f"\nragged B={B} rows={int(qo[-1])} V={V}: {B} requests checked, {nb} boundary")
