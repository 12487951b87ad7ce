"""GPU parity on the method's edge cases: the longest chain (D = 64) for greedy, sampled
and ragged verification; knobs at their degenerate values (top_p = 0 and tiny, top_k = 1
and V - 1, a temperature just above the greedy threshold, min_p = 1); rows with a single
finite logit; a one-token vocabulary; draft tokens outside the vocabulary."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_temp_gb300 import synth
from speculative_decoding_verify_temp_gb300 import tsverify as tv
from tests.gpu_util import BOUNDARY, compare_chain, dev

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


def _bf16(x):
    bits = synth.bf16_bits_from_f32(x)
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    return synth.f32_from_bf16_bits(bits), t


def test_longest_chain_d64():
    rng = np.random.default_rng(64)
    B, D, V = 3, 64, 4096
    R = D + 1
    xf, t = _bf16(rng.standard_normal((B * R, V)).astype(np.float32) * 2)
    am = xf.reshape(B, R, V)[:, :D].argmax(-1)
    drafts = am.astype(np.int32).copy()
    drafts[1, 40] = (drafts[1, 40] + 1) % V  # one rejection deep in the chain
    drafts[2, 0] = V + 5  # an id outside the vocabulary is never accepted
    g = tv.verify_chain_greedy(t, D, dev(drafts))
    gr = oracle.verify_chain_greedy(xf, D, drafts)
    for k in ("accepted_tokens", "accept_length", "accept_index"):
        np.testing.assert_array_equal(g[k].cpu().numpy(), gr[k])
    assert list(gr["accept_length"]) == [65, 41, 1]
    kw = dict(temperature=np.array([0.0, 0.05, 1.0], np.float32),
              top_k=np.array([0, 1, 50], np.int32), top_p=np.array([1.0, 0.9, 0.95], np.float32),
              seed=synth.request_seeds(B), offset=np.arange(B, dtype=np.int64))
    c = tv.chain_spec_sampling(t, True, D, dev(drafts), **{k: dev(v) for k, v in kw.items()})
    cr = oracle.chain_spec_sampling(xf, True, D, drafts, **kw)
    compare_chain(c, cr, "bf16")
    # ragged: windows of 65, 1 and 30 rows
    lens = np.array([65, 1, 30])
    qo = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rows = np.concatenate([np.arange(b * R, b * R + lens[b]) for b in range(B)])
    xr = xf[rows]
    tr = t[torch.from_numpy(rows).cuda()]
    c2 = tv.chain_spec_sampling(tr, True, D, dev(drafts), **{k: dev(v) for k, v in kw.items()},
                                qo_indptr=dev(qo))
    cr2 = oracle.chain_spec_sampling_ragged(xr, True, D, qo, drafts, **kw)
    compare_chain(c2, cr2, "bf16", row_base=qo[:-1])


def test_degenerate_knobs():
    rng = np.random.default_rng(7)
    V = 5000
    rows = 10
    x = rng.standard_normal((rows, V)).astype(np.float32) * 3
    x[3] = -np.inf
    x[3, 1234] = 2.0  # a single finite logit
    x[4, :] = 1.0  # every logit equal
    xf, t = _bf16(x)
    T = np.array([1.0, 1.0, 1.0, 0.7, 0.9, 1.5e-5, 1.0, 0.8, 1.2, 1.0], np.float32)
    k = np.array([0, 1, V - 1, 0, 3, 0, 0, 10, 0, 1], np.int32)
    p = np.array([0.0, 1.0, 1.0, 0.9, 0.5, 0.9, 1e-9, 0.9, 0.95, 0.0], np.float32)
    mp = np.array([0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 1.0, 0.5, 0.0], np.float32)
    seed, off = synth.request_seeds(rows), np.arange(rows, dtype=np.int64)
    for joint in (False, True):
        got = tv.sample_from_logits(t, 1, temperature=dev(T), top_k=dev(k), top_p=dev(p),
                                    min_p=dev(mp), joint=joint, seed=dev(seed), offset=dev(off),
                                    logprobs=True, probs=True)
        ref = oracle.sample_from_logits(xf, 1, temperature=T, top_k=k, top_p=p, min_p=mp,
                                        joint=joint, seed=seed, offset=off, probs=True)
        ok = ref["margin"] > BOUNDARY
        tok = got["tokens"].cpu().numpy()
        np.testing.assert_array_equal(tok[ok], ref["tokens"][ok])
        pr = got["probs"].cpu().numpy()
        np.testing.assert_array_equal(pr[ok] > 0, ref["probs"][ok] > 0)
        np.testing.assert_allclose(pr[ok], ref["probs"][ok], rtol=1e-5, atol=1e-6)
        amx = xf.argmax(1)
        # top_p = 0, top_k = 1, tiny top_p and min_p = 1 (unique maxima) keep only the argmax
        for r in (0, 1, 6, 9):
            assert tok[r] == amx[r]
        assert tok[3] == 1234


def test_single_token_vocabulary():
    x = np.zeros((6, 8), np.float32)  # rows padded to 8 entries (16-byte aligned), V = 1
    x[:, 0] = np.arange(6, dtype=np.float32)
    t = torch.from_numpy(x).cuda()[:, :1]
    seeds = dev(synth.request_seeds(6))
    offs = dev(np.arange(6, dtype=np.int64))
    got = tv.sample_from_logits(t, 1, temperature=dev(np.full(6, 0.7, np.float32)),
                                seed=seeds, offset=offs, logprobs=True)
    assert (got["tokens"].cpu().numpy() == 0).all()
    np.testing.assert_allclose(got["logprobs"].cpu().numpy(), 0.0, atol=1e-6)
    c = tv.chain_spec_sampling(t, True, 1, dev(np.zeros((3, 1), np.int32)),
                               temperature=dev(np.array([0.0, 0.5, 1.0], np.float32)),
                               seed=seeds[:3], offset=offs[:3])
    np.testing.assert_array_equal(c["accept_length"].cpu().numpy(), [2, 2, 2])
    np.testing.assert_array_equal(c["accepted_tokens"].cpu().numpy(), np.zeros((3, 2)))
