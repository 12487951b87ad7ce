"""GPU parity at the benchmark configurations' full sizes, in the launch configuration
bench.py times (the same calls, workspaces and outputs). Every output is checked against
the invariants of the method; a sample of requests (or rows) covering every knob kind is
checked against the oracle, computed for those requests alone (the method is per
request: coins come from each request's own seed and offset)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_temp_gb300 import synth
from speculative_decoding_verify_temp_gb300 import tsverify as tv
from tests.gpu_util import BOUNDARY, TOL, compare_chain, dev

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


@pytest.fixture(scope="module")
def step():
    """The largest verify step (B=512, D=3, V=201088 bf16) with the bench's knob mix."""
    d = synth.verify_step(B=512, D=3, V=201088, real_vocab=200019)
    bits = np.ascontiguousarray(d["logits_bits"]).view(np.int16)
    d["dev_logits"] = torch.from_numpy(bits).cuda().view(torch.bfloat16)
    return d


def _rows_f32(d, reqs, R):
    """fp32 logits of the rows of the given requests (widened from the bf16 bits)."""
    rows = np.concatenate([np.arange(b * R, (b + 1) * R) for b in reqs])
    return synth.f32_from_bf16_bits(np.ascontiguousarray(d["logits_bits"][rows])), rows


def _sample(d, per_kind=5, seed=0):
    """Requests of every kind: greedy, no knobs, top-p alone, small top-k, large top-k."""
    T, k, p = d["temperature"], d["top_k"], d["top_p"]
    kinds = [T < 1e-5,
             (T >= 1e-5) & (k == 0) & (p >= 1),
             (T >= 1e-5) & (k == 0) & (p < 1),
             (T >= 1e-5) & (k > 0) & (k <= 256),
             (T >= 1e-5) & (k > 256)]
    rng = np.random.default_rng(seed)
    out = []
    for m in kinds:  # (a workload may have no request of a kind)
        idx = np.flatnonzero(m)
        if len(idx):
            out.extend(rng.choice(idx, min(per_kind, len(idx)), replace=False).tolist())
    assert len(out) >= per_kind
    return np.array(sorted(out))


def _chain_invariants(acc, alen, drafts, D, V):
    R = D + 1
    assert alen.min() >= 1 and alen.max() <= R
    pos = np.arange(R)[None, :]
    emitted = pos < alen[:, None]
    assert ((acc >= 0) == emitted).all()
    assert (acc[emitted] < V).all()
    # the accepted drafts precede the target token
    for L in range(2, R + 1):
        m = alen == L
        np.testing.assert_array_equal(acc[m, :L - 1], drafts[m, :L - 1])


def test_verify_step_fullsize(step):
    d = step
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    kw = dict(temperature=dev(d["temperature"]), top_k=dev(d["top_k"]), top_p=dev(d["top_p"]),
              seed=dev(d["seed"]), offset=dev(d["offset"]),
              workspace=tv.make_workspace(B, R, V, torch.device("cuda")),
              outputs=tv._chain_outputs(B, R, torch.device("cuda"), False, False))
    g = tv.chain_spec_sampling(d["dev_logits"], True, D, dev(d["draft_tokens"]), **kw)
    acc = g["accepted_tokens"].cpu().numpy()
    alen = g["accept_length"].cpu().numpy()
    _chain_invariants(acc, alen, d["draft_tokens"], D, V)
    # a second call on the same workspace gives the same bits
    g2 = tv.chain_spec_sampling(d["dev_logits"], True, D, dev(d["draft_tokens"]), **kw)
    np.testing.assert_array_equal(g2["accepted_tokens"].cpu().numpy(), acc)
    reqs = _sample(d)
    x, _ = _rows_f32(d, reqs, R)
    ref = oracle.chain_spec_sampling(x, True, D, d["draft_tokens"][reqs],
                                     temperature=d["temperature"][reqs], top_k=d["top_k"][reqs],
                                     top_p=d["top_p"][reqs], seed=d["seed"][reqs],
                                     offset=d["offset"][reqs], logprobs=False)
    sub = {"accepted_tokens": torch.from_numpy(acc[reqs]),
           "accept_length": torch.from_numpy(alen[reqs])}
    compare_chain(sub, ref, "bf16", max_boundary_frac=0.1, check_logprobs=False)


def test_greedy_verify_fullsize(step):
    d = step
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    g = tv.verify_chain_greedy(d["dev_logits"], D, dev(d["draft_tokens"]),
                               tv.make_workspace(B, R, V, torch.device("cuda")))
    acc = g["accepted_tokens"].cpu().numpy()
    alen = g["accept_length"].cpu().numpy()
    _chain_invariants(acc, alen, d["draft_tokens"], D, V)
    reqs = np.arange(0, B, 17)
    x, _ = _rows_f32(d, reqs, R)
    ref = oracle.verify_chain_greedy(x, D, d["draft_tokens"][reqs])
    np.testing.assert_array_equal(alen[reqs], ref["accept_length"])
    np.testing.assert_array_equal(acc[reqs], ref["accepted_tokens"])
    np.testing.assert_allclose(g["logprobs"].cpu().numpy()[reqs], ref["logprobs"], **TOL["bf16"])


def test_gumbel_fullsize(step):
    d = step
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    Trow = np.repeat(d["temperature"], R).astype(np.float32)
    tok = tv.gumbel_max_sample(d["dev_logits"], R, dev(Trow), dev(d["seed"]), dev(d["offset"]),
                               tv.make_workspace(B, R, V, torch.device("cuda"))).cpu().numpy()
    assert ((tok >= 0) & (tok < d["real_vocab"])).all()  # -inf pads never win
    reqs = np.arange(3, B, 41)
    x, rows = _rows_f32(d, reqs, R)
    want, marg = oracle.gumbel_max_sample(x, R, Trow[rows], d["seed"][reqs], d["offset"][reqs])
    ok = marg > BOUNDARY
    np.testing.assert_array_equal(tok[rows][ok], want[ok])


def test_softmax_fullsize(step):
    d = step
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    Trow = np.repeat(d["temperature"], R).astype(np.float32)
    out = tv.softmax_temp(d["dev_logits"], dev(Trow))
    rows = np.arange(5, B * R, 257)
    got = out[torch.from_numpy(rows).cuda()].cpu().numpy()
    del out
    x = synth.f32_from_bf16_bits(np.ascontiguousarray(d["logits_bits"][rows]))
    want = oracle.softmax_temp(x, Trow[rows])
    np.testing.assert_allclose(got, want, **TOL["f32"])


def test_target_only_leg_fullsize():
    c = synth.target_only()
    B, D, V = c["B"], c["D"], c["V"]
    R = D + 1
    bits = np.ascontiguousarray(c["logits_bits"]).view(np.int16)
    cl = torch.from_numpy(bits).cuda().view(torch.bfloat16)
    g = tv.chain_spec_sampling(cl, True, D, dev(c["draft_tokens"]),
                               temperature=dev(c["temperature"]), top_k=dev(c["top_k"]),
                               top_p=dev(c["top_p"]), seed=dev(c["seed"]),
                               offset=dev(c["offset"]),
                               workspace=tv.make_workspace(B, R, V, torch.device("cuda")),
                               outputs=tv._chain_outputs(B, R, torch.device("cuda"), False, False))
    acc = g["accepted_tokens"].cpu().numpy()
    alen = g["accept_length"].cpu().numpy()
    _chain_invariants(acc, alen, c["draft_tokens"], D, V)
    reqs = _sample(c, per_kind=4, seed=1)
    x, _ = _rows_f32(c, reqs, R)
    ref = oracle.chain_spec_sampling(x, True, D, c["draft_tokens"][reqs],
                                     temperature=c["temperature"][reqs], top_k=c["top_k"][reqs],
                                     top_p=c["top_p"][reqs], seed=c["seed"][reqs],
                                     offset=c["offset"][reqs], logprobs=False)
    sub = {"accepted_tokens": torch.from_numpy(acc[reqs]),
           "accept_length": torch.from_numpy(alen[reqs])}
    compare_chain(sub, ref, "bf16", max_boundary_frac=0.1, check_logprobs=False)


def test_rejection_and_renorm_legs_fullsize():
    r = synth.rejection()
    B, D, V = r["B"], r["D"], r["V"]
    R = D + 1
    rp = torch.from_numpy(r["target_probs"]).cuda()
    rq = torch.from_numpy(r["draft_probs"]).cuda()
    g = tv.chain_spec_sampling(rp, False, D, dev(r["draft_tokens"]), draft_probs=rq,
                               seed=dev(r["seed"]), offset=dev(r["offset"]),
                               workspace=tv.make_workspace(B, R, V, torch.device("cuda")),
                               outputs=tv._chain_outputs(B, R, torch.device("cuda"), False, True))
    acc = g["accepted_tokens"].cpu().numpy()
    alen = g["accept_length"].cpu().numpy()
    _chain_invariants(acc, alen, r["draft_tokens"], D, V)
    reqs = np.arange(0, B, 23)
    rows = np.concatenate([np.arange(b * R, (b + 1) * R) for b in reqs])
    qrows = np.concatenate([np.arange(b * D, (b + 1) * D) for b in reqs])
    q2 = r["draft_probs"].reshape(B * D, V)
    ref = oracle.chain_spec_sampling(r["target_probs"][rows], False, D, r["draft_tokens"][reqs],
                                     draft_probs=q2[qrows], seed=r["seed"][reqs],
                                     offset=r["offset"][reqs])
    sub = {"accepted_tokens": torch.from_numpy(acc[reqs]),
           "accept_length": torch.from_numpy(alen[reqs]),
           "logprobs": g["logprobs"][torch.from_numpy(reqs).cuda()]}
    compare_chain(sub, ref, "f32", max_boundary_frac=0.1)
    # the renorm leg: the same probabilities with the target-only knob mix
    rrows = B * R
    rng = np.random.default_rng(1)
    kk = rng.choice(np.array(synth.TOPK_CHOICES, np.int32), rrows).astype(np.int32)
    pp = rng.choice(np.array(synth.TOPP_CHOICES, np.float32), rrows).astype(np.float32)
    out = tv.topk_topp_renorm(rp, dev(kk), dev(pp))
    srows = np.arange(7, rrows, 97)
    got = out[torch.from_numpy(srows).cuda()].cpu().numpy()
    want, marg = oracle.topk_topp_renorm(r["target_probs"][srows], kk[srows], pp[srows])
    ok = marg > BOUNDARY
    np.testing.assert_array_equal(got[ok] > 0, want[ok] > 0)
    np.testing.assert_allclose(got[ok], want[ok], **TOL["f32"])
