"""GPU parity at the benchmark configurations' full sizes, in the launch configuration
bench.py times (the same calls, workspaces and outputs). Every request of every chain
launch (and every Gumbel row) is checked against the oracle, which runs over the host
cores in slices of requests (the method is per request: coins come from each request's
own seed and offset); logprobs are on. The softmax and renorm legs, whose outputs are
whole rows of probabilities, are checked on a sample of rows. Boundary requests (a
decision within 1e-6 of flipping) are counted and printed, not failed."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_temp_gb300 import synth
from speculative_decoding_verify_temp_gb300 import tsverify as tv
from tests.gpu_util import BOUNDARY, TOL, compare_chain, dev, oracle_all

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
    kn = dict(temperature=dev(d["temperature"]), top_k=dev(d["top_k"]), top_p=dev(d["top_p"]),
              seed=dev(d["seed"]), offset=dev(d["offset"]))
    ws = tv.make_workspace(B, R, V, torch.device("cuda"))
    # the bench's call (no logprobs, no accept_index) ...
    g0 = tv.chain_spec_sampling(d["dev_logits"], True, D, dev(d["draft_tokens"]), **kn,
                                workspace=ws,
                                outputs=tv._chain_outputs(B, R, torch.device("cuda"), False, False))
    acc0 = g0["accepted_tokens"].cpu().numpy()
    alen0 = g0["accept_length"].cpu().numpy()
    _chain_invariants(acc0, alen0, d["draft_tokens"], D, V)
    # ... and the same call with every output on: the same decisions, on the same workspace
    g = tv.chain_spec_sampling(d["dev_logits"], True, D, dev(d["draft_tokens"]), **kn,
                               workspace=ws, logprobs=True)
    np.testing.assert_array_equal(g["accepted_tokens"].cpu().numpy(), acc0)
    np.testing.assert_array_equal(g["accept_length"].cpu().numpy(), alen0)
    ref = oracle_all("chain_spec_sampling", d["logits_bits"], True, R,
                     args=[(True, None), (D, None), (d["draft_tokens"], "req")],
                     per_request=dict(temperature=d["temperature"], top_k=d["top_k"],
                                      top_p=d["top_p"], seed=d["seed"], offset=d["offset"]))
    nb = compare_chain(g, ref, "bf16", max_boundary_frac=0.05)
    print(f"\nverify step B={B} D={D} V={V}: {B} requests checked, {nb} boundary")


def test_greedy_verify_fullsize(step):
    d = step
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    g = tv.verify_chain_greedy(d["dev_logits"], D, dev(d["draft_tokens"]),
                               tv.make_workspace(B, R, V, torch.device("cuda")))
    acc = g["accepted_tokens"].cpu().numpy()
    alen = g["accept_length"].cpu().numpy()
    _chain_invariants(acc, alen, d["draft_tokens"], D, V)
    ref = oracle_all("verify_chain_greedy", d["logits_bits"], True, R,
                     args=[(D, None), (d["draft_tokens"], "req")])
    np.testing.assert_array_equal(alen, ref["accept_length"])
    np.testing.assert_array_equal(acc, ref["accepted_tokens"])
    np.testing.assert_allclose(g["logprobs"].cpu().numpy(), ref["logprobs"], **TOL["bf16"])


def test_gumbel_fullsize(step):
    d = step
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    Trow = np.repeat(d["temperature"], R).astype(np.float32)
    tok = tv.gumbel_max_sample(d["dev_logits"], R, dev(Trow), dev(d["seed"]), dev(d["offset"]),
                               tv.make_workspace(B, R, V, torch.device("cuda"))).cpu().numpy()
    assert ((tok >= 0) & (tok < d["real_vocab"])).all()  # -inf pads never win
    want, marg = oracle_all("gumbel_max_sample", d["logits_bits"], True, R,
                            args=[(R, None), (Trow, "row"), (d["seed"], "req"),
                                  (d["offset"], "req")])
    ok = marg > BOUNDARY
    np.testing.assert_array_equal(tok[ok], want[ok])
    print(f"\nGumbel B={B} N={R} V={V}: {B * R} rows checked, {int((~ok).sum())} boundary")


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
                               logprobs=True)
    acc = g["accepted_tokens"].cpu().numpy()
    alen = g["accept_length"].cpu().numpy()
    _chain_invariants(acc, alen, c["draft_tokens"], D, V)
    ref = oracle_all("chain_spec_sampling", c["logits_bits"], True, R,
                     args=[(True, None), (D, None), (c["draft_tokens"], "req")],
                     per_request=dict(temperature=c["temperature"], top_k=c["top_k"],
                                      top_p=c["top_p"], seed=c["seed"], offset=c["offset"]))
    nb = compare_chain(g, ref, "bf16", max_boundary_frac=0.05)
    print(f"\ntarget-only B={B} D={D} V={V}: {B} requests checked, {nb} boundary")


def test_rejection_and_renorm_legs_fullsize():
    r = synth.rejection()
    B, D, V = r["B"], r["D"], r["V"]
    R = D + 1
    rp = torch.from_numpy(r["target_probs"]).cuda()
    rq = torch.from_numpy(r["draft_probs"]).cuda()
    g = tv.chain_spec_sampling(rp, False, D, dev(r["draft_tokens"]), draft_probs=rq,
                               seed=dev(r["seed"]), offset=dev(r["offset"]),
                               workspace=tv.make_workspace(B, R, V, torch.device("cuda")),
                               outputs=tv._chain_outputs(B, R, torch.device("cuda"), True, True))
    acc = g["accepted_tokens"].cpu().numpy()
    alen = g["accept_length"].cpu().numpy()
    _chain_invariants(acc, alen, r["draft_tokens"], D, V)
    ref = oracle_all("chain_spec_sampling", r["target_probs"], False, R,
                     args=[(False, None), (D, None), (r["draft_tokens"], "req")],
                     per_request=dict(draft_probs=r["draft_probs"], seed=r["seed"],
                                      offset=r["offset"]))
    # the residual draws here are over 151936 tokens of nearly flat mass: a coin lands
    # within 1e-6 of one of their CDF edges for several percent of the requests
    nb = compare_chain(g, ref, "f32", max_boundary_frac=0.15)
    print(f"\nrejection B={B} D={D} V={V}: {B} requests checked, {nb} boundary")
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
