"""GPU parity of the single-step sampler (joint and top-k-first filter orders, min_p,
the kept distributions written to scattered rows) and of chain sampling with min_p and
relaxed acceptance thresholds, against the oracle; and the argument checks of both."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_temp_gb300 import synth
from speculative_decoding_verify_temp_gb300 import tsverify as tv
from tests.gpu_util import BOUNDARY, TOL, compare_chain, dev, dev_logits, oracle_all

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


def _rows(rng, rows, V, dtype, ld=None):
    x = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(3.0)
    x += synth.zipf_bias(V)[None, :]
    x[1 % rows, : V // 2] = np.float32(0.25)  # ties
    if dtype == "bf16":
        bits = synth.bf16_bits_from_f32(x)
        d = dict(dtype="bf16", logits_bits=bits, logits=synth.f32_from_bf16_bits(bits))
    else:
        d = dict(dtype="f32", logits=x)
    t = dev_logits(d)
    if ld is not None and ld != V:
        buf = torch.zeros((rows, ld), dtype=t.dtype, device="cuda")
        buf[:, :V] = t
        t = buf[:, :V]
    return d, t


def _knobs(rng, rows, with_min_p):
    T = rng.uniform(0.3, 1.5, rows).astype(np.float32)
    T[rng.random(rows) < 0.2] = 0.0
    k = rng.choice(np.array([0, 1, 20, 50, 100, 300, 1000, 5000], np.int32), rows).astype(np.int32)
    p = rng.choice(np.array([1.0, 0.95, 0.9, 0.5], np.float32), rows).astype(np.float32)
    mp = None
    if with_min_p:
        mp = rng.choice(np.array([0.0, 0.01, 0.1, 0.5], np.float32), rows).astype(np.float32)
    return T, k, p, mp


@pytest.mark.parametrize("B,n,V,dtype,joint,with_min_p",
                         [(24, 1, 32000, "bf16", True, False),
                          (24, 1, 32000, "bf16", False, False),
                          (9, 3, 50007, "f32", True, True),
                          (16, 2, 4099, "bf16", False, True),
                          (3, 4, 151936, "f32", True, False)])
def test_sample_from_logits(B, n, V, dtype, joint, with_min_p):
    rng = np.random.default_rng(B * 100 + V + joint)
    rows = B * n
    ld = (V + 7) // 8 * 8
    d, t = _rows(rng, rows, V, dtype, ld)
    T, k, p, mp = _knobs(rng, rows, with_min_p)
    seed = synth.request_seeds(B)
    off = np.arange(B, dtype=np.int64) + (5 << 32)
    got = tv.sample_from_logits(t, n, temperature=dev(T), top_k=dev(k), top_p=dev(p),
                                min_p=dev(mp), joint=joint, seed=dev(seed), offset=dev(off),
                                logprobs=True)
    ref = oracle.sample_from_logits(d["logits"], n, temperature=T, top_k=k, top_p=p, min_p=mp,
                                    joint=joint, seed=seed, offset=off)
    ok = ref["margin"] > BOUNDARY
    assert (~ok).sum() <= max(2, rows // 20)
    tok = got["tokens"].cpu().numpy()
    np.testing.assert_array_equal(tok[ok], ref["tokens"][ok])
    np.testing.assert_allclose(got["logprobs"].cpu().numpy()[ok], ref["logprobs"][ok],
                               **TOL[dtype])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sample_probs_to_scattered_rows(dtype):
    """The kept distributions land at the rows probs_row names (a slot-indexed buffer,
    as draft-side sampling stores them for the next verify step); the other rows of the
    buffer are untouched; explicit coins replace Philox."""
    rng = np.random.default_rng(77)
    B, n, V = 6, 2, 20000
    rows = B * n
    d, t = _rows(rng, rows, V, dtype)
    T, k, p, mp = _knobs(rng, rows, True)
    u = rng.random(rows).astype(np.float32)
    slots = rng.permutation(3 * rows)[:rows].astype(np.int64)
    buf = torch.full((3 * rows, V + 3), 7.0, dtype=torch.float32, device="cuda")
    got = tv.sample_from_logits(t, n, temperature=dev(T), top_k=dev(k), top_p=dev(p),
                                min_p=dev(mp), joint=False, uniforms=dev(u), probs=buf,
                                probs_row=dev(slots))
    ref = oracle.sample_from_logits(d["logits"], n, temperature=T, top_k=k, top_p=p, min_p=mp,
                                    uniforms=u, probs=True)
    ok = ref["margin"] > BOUNDARY
    h = buf.cpu().numpy()
    np.testing.assert_array_equal(got["tokens"].cpu().numpy()[ok], ref["tokens"][ok])
    for r in np.flatnonzero(ok):
        row = h[slots[r], :V]
        np.testing.assert_array_equal(row > 0, ref["probs"][r] > 0)
        np.testing.assert_allclose(row, ref["probs"][r], **TOL["f32"])
    untouched = np.setdiff1d(np.arange(3 * rows), slots)
    assert (h[untouched] == 7.0).all()
    assert (h[slots, V:] == 7.0).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chain_min_p_and_relaxed_thresholds(dtype):
    rng = np.random.default_rng(5150)
    B, D, V = 20, 3, 32000
    R = D + 1
    d, t = _rows(rng, B * R, V, dtype)
    T, k, p, mp = _knobs(rng, B, True)
    am = d["logits"].reshape(B, R, V)[:, :D].argmax(-1)
    drafts = np.where(rng.random((B, D)) < 0.6, am, rng.integers(0, V, (B, D))).astype(np.int32)
    kw = dict(temperature=T, top_k=k, top_p=p, min_p=mp, seed=synth.request_seeds(B),
              offset=np.arange(B, dtype=np.int64))
    for ts, ta in [(1.0, 1.0), (0.3, 0.6), (1.0, 0.2)]:
        got = tv.chain_spec_sampling(t, True, D, dev(drafts),
                                     **{k2: dev(v) for k2, v in kw.items()},
                                     threshold_single=ts, threshold_acc=ta)
        ref = oracle.chain_spec_sampling(d["logits"], True, D, drafts, **kw, threshold_single=ts,
                                         threshold_acc=ta)
        compare_chain(got, ref, dtype, max_boundary_frac=0.1)


def test_argument_checks():
    x = torch.zeros((4, 64), device="cuda")
    ones = torch.ones(4, device="cuda")
    seeds = torch.zeros(4, dtype=torch.int64, device="cuda")
    with pytest.raises(tv.TsError):  # thresholds with draft probabilities
        tv.chain_spec_sampling(x, True, 1, torch.zeros((2, 1), dtype=torch.int32, device="cuda"),
                               draft_probs=torch.zeros((2, 64), device="cuda"),
                               seed=seeds[:2], offset=seeds[:2], threshold_acc=0.5)
    with pytest.raises(tv.TsError):  # min_p with probability targets
        tv.chain_spec_sampling(x, False, 1, torch.zeros((2, 1), dtype=torch.int32, device="cuda"),
                               seed=seeds[:2], offset=seeds[:2], min_p=ones[:2])
    with pytest.raises(tv.TsError):  # unaligned rows
        tv.sample_from_logits(torch.zeros((4, 65), device="cuda")[:, :63], 1, seed=seeds,
                              offset=seeds)
    with pytest.raises(tv.TsError):  # vocab above the row kernel's limit
        tv.sample_from_logits(torch.zeros((1, (1 << 18) + 8), device="cuda"), 1, seed=seeds[:1],
                              offset=seeds[:1])


def test_sample_fullsize():
    """The single-step sampler on the largest shape (2048 rows of 201088 bf16 logits, the
    verify step's knob mix, joint order): every row against the oracle."""
    dd = synth.verify_step(B=512, D=3, V=201088, real_vocab=200019)
    rows = 2048
    bits = np.ascontiguousarray(dd["logits_bits"]).view(np.int16)
    t = torch.from_numpy(bits).cuda().view(torch.bfloat16)
    T = np.repeat(dd["temperature"], 4).astype(np.float32)
    k = np.repeat(dd["top_k"], 4).astype(np.int32)
    p = np.repeat(dd["top_p"], 4).astype(np.float32)
    got = tv.sample_from_logits(t, 4, temperature=dev(T), top_k=dev(k), top_p=dev(p), joint=True,
                                seed=dev(dd["seed"]), offset=dev(dd["offset"]), logprobs=True)
    ref = oracle_all("sample_from_logits", dd["logits_bits"], True, 4, args=[(4, None)],
                     per_request=dict(seed=dd["seed"], offset=dd["offset"]),
                     per_row=dict(temperature=T, top_k=k, top_p=p), static=dict(joint=True))
    ok = ref["margin"] > BOUNDARY
    tok = got["tokens"].cpu().numpy()
    np.testing.assert_array_equal(tok[ok], ref["tokens"][ok])
    np.testing.assert_allclose(got["logprobs"].cpu().numpy()[ok], ref["logprobs"][ok],
                               **TOL["bf16"])
    print(f"\nsample B=512 N=4 V=201088: {rows} rows checked, {int((~ok).sum())} boundary")
    assert (~ok).sum() <= rows // 20
