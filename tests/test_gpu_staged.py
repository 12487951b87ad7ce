"""GPU parity of the cluster-staged kernel, the route for rows the streaming kernels do
not take: unaligned rows (renorm, softmax, chain) and vocabularies above 2^18 up to the
staged limit (chain sampling, softmax), every row against the oracle."""
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


def _unaligned(t):
    """The rows of t in a buffer whose row stride (V + 1 elements) is not 16-byte aligned."""
    rows, V = t.shape
    buf = torch.zeros((rows, V + 1), dtype=t.dtype, device=t.device)
    buf[:, :V] = t
    return buf[:, :V]


@pytest.mark.parametrize("V", [151936, 151937, 4099])
def test_renorm_unaligned_rows(V):
    rng = np.random.default_rng(V)
    rows = 24
    x = rng.standard_normal((rows, V)).astype(np.float64) * 2.0
    x += synth.zipf_bias(V)[None, :]
    e = np.exp(x - x.max(1, keepdims=True))
    P = (e / e.sum(1, keepdims=True)).astype(np.float32)
    P[3, :] = np.float32(1.0 / V)  # a flat row: ties everywhere
    k = rng.choice(np.array(synth.TOPK_CHOICES, np.int32), rows).astype(np.int32)
    p = rng.choice(np.array(synth.TOPP_CHOICES, np.float32), rows).astype(np.float32)
    got = tv.topk_topp_renorm(_unaligned(torch.from_numpy(P).cuda()), dev(k), dev(p)).cpu().numpy()
    want, marg = oracle.topk_topp_renorm(P, k, p)
    ok = marg > BOUNDARY
    assert (~ok).sum() <= 2
    np.testing.assert_array_equal(got[ok] > 0, want[ok] > 0)
    np.testing.assert_allclose(got[ok], want[ok], **TOL["f32"])


@pytest.mark.parametrize("V,dtype", [(300000, "bf16"), (655360, "bf16"), (327680, "f32"),
                                     (100003, "bf16")])
def test_chain_on_the_staged_route(V, dtype):
    """Chain sampling from logits of vocabularies above 2^18 (and an unaligned one)."""
    rng = np.random.default_rng(V + 5)
    B, D = 6, 3
    R = D + 1
    x = rng.standard_normal((B * R, V), dtype=np.float32) * np.float32(3.0)
    x += synth.zipf_bias(V)[None, :]
    if dtype == "bf16":
        bits = synth.bf16_bits_from_f32(x)
        xf = synth.f32_from_bf16_bits(bits)
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    else:
        xf = x
        t = torch.from_numpy(x).cuda()
    am = xf.reshape(B, R, V)[:, :D].argmax(-1)
    drafts = np.where(rng.random((B, D)) < 0.6, am, rng.integers(0, V, (B, D))).astype(np.int32)
    T = rng.uniform(0.4, 1.3, B).astype(np.float32)
    T[0] = 0.0
    k = np.array([0, 20, 1000, 0, 50, 0], np.int32)
    p = np.array([1.0, 0.9, 1.0, 0.95, 0.9, 1.0], np.float32)
    kw = dict(temperature=T, top_k=k, top_p=p, seed=synth.request_seeds(B),
              offset=np.arange(B, dtype=np.int64))
    tt = _unaligned(t) if V % 8 else t
    got = tv.chain_spec_sampling(tt, True, D, dev(drafts), **{kk: dev(v) for kk, v in kw.items()})
    ref = oracle.chain_spec_sampling(xf, True, D, drafts, **kw)
    compare_chain(got, ref, dtype, max_boundary_frac=0.2)


@pytest.mark.parametrize("V", [655360, 151937])
def test_softmax_on_the_staged_route(V):
    rng = np.random.default_rng(V + 9)
    rows = 6
    x = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    T = rng.uniform(0.5, 1.5, rows).astype(np.float32)
    bits = synth.bf16_bits_from_f32(x)
    xf = synth.f32_from_bf16_bits(bits)
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)
    tt = _unaligned(t) if V % 8 else t
    got = tv.softmax_temp(tt, dev(T)).cpu().numpy()
    want = oracle.softmax_temp(xf, T)
    np.testing.assert_allclose(got, want, **TOL["f32"])
