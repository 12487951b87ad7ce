"""GPU: a bounded wait that runs out is reported, leaves defined outputs, and does not
reach the next call.

The chain kernel's stage waits take their budget from ts_set_wait_cycles. With a budget
of one cycle the first wait of every CTA gives up before its bulk copy lands (no fault,
no hang: the CTA stops issuing, waits on the long budget for the copies it has in flight,
and exits at the next row boundary). The call must then report TS_ERR_TIMEOUT through
ts_device_error (bit 24 of the word; bit 25, a copy that never landed, must stay clear),
leave accept_length = 0 on every request it did not finish (and correct values on any it
did), and the next call with the default budget must match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_temp_gb300 import synth
from speculative_decoding_verify_temp_gb300 import tsverify as tv
from tests.gpu_util import compare_chain, dev, dev_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    oracle.build()
    tv.device_error(clear=True)
    yield
    tv.set_wait_cycles(0)
    tv.device_error(clear=True)


def _workload(B=24, D=3, V=50000):
    rng = np.random.default_rng(4242)
    R = D + 1
    x = rng.standard_normal((B * R, V), dtype=np.float32) * np.float32(3.0)
    x += synth.zipf_bias(V)[None, :]
    bits = synth.bf16_bits_from_f32(x)
    d = dict(dtype="bf16", logits_bits=bits, logits=synth.f32_from_bf16_bits(bits))
    T = rng.uniform(0.3, 1.5, B).astype(np.float32)
    T[rng.random(B) < 0.25] = 0.0
    k = rng.choice(np.array(synth.TOPK_CHOICES, np.int32), B).astype(np.int32)
    tp = rng.choice(np.array(synth.TOPP_CHOICES, np.float32), B).astype(np.float32)
    am = d["logits"].reshape(B, R, V)[:, :D].argmax(-1)
    drafts = np.where(rng.random((B, D)) < 0.6, am, rng.integers(0, V, (B, D))).astype(np.int32)
    kw = dict(temperature=T, top_k=k, top_p=tp, seed=synth.request_seeds(B),
              offset=np.arange(B, dtype=np.int64))
    return d, D, drafts, kw


def _call(d, D, drafts, kw, ws):
    B = drafts.shape[0]
    R = D + 1
    outs = (torch.full((B, R), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), 7, dtype=torch.int32, device="cuda"), None, None)
    return tv.chain_spec_sampling(dev_logits(d), True, D, dev(drafts),
                                  **{k: dev(v) for k, v in kw.items()}, workspace=ws,
                                  outputs=outs)


def test_wait_budget_runs_out_then_next_call_is_clean():
    d, D, drafts, kw = _workload()
    B, V = drafts.shape[0], d["logits"].shape[1]
    ref = oracle.chain_spec_sampling(d["logits"], True, D, drafts, **kw, logprobs=False)
    ws = tv.make_workspace(B, D + 1, V)
    compare_chain(_call(d, D, drafts, kw, ws), ref, "bf16")
    assert tv.device_error(clear=True) == 0

    tv.set_wait_cycles(1)
    try:
        r = _call(d, D, drafts, kw, ws)
        torch.cuda.synchronize()
    finally:
        tv.set_wait_cycles(0)
    word = tv.device_error(clear=True)
    assert word & (1 << 24), hex(word)
    assert not word & (1 << 25), hex(word)
    alen = r["accept_length"].cpu().numpy()
    done = alen != 0
    assert (~done).any()  # the requests the CTAs gave up on read 0
    np.testing.assert_array_equal(alen[done], ref["accept_length"][done])

    # the same workspace, the default budget: a clean call
    compare_chain(_call(d, D, drafts, kw, ws), ref, "bf16")
    assert tv.device_error(clear=True) == 0
