"""The greedy verification entry point that allocates nothing.

Callers that cannot give the library device memory (a host binding the C ABI without a
device allocator, or code whose device memory is a fixed budget owned by another
allocator) use ts_verify_chain_greedy_static, whose scratch is a fixed array inside the
library. This checks it, through the C ABI, against the workspace entry point on two
calls in a row with different inputs (the second call must not see the first call's
scratch), and that it rejects a call larger than its fixed scratch. The file is named to
be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _static_fn():
    from speculative_decoding_verify_temp_gb300 import tsverify as tv

    lib = ctypes.CDLL(tv.LIB_PATH)
    f = lib.ts_verify_chain_greedy_static
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    f.argtypes = [P, ctypes.c_int, i64, i32, i64, i64, P, P, P, P, P, P]
    f.restype = ctypes.c_int
    lib.ts_last_error_message.restype = ctypes.c_char_p
    return f, lib


def _inputs(seed, B, D, V):
    from speculative_decoding_verify_temp_gb300 import synth

    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B * (D + 1), V), dtype=np.float32) * np.float32(3.0)
    x += synth.zipf_bias(V)[None, :]
    bits = synth.bf16_bits_from_f32(x)
    f32 = synth.f32_from_bf16_bits(bits)
    am = f32.reshape(B, D + 1, V)[:, :D].argmax(-1)
    drafts = np.where(rng.random((B, D)) < 0.7, am, rng.integers(0, V, (B, D))).astype(np.int32)
    logits = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    return logits, torch.from_numpy(drafts).cuda()


def test_static_scratch_entry_point_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    from speculative_decoding_verify_temp_gb300 import tsverify as tv

    f, lib = _static_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, (B, D, V) in [(1, (64, 3, 32000)), (2, (512, 3, 8192))]:
        logits, drafts = _inputs(seed, B, D, V)
        R = D + 1
        ref = tv.verify_chain_greedy(logits, D, drafts)
        acc = torch.full((B, R), -7, dtype=torch.int32, device="cuda")
        alen = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        aidx = torch.full((B, R), -7, dtype=torch.int32, device="cuda")
        lp = torch.full((B, R), 7.0, dtype=torch.float32, device="cuda")
        st = f(ctypes.c_void_p(logits.data_ptr()), 1, B, D, V, V,
               ctypes.c_void_p(drafts.data_ptr()), ctypes.c_void_p(acc.data_ptr()),
               ctypes.c_void_p(alen.data_ptr()), ctypes.c_void_p(aidx.data_ptr()),
               ctypes.c_void_p(lp.data_ptr()), stream)
        assert st == 0, lib.ts_last_error_message()
        torch.cuda.synchronize()
        assert torch.equal(acc, ref["accepted_tokens"])
        assert torch.equal(alen, ref["accept_length"])
        assert torch.equal(aidx, ref["accept_index"])
        np.testing.assert_allclose(lp.cpu().numpy(), ref["logprobs"].cpu().numpy(),
                                   rtol=2e-3, atol=1e-6)
    # beyond the fixed scratch: rejected on the host, nothing launched
    st = f(ctypes.c_void_p(logits.data_ptr()), 1, 1024, 3, V, V,
           ctypes.c_void_p(drafts.data_ptr()), ctypes.c_void_p(acc.data_ptr()),
           ctypes.c_void_p(alen.data_ptr()), None, None, stream)
    assert st == 1 and b"static scratch" in lib.ts_last_error_message()
