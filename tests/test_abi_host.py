"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, it
exports every call the header declares, the workspace size is consistent, and invalid
arguments are rejected on the host before anything is launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ts_verify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verify_temp_gb300 import build, tsverify

    build.build()
    return tsverify.load()


def declared_calls():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ts_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_six_calls():
    names = declared_calls()
    for n in ["ts_softmax_temp", "ts_topk_topp_renorm", "ts_verify_chain_greedy",
              "ts_chain_spec_sampling", "ts_gumbel_max_sample", "ts_gather_logprobs"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(os.path.join(ROOT, "speculative_decoding_verify_temp_gb300",
                                   "libtsverify.so"))
    missing = [n for n in declared_calls() if not hasattr(raw, n)]
    assert not missing, missing


def test_workspace_size(lib):
    a = lib.ts_workspace_size(64, 4, 32000)
    b = lib.ts_workspace_size(128, 4, 32000)
    assert 0 < a < b
    assert a % 256 == 0
    assert lib.ts_workspace_size(0, 4, 100) == 0


def _err(lib):
    return lib.ts_last_error_message().decode()


def test_invalid_arguments_are_rejected_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(256)  # never dereferenced: validation fails first
    # vocab = 0
    st = lib.ts_verify_chain_greedy(fake, 0, 4, 3, 0, 0, fake, fake, fake, None, None, fake,
                                    1 << 20, None)
    assert st == 1 and "vocab" in _err(lib)
    # D out of range
    st = lib.ts_verify_chain_greedy(fake, 0, 4, 65, 100, 100, fake, fake, fake, None, None,
                                    fake, 1 << 20, None)
    assert st == 1 and "D must" in _err(lib)
    # ld < vocab
    st = lib.ts_softmax_temp(fake, 0, 4, 100, 99, None, fake, None)
    assert st == 1 and "ld" in _err(lib)
    # unknown dtype
    st = lib.ts_softmax_temp(fake, 7, 4, 100, 100, None, fake, None)
    assert st == 2
    # workspace too small
    st = lib.ts_gumbel_max_sample(fake, 0, 4, 2, 100, 100, fake, fake, fake, fake, P(512), 16,
                                  None)
    assert st == 1 and "workspace" in _err(lib)
    # bf16 probabilities are not accepted
    st = lib.ts_gather_logprobs(fake, 1, 1, 4, 100, 100, fake, fake, None, 0, None)
    assert st == 2
    # chain without coins
    from speculative_decoding_verify_temp_gb300.tsverify import ChainArgs
    a = ChainArgs()
    a.target = 256
    a.target_dtype = 0
    a.target_is_logits = 1
    a.batch, a.D, a.vocab, a.ld = 2, 1, 10, 10
    a.draft_tokens = 256
    a.accepted_tokens = 256
    a.accept_length = 256
    st = lib.ts_chain_spec_sampling(ctypes.byref(a), P(512), 1 << 20, None)
    assert st == 1 and "seed" in _err(lib)


def test_staged_vocabulary_limit_is_rejected_before_launch(lib):
    # rows the streaming kernels cannot take (here: an ld that breaks 16-byte alignment)
    # go to the cluster-staged kernel, which holds at most 655360 bf16 / 327680 fp32
    # tokens a row; longer rows are rejected on the host
    P = ctypes.c_void_p
    fake = P(256)
    V = 700000
    st = lib.ts_softmax_temp(fake, 1, 2, V, V + 1, None, fake, None)
    assert st == 1 and "staged limit" in _err(lib)
    V = 330000
    st = lib.ts_topk_topp_renorm(fake, 2, V, V + 1, None, None, P(4096), None)
    assert st == 1 and "staged limit" in _err(lib)
    from speculative_decoding_verify_temp_gb300.tsverify import ChainArgs
    a = ChainArgs()
    a.target = 256
    a.target_dtype = 1
    a.target_is_logits = 1
    a.batch, a.D, a.vocab, a.ld = 2, 1, 700000, 700000
    a.draft_tokens = a.accepted_tokens = a.accept_length = 256
    a.seed = a.offset = 256
    st = lib.ts_chain_spec_sampling(ctypes.byref(a), P(512), 1 << 40, None)
    assert st == 1 and "staged limit" in _err(lib)


def test_in_place_renorm_needs_contiguous_rows(lib):
    P = ctypes.c_void_p
    p = P(4096)
    st = lib.ts_topk_topp_renorm(p, 2, 100, 104, None, None, p, None)
    assert st == 1 and "in-place" in _err(lib)


def test_next_entry_points_reject_invalid_arguments_before_launch(lib):
    from speculative_decoding_verify_temp_gb300.tsverify import ChainArgs, SampleArgs
    P = ctypes.c_void_p

    def sample_args(**kw):
        a = SampleArgs()
        a.logits, a.dtype, a.n_per_req, a.batch, a.vocab, a.ld = 256, 1, 1, 4, 64, 64
        a.seed = a.offset = a.tokens = 256
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    def call(a):
        return lib.ts_sample_from_logits(ctypes.byref(a), P(512), 1 << 30, None)

    assert call(sample_args(batch=0)) == 1 and "batch" in _err(lib)  # empty
    assert call(sample_args(n_per_req=0)) == 1 and "n_per_req" in _err(lib)
    assert call(sample_args(filter_order=2)) == 1 and "filter_order" in _err(lib)
    assert call(sample_args(probs=256, ld_probs=10)) == 1 and "ld_probs" in _err(lib)
    assert call(sample_args(ld=65, vocab=65)) == 1 and "aligned" in _err(lib)  # 130-byte rows
    assert call(sample_args(seed=None)) == 1 and "seed" in _err(lib)
    assert call(sample_args(dtype=9)) == 2

    def chain_args(**kw):
        a = ChainArgs()
        a.target, a.target_dtype, a.target_is_logits = 256, 1, 1
        a.batch, a.D, a.vocab, a.ld = 2, 1, 64, 64
        a.draft_tokens = a.accepted_tokens = a.accept_length = a.seed = a.offset = 256
        for k, v in kw.items():
            setattr(a, k, v)
        return a

    def ccall(a):
        return lib.ts_chain_spec_sampling(ctypes.byref(a), P(512), 1 << 30, None)

    assert ccall(chain_args(batch=0)) == 1  # empty
    assert ccall(chain_args(draft_probs=256, ld_draft=64, threshold_acc=0.5)) == 1
    assert "target-only" in _err(lib)
    assert ccall(chain_args(target_is_logits=0, target_dtype=0, min_p=256)) == 1
    assert "logit targets" in _err(lib)
    assert ccall(chain_args(qo_indptr=256, total_rows=5)) == 1 and "total_rows" in _err(lib)
    assert ccall(chain_args(qo_indptr=256, total_rows=0)) == 1 and "total_rows" in _err(lib)
    # ragged greedy: total_rows out of range, missing qo_indptr
    st = lib.ts_verify_chain_greedy_ragged(P(256), 1, 2, 1, 64, 64, P(256), 5, P(256), P(256),
                                           P(256), None, None, P(512), 1 << 30, None)
    assert st == 1 and "total_rows" in _err(lib)
    st = lib.ts_verify_chain_greedy_ragged(P(256), 1, 2, 1, 64, 64, None, 3, P(256), P(256),
                                           P(256), None, None, P(512), 1 << 30, None)
    assert st == 1 and "qo_indptr" in _err(lib)
    # an empty Gumbel call
    st = lib.ts_gumbel_max_sample(P(256), 0, 0, 4, 100, 100, P(256), P(256), P(256), P(256),
                                  P(512), 1 << 30, None)
    assert st == 1
