"""GB300-native speculative-decoding verify-and-sample step.

The product is ``libtsverify.so`` (C ABI declared in ``include/ts_verify.h``, kernels
for sm_103a under ``csrc/``); ``tsverify`` is its thin ctypes binding and ``synth``
the seeded synthetic input generator shared by the tests and the benchmark.
"""
from . import tsverify  # noqa: F401
from .tsverify import (  # noqa: F401
    chain_spec_sampling,
    gather_logprobs,
    gumbel_max_sample,
    make_workspace,
    softmax_temp,
    topk_topp_renorm,
    verify_chain_greedy,
)
