"""Pins for the oracle's Philox4x32-10 and its uniform streams (CPU only).

The block function is checked against an independent implementation, Triton's
``philox_impl`` run by Triton's CPU interpreter (same published algorithm,
third-party code). The stream layout itself (which counter a coin uses) is a
reading, not something the pages fix: it is checked for its stated structure
and for statistical soundness only.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
from scipy import stats

_TRITON_SCRIPT = textwrap.dedent(
    r"""
    import os, sys
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def k(c_ptr, k_ptr, out_ptr, N: tl.constexpr):
        i = tl.arange(0, N)
        c0 = tl.load(c_ptr + 4 * i + 0).to(tl.uint32, bitcast=True)
        c1 = tl.load(c_ptr + 4 * i + 1).to(tl.uint32, bitcast=True)
        c2 = tl.load(c_ptr + 4 * i + 2).to(tl.uint32, bitcast=True)
        c3 = tl.load(c_ptr + 4 * i + 3).to(tl.uint32, bitcast=True)
        k0 = tl.load(k_ptr + 2 * i + 0).to(tl.uint32, bitcast=True)
        k1 = tl.load(k_ptr + 2 * i + 1).to(tl.uint32, bitcast=True)
        o0, o1, o2, o3 = tl.random.philox_impl(c0, c1, c2, c3, k0, k1, 10)
        tl.store(out_ptr + 4 * i + 0, o0.to(tl.int32, bitcast=True))
        tl.store(out_ptr + 4 * i + 1, o1.to(tl.int32, bitcast=True))
        tl.store(out_ptr + 4 * i + 2, o2.to(tl.int32, bitcast=True))
        tl.store(out_ptr + 4 * i + 3, o3.to(tl.int32, bitcast=True))

    ctr = np.load(sys.argv[1]); key = np.load(sys.argv[2])
    n = ctr.shape[0]
    c = torch.from_numpy(ctr.view(np.int32).reshape(-1).copy())
    kk = torch.from_numpy(key.view(np.int32).reshape(-1).copy())
    out = torch.zeros_like(c)
    k[(1,)](c, kk, out, N=n)
    np.save(sys.argv[3], out.numpy().view(np.uint32).reshape(n, 4))
    """
)


def _triton_philox(tmp_path, ctr, key):
    pytest.importorskip("triton")
    script = tmp_path / "tri.py"
    script.write_text(_TRITON_SCRIPT)
    np.save(tmp_path / "c.npy", ctr)
    np.save(tmp_path / "k.npy", key)
    env = dict(os.environ, TRITON_INTERPRET="1", CUDA_VISIBLE_DEVICES="")
    subprocess.run([sys.executable, str(script), str(tmp_path / "c.npy"),
                    str(tmp_path / "k.npy"), str(tmp_path / "o.npy")],
                   check=True, env=env, timeout=600)
    return np.load(tmp_path / "o.npy")


def test_philox_block_matches_independent_implementation(orc, tmp_path):
    rng = np.random.default_rng(7)
    n = 64
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    key[0] = 0
    ctr[1] = 0xFFFFFFFF
    key[1] = 0xFFFFFFFF
    ref = _triton_philox(tmp_path, ctr, key)
    mine = np.stack([orc.philox4x32_10(ctr[i], key[i]) for i in range(n)])
    np.testing.assert_array_equal(mine, ref)


def test_u01_endpoints_and_exactness(orc):
    assert orc.u01(0) == 2.0**-24
    assert orc.u01(0xFFFFFFFF) == 1.0 - 2.0**-24
    assert orc.u01(0x1FF) == 2.0**-24  # the low 9 bits are dropped
    assert orc.u01(0x200) == 3 * 2.0**-24
    rng = np.random.default_rng(3)
    for x in rng.integers(0, 2**32, size=200, dtype=np.uint64):
        u = orc.u01(int(x))
        m = u * 2**24
        assert m == int(m) and int(m) % 2 == 1  # an odd multiple of 2^-24
        assert 0.0 < u < 1.0
        assert np.float32(u) == u


def test_u01_is_monotone_in_the_word(orc):
    xs = np.sort(np.random.default_rng(4).integers(0, 2**32, 500, dtype=np.uint64))
    us = [orc.u01(int(x)) for x in xs]
    assert all(a <= b for a, b in zip(us, us[1:]))


def test_coin_and_gumbel_streams_follow_the_stated_counters(orc):
    seed = 0x0123456789ABCDEF
    off = 0x0000000500000007
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    for j in range(5):
        w = orc.philox4x32_10([j, 0xFFFFFFFF, off & 0xFFFFFFFF, off >> 32], key)
        assert orc.verify_coin(seed, off, j) == np.float32(orc.u01(int(w[0])))
    for n in range(3):
        for v in [0, 1, 2, 3, 4, 7, 1001]:
            w = orc.philox4x32_10([v >> 2, n, off & 0xFFFFFFFF, off >> 32], key)
            assert orc.gumbel_u01(seed, off, n, v) == np.float32(orc.u01(int(w[v & 3])))


def test_negative_seed_uses_its_64_bit_pattern(orc):
    # int64 seeds are keyed by their two's-complement bit pattern
    assert orc.verify_coin(-1, 3, 0) == orc.verify_coin(2**64 - 1, 3, 0)


def test_uniforms_are_uniform_and_decorrelated(orc):
    n = 20000
    us = np.array([orc.gumbel_u01(42, 9, 0, v) for v in range(n)], np.float64)
    counts, _ = np.histogram(us, bins=64, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 1e-4
    r = np.corrcoef(us[:-1], us[1:])[0, 1]
    assert abs(r) < 0.03
    assert len(np.unique(us)) > 0.99 * n
    coins = np.array([orc.verify_coin(s, 0, 0) for s in range(n)], np.float64)
    counts, _ = np.histogram(coins, bins=64, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 1e-4
