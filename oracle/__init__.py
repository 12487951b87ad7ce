"""Oracle for the speculative-decoding verify-and-sample step.

TEST INFRASTRUCTURE ONLY. A plain, slow, single-threaded C restatement of the
step (``philox.c``, ``oracle.c``) with a ctypes front end. Only the tests, the
package smoke check and the benchmark's CPU-baseline leg may import it; the
CUDA library never does, and the two share no code.

Every function takes numpy arrays. Value arrays are float32 ``[rows, V]``
(bf16 inputs are widened to float32 by the caller, which is exact); results
are float64 where the oracle computes them in fp64.

Parity-unpinned parts: the Philox *stream layout* (which counter a coin or a
Gumbel element uses) is a reading of the pages, not something they fix, so it
is pinned only against itself (and the block function against an independent
implementation); every other function is pinned by the tests under
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liborc.so")
_SRC = [os.path.join(_HERE, "philox.c"), os.path.join(_HERE, "oracle.c")]
_lib = None

GREEDY_T = 1e-5


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no fused multiply-add)."""
    newest = max(os.path.getmtime(s) for s in _SRC + [os.path.join(_HERE, "orc.h")])
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp] + _SRC + ["-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_u01.argtypes = [ctypes.c_uint32]
        L.orc_u01.restype = f32
        L.orc_verify_coin.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
        L.orc_verify_coin.restype = f32
        L.orc_gumbel_u01.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                     ctypes.c_uint32]
        L.orc_gumbel_u01.restype = f32
        L.orc_argmax.argtypes = [P, i64]
        L.orc_argmax.restype = i64
        L.orc_filter_row.argtypes = [P, i64, ctypes.c_int, f32, i32, f32, P, P]
        L.orc_filter_row.restype = ctypes.c_double
        L.orc_softmax_temp.argtypes = [P, i64, i64, i64, P, P]
        L.orc_topk_topp_renorm.argtypes = [P, i64, i64, i64, P, P, P, P]
        L.orc_verify_chain_greedy.argtypes = [P, i64, i32, i64, i64, P, P, P, P, P]
        L.orc_chain_spec_sampling.argtypes = [P, ctypes.c_int, i64, i32, i64, i64, P, P, P,
                                              P, i64, P, P, P, P, P, P, P, P, P]
        L.orc_gumbel_max_sample.argtypes = [P, i64, i32, i64, i64, P, P, P, P, P]
        L.orc_gather_logprobs.argtypes = [P, ctypes.c_int, i64, i64, i64, P, P]
        L.orc_filter_row_ex.argtypes = [P, i64, ctypes.c_int, f32, i32, f32, f32, ctypes.c_int,
                                        P, P]
        L.orc_filter_row_ex.restype = ctypes.c_double
        L.orc_chain_spec_sampling_ex.argtypes = [P, ctypes.c_int, i64, i32, i64, i64, P, P, P,
                                                 P, f32, f32, P, i64, P, P, P, P, P, P, P, P,
                                                 P]
        L.orc_sample_from_logits.argtypes = [P, i64, i32, i64, i64, P, P, P, P, ctypes.c_int,
                                             P, P, P, P, P, P, P]
        L.orc_verify_chain_greedy_ragged.argtypes = [P, i64, i32, i64, i64, P, P, P, P, P, P]
        L.orc_chain_spec_sampling_ragged.argtypes = [P, ctypes.c_int, i64, i32, i64, i64, P, P,
                                                     P, P, P, f32, f32, P, i64, P, P, P, P, P,
                                                     P, P, P, P]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _i64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int64)


# ---- Philox ------------------------------------------------------------------

def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def u01(x: int) -> float:
    return float(np.float32(_load().orc_u01(int(x) & 0xFFFFFFFF)))


def verify_coin(seed: int, offset: int, j: int) -> np.float32:
    return np.float32(_load().orc_verify_coin(int(seed) & (2**64 - 1),
                                              int(offset) & (2**64 - 1), j))


def gumbel_u01(seed: int, offset: int, n: int, v: int) -> np.float32:
    return np.float32(_load().orc_gumbel_u01(int(seed) & (2**64 - 1),
                                             int(offset) & (2**64 - 1), n, v))


# ---- rows ----------------------------------------------------------------------

def argmax(x) -> int:
    x = _f32(x)
    return int(_load().orc_argmax(_ptr(x), x.shape[-1]))


def filter_row(vals, is_logits: bool, T: float = 1.0, top_k: int = 0, top_p: float = 1.0,
               min_p: float = 0.0, joint: bool = False):
    """p'' of one row and the decision margin (top-k first unless joint; min_p last)."""
    v = _f32(vals).reshape(-1)
    out = np.zeros(v.shape[0], dtype=np.float64)
    am = ctypes.c_int64(0)
    if min_p == 0.0 and not joint:
        m = _load().orc_filter_row(_ptr(v), v.shape[0], int(is_logits), T, int(top_k),
                                   float(top_p), _ptr(out), ctypes.byref(am))
    else:
        m = _load().orc_filter_row_ex(_ptr(v), v.shape[0], int(is_logits), T, int(top_k),
                                      float(top_p), float(min_p), int(joint), _ptr(out),
                                      ctypes.byref(am))
    return out, m


# ---- the operations --------------------------------------------------------------

def softmax_temp(logits, temperature=None) -> np.ndarray:
    x = _f32(logits)
    rows, V = x.shape
    out = np.zeros((rows, V), dtype=np.float64)
    _load().orc_softmax_temp(_ptr(x), rows, V, V, _ptr(_f32(temperature)), _ptr(out))
    return out


def topk_topp_renorm(probs, top_k=None, top_p=None):
    x = _f32(probs)
    rows, V = x.shape
    out = np.zeros((rows, V), dtype=np.float64)
    marg = np.zeros(rows, dtype=np.float64)
    _load().orc_topk_topp_renorm(_ptr(x), rows, V, V, _ptr(_i32(top_k)), _ptr(_f32(top_p)),
                                 _ptr(out), _ptr(marg))
    return out, marg


def verify_chain_greedy(logits, D: int, draft_tokens, logprobs: bool = True) -> dict:
    x = _f32(logits)
    rows, V = x.shape
    R = D + 1
    B = rows // R
    dt = _i32(draft_tokens).reshape(B, D) if D > 0 else np.zeros((B, 0), np.int32)
    acc = np.zeros((B, R), np.int32)
    alen = np.zeros(B, np.int32)
    aidx = np.zeros((B, R), np.int32)
    lp = np.zeros((B, R), np.float64) if logprobs else None
    _load().orc_verify_chain_greedy(_ptr(x), B, D, V, V, _ptr(np.ascontiguousarray(dt)),
                                    _ptr(acc), _ptr(alen), _ptr(aidx), _ptr(lp))
    return dict(accepted_tokens=acc, accept_length=alen, accept_index=aidx, logprobs=lp)


def chain_spec_sampling(target, target_is_logits: bool, D: int, draft_tokens, *,
                        draft_probs=None, temperature=None, top_k=None, top_p=None,
                        seed=None, offset=None, uniforms=None, logprobs: bool = True,
                        min_p=None, threshold_single: float = 1.0,
                        threshold_acc: float = 1.0) -> dict:
    x = _f32(target)
    rows, V = x.shape
    R = D + 1
    B = rows // R
    dt = np.ascontiguousarray(_i32(draft_tokens).reshape(B, D))
    q = None
    if draft_probs is not None:
        q = _f32(draft_probs).reshape(B * D, V)
    if uniforms is None and (seed is None or offset is None):
        raise ValueError("either uniforms or seed and offset are required")
    acc = np.zeros((B, R), np.int32)
    alen = np.zeros(B, np.int32)
    aidx = np.zeros((B, R), np.int32)
    lp = np.zeros((B, R), np.float64) if logprobs else None
    marg = np.zeros(B, np.float64)
    uni = None if uniforms is None else _f32(uniforms).reshape(B, R)
    if min_p is None and threshold_single == 1.0 and threshold_acc == 1.0:
        _load().orc_chain_spec_sampling(
            _ptr(x), int(target_is_logits), B, D, V, V, _ptr(_f32(temperature)),
            _ptr(_i32(top_k)), _ptr(_f32(top_p)), _ptr(q), V, _ptr(dt), _ptr(_i64(seed)),
            _ptr(_i64(offset)), _ptr(uni), _ptr(acc), _ptr(alen), _ptr(aidx), _ptr(lp),
            _ptr(marg))
    else:
        _load().orc_chain_spec_sampling_ex(
            _ptr(x), int(target_is_logits), B, D, V, V, _ptr(_f32(temperature)),
            _ptr(_i32(top_k)), _ptr(_f32(top_p)), _ptr(_f32(min_p)), float(threshold_single),
            float(threshold_acc), _ptr(q), V, _ptr(dt), _ptr(_i64(seed)), _ptr(_i64(offset)),
            _ptr(uni), _ptr(acc), _ptr(alen), _ptr(aidx), _ptr(lp), _ptr(marg))
    return dict(accepted_tokens=acc, accept_length=alen, accept_index=aidx, logprobs=lp,
                margin=marg)


def verify_chain_greedy_ragged(logits, D: int, qo_indptr, draft_tokens) -> dict:
    """Greedy verification of packed rows: request b owns rows qo_indptr[b] ..
    qo_indptr[b+1] - 1; drafts [B, D] padded; outputs padded to [B, D+1]."""
    x = _f32(logits)
    V = x.shape[1]
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    B = qo.shape[0] - 1
    R = D + 1
    dt = np.ascontiguousarray(_i32(draft_tokens).reshape(B, max(D, 0)))
    acc = np.zeros((B, R), np.int32)
    alen = np.zeros(B, np.int32)
    aidx = np.zeros((B, R), np.int32)
    lp = np.zeros((B, R), np.float64)
    _load().orc_verify_chain_greedy_ragged(_ptr(x), B, D, V, V, _ptr(qo), _ptr(dt), _ptr(acc),
                                           _ptr(alen), _ptr(aidx), _ptr(lp))
    return dict(accepted_tokens=acc, accept_length=alen, accept_index=aidx, logprobs=lp)


def chain_spec_sampling_ragged(target, target_is_logits: bool, D: int, qo_indptr,
                               draft_tokens, *, draft_probs=None, temperature=None, top_k=None,
                               top_p=None, min_p=None, threshold_single: float = 1.0,
                               threshold_acc: float = 1.0, seed=None, offset=None,
                               uniforms=None) -> dict:
    """Chain sampling of packed rows (request b owns rows qo_indptr[b] ..); knobs, seeds
    and offsets per request; drafts [B, D], draft probs [B*D, V] and uniforms [B, D+1]
    padded; outputs padded to [B, D+1]."""
    x = _f32(target)
    V = x.shape[1]
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    B = qo.shape[0] - 1
    R = D + 1
    dt = np.ascontiguousarray(_i32(draft_tokens).reshape(B, max(D, 0)))
    q = None if draft_probs is None else _f32(draft_probs).reshape(B * D, V)
    if uniforms is None and (seed is None or offset is None):
        raise ValueError("either uniforms or seed and offset are required")
    acc = np.zeros((B, R), np.int32)
    alen = np.zeros(B, np.int32)
    aidx = np.zeros((B, R), np.int32)
    lp = np.zeros((B, R), np.float64)
    marg = np.zeros(B, np.float64)
    _load().orc_chain_spec_sampling_ragged(
        _ptr(x), int(target_is_logits), B, D, V, V, _ptr(qo), _ptr(_f32(temperature)),
        _ptr(_i32(top_k)), _ptr(_f32(top_p)), _ptr(_f32(min_p)), float(threshold_single),
        float(threshold_acc), _ptr(q), V, _ptr(dt), _ptr(_i64(seed)), _ptr(_i64(offset)),
        _ptr(None if uniforms is None else _f32(uniforms).reshape(B, R)), _ptr(acc),
        _ptr(alen), _ptr(aidx), _ptr(lp), _ptr(marg))
    return dict(accepted_tokens=acc, accept_length=alen, accept_index=aidx, logprobs=lp,
                margin=marg)


def sample_from_logits(logits, n_per_req: int = 1, *, temperature=None, top_k=None,
                       top_p=None, min_p=None, joint: bool = False, seed=None, offset=None,
                       uniforms=None, probs: bool = False) -> dict:
    """Single-step sampling of every row (knobs per row; seed and offset per request of
    n_per_req rows). Returns tokens, logprobs, margin and, with probs, the kept
    distributions."""
    x = _f32(logits)
    rows, V = x.shape
    B = rows // n_per_req
    if uniforms is None and (seed is None or offset is None):
        raise ValueError("either uniforms or seed and offset are required")
    tok = np.zeros(rows, np.int32)
    lp = np.zeros(rows, np.float64)
    marg = np.zeros(rows, np.float64)
    pr = np.zeros((rows, V), np.float64) if probs else None
    _load().orc_sample_from_logits(
        _ptr(x), B, n_per_req, V, V, _ptr(_f32(temperature)), _ptr(_i32(top_k)),
        _ptr(_f32(top_p)), _ptr(_f32(min_p)), int(joint), _ptr(_i64(seed)), _ptr(_i64(offset)),
        _ptr(_f32(uniforms)), _ptr(tok), _ptr(pr), _ptr(lp), _ptr(marg))
    return dict(tokens=tok, logprobs=lp, margin=marg, probs=pr)


def gumbel_max_sample(logits, n_per_req: int, temperature, seed, offset):
    x = _f32(logits)
    rows, V = x.shape
    B = rows // n_per_req
    tok = np.zeros(rows, np.int32)
    marg = np.zeros(rows, np.float64)
    _load().orc_gumbel_max_sample(_ptr(x), B, n_per_req, V, V, _ptr(_f32(temperature)),
                                  _ptr(_i64(seed)), _ptr(_i64(offset)), _ptr(tok),
                                  _ptr(marg))
    return tok, marg


def gather_logprobs(x, is_probs: bool, tokens) -> np.ndarray:
    a = _f32(x)
    rows, V = a.shape
    out = np.zeros(rows, np.float64)
    _load().orc_gather_logprobs(_ptr(a), int(is_probs), rows, V, V,
                                _ptr(_i32(tokens)), _ptr(out))
    return out
