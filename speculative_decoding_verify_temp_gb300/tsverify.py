"""Thin ctypes binding over libtsverify.so.

Argument marshalling only: each function takes torch tensors, passes their device
pointers, sizes and the current CUDA stream to the C call of the same name, and
raises ``TsError`` on a non-zero status. No computation happens here and there is
no fallback: if the library is missing or a call fails, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtsverify.so")

TS_F32, TS_BF16 = 0, 1
GREEDY_T = 1e-5
MAX_DRAFT = 64
_lib = None


class TsError(RuntimeError):
    def __init__(self, call: str, status: int, message: str):
        super().__init__(f"{call} failed with status {status}: {message}")
        self.status = status


class ChainArgs(ctypes.Structure):
    _fields_ = [
        ("target", ctypes.c_void_p),
        ("target_dtype", ctypes.c_int32),
        ("target_is_logits", ctypes.c_int32),
        ("batch", ctypes.c_int64),
        ("D", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("vocab", ctypes.c_int64),
        ("ld", ctypes.c_int64),
        ("temperature", ctypes.c_void_p),
        ("top_k", ctypes.c_void_p),
        ("top_p", ctypes.c_void_p),
        ("draft_probs", ctypes.c_void_p),
        ("ld_draft", ctypes.c_int64),
        ("draft_tokens", ctypes.c_void_p),
        ("seed", ctypes.c_void_p),
        ("offset", ctypes.c_void_p),
        ("uniforms", ctypes.c_void_p),
        ("accepted_tokens", ctypes.c_void_p),
        ("accept_length", ctypes.c_void_p),
        ("accept_index", ctypes.c_void_p),
        ("logprobs", ctypes.c_void_p),
        ("min_p", ctypes.c_void_p),
        ("threshold_single", ctypes.c_float),
        ("threshold_acc", ctypes.c_float),
        ("qo_indptr", ctypes.c_void_p),
        ("total_rows", ctypes.c_int64),
    ]


TS_FILTER_TOP_K_FIRST = 0
TS_FILTER_JOINT = 1


class SampleArgs(ctypes.Structure):
    """ts_sample_args of include/ts_verify.h."""
    _fields_ = [
        ("logits", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("n_per_req", ctypes.c_int32),
        ("batch", ctypes.c_int64),
        ("vocab", ctypes.c_int64),
        ("ld", ctypes.c_int64),
        ("temperature", ctypes.c_void_p),
        ("top_k", ctypes.c_void_p),
        ("top_p", ctypes.c_void_p),
        ("min_p", ctypes.c_void_p),
        ("filter_order", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("seed", ctypes.c_void_p),
        ("offset", ctypes.c_void_p),
        ("uniforms", ctypes.c_void_p),
        ("tokens", ctypes.c_void_p),
        ("logprobs", ctypes.c_void_p),
        ("probs", ctypes.c_void_p),
        ("ld_probs", ctypes.c_int64),
        ("probs_row", ctypes.c_void_p),
    ]


def load():
    """Loads libtsverify.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    st = ctypes.c_int
    L.ts_workspace_size.argtypes = [i64, i32, i64]
    L.ts_workspace_size.restype = ctypes.c_size_t
    L.ts_workspace_init.argtypes = [P, ctypes.c_size_t, P]
    L.ts_workspace_init.restype = st
    L.ts_last_error_message.argtypes = []
    L.ts_last_error_message.restype = ctypes.c_char_p
    L.ts_device_error.argtypes = [P, ctypes.c_int]
    L.ts_device_error.restype = st
    L.ts_set_wait_cycles.argtypes = [ctypes.c_uint64]
    L.ts_set_wait_cycles.restype = st
    L.ts_softmax_temp.argtypes = [P, ctypes.c_int, i64, i64, i64, P, P, P]
    L.ts_softmax_temp.restype = st
    L.ts_topk_topp_renorm.argtypes = [P, i64, i64, i64, P, P, P, P]
    L.ts_topk_topp_renorm.restype = st
    L.ts_verify_chain_greedy.argtypes = [P, ctypes.c_int, i64, i32, i64, i64, P, P, P, P, P, P,
                                         ctypes.c_size_t, P]
    L.ts_verify_chain_greedy.restype = st
    L.ts_chain_spec_sampling.argtypes = [ctypes.POINTER(ChainArgs), P, ctypes.c_size_t, P]
    L.ts_chain_spec_sampling.restype = st
    L.ts_gumbel_max_sample.argtypes = [P, ctypes.c_int, i64, i32, i64, i64, P, P, P, P, P,
                                       ctypes.c_size_t, P]
    L.ts_gumbel_max_sample.restype = st
    L.ts_gather_logprobs.argtypes = [P, ctypes.c_int, i32, i64, i64, i64, P, P, P,
                                     ctypes.c_size_t, P]
    L.ts_gather_logprobs.restype = st
    L.ts_sample_from_logits.argtypes = [ctypes.POINTER(SampleArgs), P, ctypes.c_size_t, P]
    L.ts_verify_chain_greedy_ragged.argtypes = [P, ctypes.c_int, i64, i32, i64, i64, P, i64, P,
                                                P, P, P, P, P, ctypes.c_size_t, P]
    L.ts_verify_chain_greedy_ragged.restype = st
    L.ts_sample_from_logits.restype = st
    _lib = L
    return L


def _check(call: str, status: int):
    if status != 0:
        msg = load().ts_last_error_message().decode(errors="replace")
        raise TsError(call, status, msg)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t) -> int:
    if t.dtype == torch.float32:
        return TS_F32
    if t.dtype == torch.bfloat16:
        return TS_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _rows(x):
    """(rows, vocab, ld) of a 2-D row-major tensor whose rows may be padded."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit stride in the last dimension")
    return x.shape[0], x.shape[1], x.stride(0)


def workspace_size(batch: int, rows_per_req: int, vocab: int) -> int:
    return int(load().ts_workspace_size(batch, rows_per_req, vocab))


def make_workspace(batch: int, rows_per_req: int, vocab: int, device=None, stream=None):
    """A zero-filled workspace for calls of this size (reusable: calls leave it zeroed)."""
    n = workspace_size(batch, rows_per_req, vocab)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check("ts_workspace_init", load().ts_workspace_init(_p(ws), n, _stream(stream)))
    return ws


def device_error(clear: bool = True) -> int:
    """The device error word (0: no bounded wait gave up). Synchronises the device."""
    w = ctypes.c_uint32(0)
    st = load().ts_device_error(ctypes.byref(w), int(clear))
    if st not in (0, 4):
        _check("ts_device_error", st)
    return int(w.value)


def set_wait_cycles(cycles: int) -> None:
    """Sets the chain kernel's stage-wait budget in SM clock cycles (0: the default)."""
    _check("ts_set_wait_cycles", load().ts_set_wait_cycles(int(cycles)))


def _dense_out(out, rows, V, device):
    """A [rows, V] contiguous fp32 output (the C ABI writes rows of V floats back to back)."""
    if out is None:
        return torch.empty((rows, V), dtype=torch.float32, device=device)
    if out.dtype != torch.float32 or tuple(out.shape) != (rows, V) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous fp32 tensor of shape ({rows}, {V})")
    return out


def softmax_temp(logits, temperature=None, out=None, stream=None):
    rows, V, ld = _rows(logits)
    out = _dense_out(out, rows, V, logits.device)
    _check("ts_softmax_temp", load().ts_softmax_temp(
        _p(logits), _dtype(logits), rows, V, ld, _p(temperature), _p(out), _stream(stream)))
    return out


def topk_topp_renorm(probs, top_k=None, top_p=None, out=None, stream=None):
    rows, V, ld = _rows(probs)
    out = _dense_out(out, rows, V, probs.device)
    _check("ts_topk_topp_renorm", load().ts_topk_topp_renorm(
        _p(probs), rows, V, ld, _p(top_k), _p(top_p), _p(out), _stream(stream)))
    return out


def _chain_outputs(B, R, device, accept_index, logprobs):
    acc = torch.empty((B, R), dtype=torch.int32, device=device)
    alen = torch.empty((B,), dtype=torch.int32, device=device)
    aidx = torch.empty((B, R), dtype=torch.int32, device=device) if accept_index else None
    lp = torch.empty((B, R), dtype=torch.float32, device=device) if logprobs else None
    return acc, alen, aidx, lp


def verify_chain_greedy(target_logits, D: int, draft_tokens, workspace=None, *,
                        accept_index: bool = True, logprobs: bool = True, outputs=None,
                        stream=None):
    rows, V, ld = _rows(target_logits)
    R = D + 1
    B = rows // R
    if workspace is None:
        workspace = make_workspace(B, R, V, target_logits.device, stream)
    acc, alen, aidx, lp = outputs or _chain_outputs(B, R, target_logits.device, accept_index,
                                                    logprobs)
    _check("ts_verify_chain_greedy", load().ts_verify_chain_greedy(
        _p(target_logits), _dtype(target_logits), B, D, V, ld, _p(draft_tokens), _p(acc),
        _p(alen), _p(aidx), _p(lp), _p(workspace), workspace.numel(), _stream(stream)))
    return dict(accepted_tokens=acc, accept_length=alen, accept_index=aidx, logprobs=lp)


def verify_chain_greedy_ragged(target_logits, D: int, qo_indptr, draft_tokens, workspace=None,
                               *, accept_index: bool = True, logprobs: bool = True,
                               outputs=None, stream=None):
    """Greedy verification of packed rows (request b owns rows qo_indptr[b] ..
    qo_indptr[b+1] - 1, qo_indptr int32 [B+1] on the device); outputs [B, D+1]."""
    rows, V, ld = _rows(target_logits)
    R = D + 1
    B = qo_indptr.numel() - 1
    if workspace is None:
        workspace = make_workspace(B, R, V, target_logits.device, stream)
    acc, alen, aidx, lp = outputs or _chain_outputs(B, R, target_logits.device, accept_index,
                                                    logprobs)
    _check("ts_verify_chain_greedy_ragged", load().ts_verify_chain_greedy_ragged(
        _p(target_logits), _dtype(target_logits), B, D, V, ld, _p(qo_indptr), rows,
        _p(draft_tokens), _p(acc), _p(alen), _p(aidx), _p(lp), _p(workspace), workspace.numel(),
        _stream(stream)))
    return dict(accepted_tokens=acc, accept_length=alen, accept_index=aidx, logprobs=lp)


def chain_spec_sampling(target, target_is_logits: bool, D: int, draft_tokens, *,
                        draft_probs=None, temperature=None, top_k=None, top_p=None,
                        seed=None, offset=None, uniforms=None, workspace=None,
                        accept_index: bool = True, logprobs: bool = True, outputs=None,
                        stream=None, min_p=None, threshold_single: float = 1.0,
                        threshold_acc: float = 1.0, qo_indptr=None):
    """Chain sampling of [B*(D+1), V] rows, or, with qo_indptr (int32 [B+1] on the
    device), of packed rows: request b owns rows qo_indptr[b] .. qo_indptr[b+1] - 1."""
    rows, V, ld = _rows(target)
    R = D + 1
    B = rows // R if qo_indptr is None else qo_indptr.numel() - 1
    if workspace is None:
        workspace = make_workspace(B, R, V, target.device, stream)
    acc, alen, aidx, lp = outputs or _chain_outputs(B, R, target.device, accept_index, logprobs)
    a = ChainArgs()
    a.target = target.data_ptr()
    a.target_dtype = _dtype(target)
    a.target_is_logits = int(bool(target_is_logits))
    a.batch, a.D, a.vocab, a.ld = B, D, V, ld
    a.temperature = None if temperature is None else temperature.data_ptr()
    a.top_k = None if top_k is None else top_k.data_ptr()
    a.top_p = None if top_p is None else top_p.data_ptr()
    if draft_probs is not None:
        q = draft_probs.reshape(-1, draft_probs.shape[-1]) if draft_probs.dim() == 3 else draft_probs
        a.draft_probs = q.data_ptr()
        a.ld_draft = q.stride(0)
    a.draft_tokens = None if draft_tokens is None else draft_tokens.data_ptr()
    a.seed = None if seed is None else seed.data_ptr()
    a.offset = None if offset is None else offset.data_ptr()
    a.uniforms = None if uniforms is None else uniforms.data_ptr()
    a.accepted_tokens = acc.data_ptr()
    a.accept_length = alen.data_ptr()
    a.accept_index = None if aidx is None else aidx.data_ptr()
    a.logprobs = None if lp is None else lp.data_ptr()
    a.min_p = None if min_p is None else min_p.data_ptr()
    a.threshold_single = float(threshold_single)
    a.threshold_acc = float(threshold_acc)
    if qo_indptr is not None:
        a.qo_indptr = qo_indptr.data_ptr()
        a.total_rows = rows
    _check("ts_chain_spec_sampling", load().ts_chain_spec_sampling(
        ctypes.byref(a), _p(workspace), workspace.numel(), _stream(stream)))
    return dict(accepted_tokens=acc, accept_length=alen, accept_index=aidx, logprobs=lp)


def sample_from_logits(logits, n_per_req: int = 1, *, temperature=None, top_k=None, top_p=None,
                       min_p=None, joint: bool = False, seed=None, offset=None, uniforms=None,
                       workspace=None, logprobs: bool = False, probs=None, probs_row=None,
                       out=None, stream=None):
    """Single-step sampling of each row. probs: True for a new [rows, V] fp32 tensor of
    the kept distributions, or a 2-D fp32 tensor that probs_row (int64 [rows]) indexes."""
    rows, V, ld = _rows(logits)
    B = rows // n_per_req
    dev = logits.device
    if workspace is None:
        workspace = make_workspace(rows, 1, V, dev, stream)
    tok = out if out is not None else torch.empty((rows,), dtype=torch.int32, device=dev)
    lp = torch.empty((rows,), dtype=torch.float32, device=dev) if logprobs else None
    if probs is True:
        probs = torch.empty((rows, V), dtype=torch.float32, device=dev)
    a = SampleArgs()
    a.logits = logits.data_ptr()
    a.dtype = _dtype(logits)
    a.n_per_req = n_per_req
    a.batch, a.vocab, a.ld = B, V, ld
    for name, t in (("temperature", temperature), ("top_k", top_k), ("top_p", top_p),
                    ("min_p", min_p), ("seed", seed), ("offset", offset),
                    ("uniforms", uniforms), ("probs_row", probs_row)):
        setattr(a, name, None if t is None else t.data_ptr())
    a.filter_order = TS_FILTER_JOINT if joint else TS_FILTER_TOP_K_FIRST
    a.tokens = tok.data_ptr()
    a.logprobs = None if lp is None else lp.data_ptr()
    if probs is not None:
        a.probs = probs.data_ptr()
        a.ld_probs = probs.stride(0)
    _check("ts_sample_from_logits", load().ts_sample_from_logits(
        ctypes.byref(a), _p(workspace), workspace.numel(), _stream(stream)))
    return dict(tokens=tok, logprobs=lp, probs=probs)


def gumbel_max_sample(logits, n_per_req: int, temperature, seed, offset, workspace=None,
                      out=None, stream=None):
    rows, V, ld = _rows(logits)
    B = rows // n_per_req
    if workspace is None:
        workspace = make_workspace(B, n_per_req, V, logits.device, stream)
    if out is None:
        out = torch.empty((rows,), dtype=torch.int32, device=logits.device)
    _check("ts_gumbel_max_sample", load().ts_gumbel_max_sample(
        _p(logits), _dtype(logits), B, n_per_req, V, ld, _p(temperature), _p(seed), _p(offset),
        _p(out), _p(workspace), workspace.numel(), _stream(stream)))
    return out


def gather_logprobs(x, tokens, is_probs: bool = False, workspace=None, out=None, stream=None):
    rows, V, ld = _rows(x)
    if workspace is None and not is_probs:
        workspace = make_workspace(rows, 1, V, x.device, stream)
    if out is None:
        out = torch.empty((rows,), dtype=torch.float32, device=x.device)
    nbytes = 0 if workspace is None else workspace.numel()
    _check("ts_gather_logprobs", load().ts_gather_logprobs(
        _p(x), _dtype(x), int(bool(is_probs)), rows, V, ld, _p(tokens), _p(out), _p(workspace),
        nbytes, _stream(stream)))
    return out
