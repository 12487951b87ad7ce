"""Helpers for the GPU parity tests: device tensors from the seeded inputs, and the
comparison rules (exact for integers; boundary decisions counted, not failed)."""
import multiprocessing
import os

import numpy as np
import torch

# Tolerances for probabilities and logprobs, by input dtype.
TOL = {"f32": dict(rtol=1e-5, atol=1e-6), "bf16": dict(rtol=2e-3, atol=1e-6)}
BOUNDARY = 1e-6  # a decision closer than this to flipping is a boundary case


def dev_logits(d, key="logits"):
    """The workload's logits as a device tensor of its own dtype."""
    if d.get("dtype") == "bf16":
        bits = np.ascontiguousarray(d["logits_bits"]).view(np.int16)
        return torch.from_numpy(bits).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(d[key])).cuda()


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def compare_chain(gpu: dict, ref: dict, dtype: str = "f32", max_boundary_frac: float = 0.05,
                  check_logprobs: bool = True, row_base=None):
    """Exact token/length/index parity on every request the oracle does not flag as a
    boundary case; logprobs within tolerance on the emitted positions. Returns the
    number of boundary requests. A draw over a flat distribution of V tokens lands
    within 1e-6 of a CDF edge with probability about 2e-6 * V, so the bound on the
    count of boundary requests is a sanity bound, not part of the parity rule.
    row_base: the first (packed) row of each request of a ragged batch; accept_index holds
    row_base[b] + j (rectangular: b * R + j)."""
    acc = gpu["accepted_tokens"].cpu().numpy()
    alen = gpu["accept_length"].cpu().numpy()
    margin = ref.get("margin")
    ok = np.ones(len(alen), bool) if margin is None else (margin > BOUNDARY)
    nb = int((~ok).sum())
    assert nb <= max(3, int(max_boundary_frac * len(alen))), f"{nb} boundary requests"
    np.testing.assert_array_equal(alen[ok], ref["accept_length"][ok])
    np.testing.assert_array_equal(acc[ok], ref["accepted_tokens"][ok])
    # invariants hold everywhere, boundary cases included
    R = acc.shape[1]
    assert alen.min() >= 1 and alen.max() <= R
    pos = np.arange(R)[None, :]
    assert ((acc >= 0) == (pos < alen[:, None])).all()
    if gpu.get("accept_index") is not None:
        aidx = gpu["accept_index"].cpu().numpy()
        base = np.arange(len(alen)) * R if row_base is None else np.asarray(row_base)
        want = np.where(pos < alen[:, None], base[:, None] + pos, -1)
        np.testing.assert_array_equal(aidx, want)
    if check_logprobs and gpu.get("logprobs") is not None and ref.get("logprobs") is not None:
        lp = gpu["logprobs"].cpu().numpy()
        np.testing.assert_allclose(lp[ok], ref["logprobs"][ok], **TOL[dtype])
    return nb


# ---- the oracle over whole launches, on every host core --------------------------------

def _oracle_worker(task):
    """One slice of requests through the oracle (runs in a spawned process)."""
    import oracle
    from speculative_decoding_verify_temp_gb300 import synth

    fn, rows, bf16, args, kw = task
    x = synth.f32_from_bf16_bits(rows) if bf16 else rows
    return getattr(oracle, fn)(x, *args, **kw)


def _slices(n, parts):
    step = max(1, -(-n // parts))
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def oracle_all(fn, rows, bf16, R, args=(), per_request=None, static=None, procs=None,
               per_row=None):
    """oracle.<fn>(x, *args, **kw) over every request of a launch, the requests split over
    the host cores (the method is per request: each request's coins come from its own seed
    and offset, so the slices are independent). rows: the launch's [B*R, V] values as bf16
    bits (bf16=True) or fp32. args: positional arguments, each (array, "row" | "req" |
    None) - sliced by rows, by requests, or passed whole; per_request: keyword arrays of
    one entry per request (None allowed); per_row: keyword arrays of one entry per row;
    static: keyword arguments passed as they are.
    Dict results (the chain calls) and tuple results are concatenated."""
    B = rows.shape[0] // R
    procs = procs or max(1, min(os.cpu_count() or 1, 32))
    per_request = per_request or {}
    tasks = []
    for b0, b1 in _slices(B, procs):
        a = []
        for arr, by in args:
            a.append(arr[b0 * R:b1 * R] if by == "row" else arr[b0:b1] if by == "req" else arr)
        kw = {k: (None if v is None else v[b0:b1]) for k, v in per_request.items()}
        kw.update({k: (None if v is None else v[b0 * R:b1 * R])
                   for k, v in (per_row or {}).items()})
        kw.update(static or {})
        tasks.append((fn, np.ascontiguousarray(rows[b0 * R:b1 * R]), bf16, tuple(a), kw))
    with multiprocessing.get_context("spawn").Pool(len(tasks)) as pool:
        parts = pool.map(_oracle_worker, tasks)
    if isinstance(parts[0], dict):
        # accept_index holds flat row numbers b*R + j: each slice counts from its own first
        # request
        bases = [b0 for b0, _ in _slices(B, procs)]
        for p, b0 in zip(parts, bases):
            if p.get("accept_index") is not None:
                ai = p["accept_index"]
                p["accept_index"] = np.where(ai >= 0, ai + b0 * R, ai)
        return {k: (None if parts[0][k] is None else np.concatenate([p[k] for p in parts]))
                for k in parts[0]}
    return tuple(np.concatenate([p[i] for p in parts]) for i in range(len(parts[0])))


def _ragged_worker(task):
    import oracle
    from speculative_decoding_verify_temp_gb300 import synth

    fn, rows, bf16, D, qo, pre, drafts, kw = task
    x = synth.f32_from_bf16_bits(rows) if bf16 else rows
    return getattr(oracle, fn)(x, *pre, D, qo, drafts, **kw)


def oracle_ragged_all(fn, rows, bf16, D, qo, args=(), per_request=None, static=None, procs=None):
    """oracle.<fn> (a ragged call: fn(x, [is_logits,] D, qo_indptr, drafts, **kw)) over every
    request of a packed launch, requests split over the host cores with their packed rows
    (qo rebased per slice). args: (is_logits,) or () before D; per_request: keyword
    arrays of one entry (or row of entries) per request, drafts included under
    "draft_tokens"; accept_index comes back as packed row numbers of the whole launch."""
    B = len(qo) - 1
    procs = procs or max(1, min(os.cpu_count() or 1, 32))
    per_request = dict(per_request or {})
    drafts = per_request.pop("draft_tokens")
    tasks, bases = [], []
    for b0, b1 in _slices(B, procs):
        r0, r1 = int(qo[b0]), int(qo[b1])
        sub_qo = (np.asarray(qo[b0:b1 + 1]) - r0).astype(np.int32)
        kw = {k: (None if v is None else v[b0:b1]) for k, v in per_request.items()}
        kw.update(static or {})
        tasks.append((fn, np.ascontiguousarray(rows[r0:r1]), bf16, D, sub_qo, tuple(args),
                      np.ascontiguousarray(drafts[b0:b1]), kw))
        bases.append(r0)
    with multiprocessing.get_context("spawn").Pool(len(tasks)) as pool:
        parts = pool.map(_ragged_worker, tasks)
    for p, r0 in zip(parts, bases):
        ai = p["accept_index"]
        p["accept_index"] = np.where(ai >= 0, ai + r0, ai)
    return {k: (None if parts[0].get(k) is None else np.concatenate([p[k] for p in parts]))
            for k in parts[0]}
