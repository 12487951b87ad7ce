"""Helpers for the GPU parity tests: device tensors from the seeded inputs, and the
comparison rules (exact for integers; boundary decisions counted, not failed)."""
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
                  check_logprobs: bool = True):
    """Exact token/length/index parity on every request the oracle does not flag as a
    boundary case; logprobs within tolerance on the emitted positions. Returns the
    number of boundary requests. A draw over a flat distribution of V tokens lands
    within 1e-6 of a CDF edge with probability about 2e-6 * V, so the bound on the
    count of boundary requests is a sanity bound, not part of the parity rule."""
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
        want = np.where(pos < alen[:, None], np.arange(len(alen))[:, None] * R + pos, -1)
        np.testing.assert_array_equal(aidx, want)
    if check_logprobs and gpu.get("logprobs") is not None and ref.get("logprobs") is not None:
        lp = gpu["logprobs"].cpu().numpy()
        np.testing.assert_allclose(lp[ok], ref["logprobs"][ok], **TOL[dtype])
    return nb
