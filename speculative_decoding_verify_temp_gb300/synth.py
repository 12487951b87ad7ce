"""Seeded synthetic inputs for the verify-and-sample step.

Both the CUDA path and the oracle are fed from here, so this module holds none
of the step's own arithmetic: it draws random logits, knobs, seeds and draft
tokens with numpy's PCG64 and packs them. Two recipes need a probability
vector to draw from (draft tokens "sampled from" a distribution, and the
rejection workload whose inputs *are* probabilities); they use numpy's own
``exp``/``cumsum`` directly, as input preparation, and neither side of the
parity check calls them.

Workloads (sizes are the defaults of each builder):
  tiny_verify      B=4,   D=3, V=1024,   fp32 logits ~ N(0, 2^2)
  greedy_verify    B=64,  D=3, V=32000,  bf16 logits ~ N(0, 3^2) + Zipf(1.1) bias
  target_only      B=128, D=4, V=128256, bf16 + Zipf; per-request T, top-k, top-p
  rejection        B=256, D=7, V=151936, fp32 draft/target probabilities
  gumbel           B=512, N=4, V=201088 (200019 real ids, -inf pads), bf16 + Zipf
The Zipf(s) log-frequency bias of token id i is -s * ln(i + 1): ids are taken
to be in frequency-rank order.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20261202
TOPK_CHOICES = (0, 20, 50, 1000)
TOPP_CHOICES = (1.0, 0.95, 0.9)
MASK64 = (1 << 64) - 1


# ---- representation helpers ---------------------------------------------------

def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    # finite values and infinities stay below 0xFFFF8000, so the sum cannot wrap
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def zipf_bias(V: int, s: float = 1.1) -> np.ndarray:
    return (-s * np.log(np.arange(V, dtype=np.float64) + 1.0)).astype(np.float32)


def splitmix64(x: int) -> int:
    z = (x + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def request_seeds(B: int, base: int = 0xC0FFEE) -> np.ndarray:
    """Full 64-bit per-request seeds, stored as int64 (two's complement)."""
    vals = [splitmix64(base + b) for b in range(B)]
    return np.array(vals, dtype=np.uint64).view(np.int64)


def _rng(cfg_id: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + cfg_id + 1000 * salt))


def _sample_rows(rng, logp: np.ndarray) -> np.ndarray:
    """One draw per row from the distribution proportional to exp(logp) (input prep)."""
    out = np.empty(logp.shape[0], dtype=np.int32)
    for r in range(logp.shape[0]):
        z = logp[r].astype(np.float64)
        z = np.exp(z - z.max())
        c = np.cumsum(z)
        out[r] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")),
                     logp.shape[1] - 1)
    return out


def _logits(rng, rows: int, V: int, sigma: float, zipf: bool, bf16: bool):
    x = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(sigma)
    if zipf:
        x += zipf_bias(V)[None, :]
    if bf16:
        bits = bf16_bits_from_f32(x)
        return bits, f32_from_bf16_bits(bits)
    return None, x


# ---- workloads ------------------------------------------------------------------

def tiny_verify(B: int = 4, D: int = 3, V: int = 1024, cfg_id: int = 0) -> dict:
    """fp32 logits ~ N(0, 2^2); draft probs = softmax(logits + N(0, 0.5^2)) of rows
    0..D-1, drafts drawn from them; T = 1, no top-k/top-p; seed 1234, offset = b."""
    rng = _rng(cfg_id)
    R = D + 1
    _, logits = _logits(rng, B * R, V, 2.0, False, False)
    lg = logits.reshape(B, R, V)
    noisy = lg[:, :D, :].astype(np.float64) + rng.standard_normal((B, D, V)) * 0.5
    e = np.exp(noisy - noisy.max(axis=-1, keepdims=True))
    q = (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    drafts = _sample_rows(rng, np.log(np.maximum(q.reshape(B * D, V), 1e-38))).reshape(B, D)
    return dict(B=B, D=D, V=V, dtype="f32", logits=logits, draft_probs=q,
                draft_tokens=drafts, seed=np.full(B, 1234, np.int64),
                offset=np.arange(B, dtype=np.int64))


def greedy_verify(B: int = 64, D: int = 3, V: int = 32000, cfg_id: int = 1) -> dict:
    """bf16 logits ~ N(0, 3^2) + Zipf bias; draft j = argmax of row j w.p. 0.7,
    else a uniform random id."""
    rng = _rng(cfg_id)
    R = D + 1
    bits, f32 = _logits(rng, B * R, V, 3.0, True, True)
    am = np.argmax(f32.reshape(B, R, V)[:, :D, :], axis=-1).astype(np.int32)
    rnd = rng.integers(0, V, size=(B, D), dtype=np.int32)
    drafts = np.where(rng.random((B, D)) < 0.7, am, rnd).astype(np.int32)
    return dict(B=B, D=D, V=V, dtype="bf16", logits_bits=bits, logits=f32,
                draft_tokens=drafts)


def target_only(B: int = 128, D: int = 4, V: int = 128256, cfg_id: int = 2,
                greedy_frac: float = 0.0) -> dict:
    """bf16 logits ~ N(0, 3^2) + Zipf; per request T ~ U[0.5, 1.2], top_k and top_p
    drawn uniformly from their choice sets; draft j drawn from softmax(row j / T)
    w.p. 0.6, else a uniform random id; Philox seed per request."""
    rng = _rng(cfg_id)
    R = D + 1
    bits, f32 = _logits(rng, B * R, V, 3.0, True, True)
    T = rng.uniform(0.5, 1.2, size=B).astype(np.float32)
    if greedy_frac > 0:
        T[rng.random(B) < greedy_frac] = 0.0
    top_k = rng.choice(np.array(TOPK_CHOICES, np.int32), size=B).astype(np.int32)
    top_p = rng.choice(np.array(TOPP_CHOICES, np.float32), size=B).astype(np.float32)
    lg = f32.reshape(B, R, V)[:, :D, :]
    Tr = np.maximum(T, 1e-3)[:, None, None]
    sampled = _sample_rows(rng, (lg / Tr).reshape(B * D, V)).reshape(B, D)
    rnd = rng.integers(0, V, size=(B, D), dtype=np.int32)
    drafts = np.where(rng.random((B, D)) < 0.6, sampled, rnd).astype(np.int32)
    return dict(B=B, D=D, V=V, dtype="bf16", logits_bits=bits, logits=f32,
                temperature=T, top_k=top_k, top_p=top_p, draft_tokens=drafts,
                seed=request_seeds(B), offset=np.arange(B, dtype=np.int64))


def rejection(B: int = 256, D: int = 7, V: int = 151936, cfg_id: int = 3) -> dict:
    """fp32 draft logits ~ N(0, 2.5^2), target logits = draft + N(0, 0.7^2); the
    inputs are their softmaxes at T = 1 (fp32); drafts drawn from the draft probs."""
    rng = _rng(cfg_id)
    R = D + 1
    dl = rng.standard_normal((B, R, V), dtype=np.float32) * np.float32(2.5)
    tl = dl + rng.standard_normal((B, R, V), dtype=np.float32) * np.float32(0.7)

    def probs(z):
        out = np.empty(z.shape, np.float32)
        for b in range(z.shape[0]):
            y = z[b].astype(np.float64)
            y = np.exp(y - y.max(axis=-1, keepdims=True))
            out[b] = (y / y.sum(axis=-1, keepdims=True)).astype(np.float32)
        return out

    q = probs(dl[:, :D, :])
    p = probs(tl)
    drafts = _sample_rows(rng, dl[:, :D, :].reshape(B * D, V)).reshape(B, D)
    return dict(B=B, D=D, V=V, dtype="f32", target_probs=p.reshape(B * R, V),
                draft_probs=q, draft_tokens=drafts, seed=request_seeds(B),
                offset=np.arange(B, dtype=np.int64))


def gumbel(B: int = 512, N: int = 4, V: int = 201088, real_vocab: int = 200019,
           cfg_id: int = 4, greedy_frac: float = 0.25, want_f32: bool = True) -> dict:
    """bf16 logits ~ N(0, 3^2) + Zipf over the real ids, -inf pads up to V; per
    request T ~ U[0.3, 1.5], T = 0 (greedy) for greedy_frac of the requests."""
    rng = _rng(cfg_id)
    rows = B * N
    real = min(real_vocab, V)
    x = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(3.0)
    x[:, :real] += zipf_bias(real)[None, :]
    x[:, real:] = -np.inf
    bits = bf16_bits_from_f32(x)
    del x
    T = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    T[rng.random(B) < greedy_frac] = 0.0
    return dict(B=B, N=N, V=V, real_vocab=real, dtype="bf16", logits_bits=bits,
                logits=f32_from_bf16_bits(bits) if want_f32 else None,
                temperature_req=T, temperature=np.repeat(T, N).astype(np.float32),
                seed=request_seeds(B), offset=np.arange(B, dtype=np.int64))


def verify_step(B: int = 512, D: int = 3, V: int = 201088, real_vocab: int = 200019,
                cfg_id: int = 5, greedy_frac: float = 0.25, want_f32: bool = False,
                sample_drafts: bool = True) -> dict:
    """The largest verify step: B requests of D+1 rows over the padded vocabulary of
    the Gumbel workload (bf16 N(0, 3^2) + Zipf, -inf pads), with the target-only
    knob distributions (T ~ U[0.3, 1.5] with greedy_frac greedy requests, top_k and
    top_p from their choice sets). Draft j is drawn from softmax(row j / T) w.p. 0.6
    (argmax for greedy requests), else a uniform random real id."""
    rng = _rng(cfg_id)
    R = D + 1
    rows = B * R
    real = min(real_vocab, V)
    x = rng.standard_normal((rows, V), dtype=np.float32) * np.float32(3.0)
    x[:, :real] += zipf_bias(real)[None, :]
    x[:, real:] = -np.inf
    bits = bf16_bits_from_f32(x)
    del x
    f32 = f32_from_bf16_bits(bits)
    T = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    T[rng.random(B) < greedy_frac] = 0.0
    top_k = rng.choice(np.array(TOPK_CHOICES, np.int32), size=B).astype(np.int32)
    top_p = rng.choice(np.array(TOPP_CHOICES, np.float32), size=B).astype(np.float32)
    lg = f32.reshape(B, R, V)[:, :D, :real]
    if sample_drafts:
        Tr = np.maximum(T, 1e-2)[:, None, None]
        sampled = _sample_rows(rng, (lg / Tr).reshape(B * D, real)).reshape(B, D)
    else:
        sampled = np.argmax(lg, axis=-1).astype(np.int32)
    am = np.argmax(lg, axis=-1).astype(np.int32)
    sampled = np.where((T == 0)[:, None], am, sampled)
    rnd = rng.integers(0, real, size=(B, D), dtype=np.int32)
    drafts = np.where(rng.random((B, D)) < 0.6, sampled, rnd).astype(np.int32)
    return dict(B=B, D=D, V=V, real_vocab=real, dtype="bf16", logits_bits=bits,
                logits=f32 if want_f32 else None, temperature=T, top_k=top_k,
                top_p=top_p, draft_tokens=drafts, seed=request_seeds(B),
                offset=np.arange(B, dtype=np.int64))
