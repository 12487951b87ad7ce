#!/usr/bin/env python
"""Benchmark of the verify-and-sample step on GB300.

Default workload (the largest verify step): 512 requests x (D+1 = 4) target rows over a
201088-token vocabulary (200019 real ids, -inf pads), bf16 logits ~ N(0, 3^2) + Zipf(1.1)
bias, per-request temperature ~ U[0.3, 1.5] with 25% greedy requests, top_k in
{0, 20, 50, 1000}, top_p in {1.0, 0.95, 0.9}, drafts drawn from the target row w.p. 0.6.
One step = one ts_chain_spec_sampling call (target-only, from logits): softmax with
temperature, fused top-k/top-p renorm, accept tests, chain scan and the corrected/bonus
draw, for every row, in one launch. Inputs (824 MB) exceed the 129 MB L2, so no flush.

Metric: verified rows/s = batch*(D+1) / step time (whole job over all GPUs), plus the
achieved HBM bandwidth of the step (logit bytes read once) against the measured peak.
Extra "legs" time the other calls on their workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-legs]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified rows/sec (batch×(D+1)) and achieved HBM GB/s vs 8 TB/s peak"
WORKLOAD = "verify step: target-only chain sampling from bf16 logits, B=512, D=3, V=201088"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-legs", action="store_true")
    ap.add_argument("--legs-only", action="store_true",
                    help="time only the legs (no headline step, no CPU baseline): profiling")
    ap.add_argument("--leg", default=None,
                    help="run only the legs whose name contains this string")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the oracle checks of the legs' outputs (boundary counts)")
    ap.add_argument("--cpu-sample", type=int, default=48,
                    help="requests in the single-core CPU baseline sample "
                         "(0: no CPU baseline, for profiling runs)")
    ap.add_argument("--knobs", default=None,
                    help="T,top_k,top_p applied to every request (profiling one selection route)")
    ap.add_argument("--batch", type=int, default=512,
                    help="requests per step (512 = the benchmark workload; smaller for profiling)")
    return ap.parse_args()


# ---- distributed plumbing (replicas: no data-path collective) ---------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def dist_init(backend: str):
    import torch.distributed as dist

    rank, local, world = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (the job is as slow as its slowest rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- measurement helpers ----------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_entry(kernel: str, workload: str):
    """The whole record of an ncu capture of this kernel and workload (or None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            return json.load(f).get(f"{kernel}|{workload}")
    except Exception:
        return None


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture of this kernel and workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(f"{kernel}|{workload}")
        if e is None or e.get("bytes_per_launch") is None:
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


def time_device(fn, steps: int, warmup: int, device, per_step: bool = False, flush=None):
    """Mean device time of one fn() call over `steps` timed calls (CUDA events on the
    launching stream, barrier + synchronize on both sides, max over ranks). With per_step,
    also the 10th, 50th and 90th percentiles of the per-call times (an event between
    consecutive calls). With flush (a device buffer larger than L2), the buffer is written
    before every call, outside the events, so each call starts with a cold L2."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    s = torch.cuda.current_stream()
    if flush is not None:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(s)
            fn()
            ev[i][1].record(s)
        torch.cuda.synchronize()
        barrier()
        each = np.array([a.elapsed_time(b) for a, b in ev])
        ms = max_over_ranks(float(each.mean()), device)
        if not per_step:
            return ms
        return ms, {"p10": float(np.percentile(each, 10)), "p50": float(np.percentile(each, 50)),
                    "p90": float(np.percentile(each, 90))}
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1 if per_step else 2)]
    ev[0].record(s)
    for i in range(steps):
        fn()
        if per_step:
            ev[i + 1].record(s)
    if not per_step:
        ev[1].record(s)
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(ev[0].elapsed_time(ev[-1]) / steps, device)
    if not per_step:
        return ms
    each = np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(steps)])
    return ms, {"p10": float(np.percentile(each, 10)), "p50": float(np.percentile(each, 50)),
                "p90": float(np.percentile(each, 90))}


# ---- the workload -----------------------------------------------------------------------

def main_workload(batch: int = 512, knobs=None):
    from speculative_decoding_verify_temp_gb300 import synth

    d = synth.verify_step(B=batch, D=3, V=201088, real_vocab=200019)
    if knobs:
        T, k, p = knobs.split(",")
        d["temperature"][:] = float(T)
        d["top_k"][:] = int(k)
        d["top_p"][:] = float(p)
    return d


def _oracle_slice(task):
    """One slice of requests through the oracle (runs in a spawned process)."""
    import oracle
    from speculative_decoding_verify_temp_gb300 import synth

    bits, D, drafts, kw = task
    return oracle.chain_spec_sampling(synth.f32_from_bf16_bits(bits), True, D, drafts,
                                      logprobs=False, **kw)


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip() in ("model name", "Model", "CPU part"):
                    return v.strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(d, nreq: int, gpu_out=None):
    """The oracle, as it stands, on the host cores: on one core over the first nreq
    requests, and over every core (requests in slices, one spawned process each) over the
    whole step. The whole-step run also checks the GPU's outputs of the same step request
    by request (exact tokens and lengths outside the boundary band)."""
    import multiprocessing

    import oracle
    from speculative_decoding_verify_temp_gb300 import synth

    oracle.build()
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    nreq = min(nreq, B)
    keys = ("temperature", "top_k", "top_p", "seed", "offset")
    x = synth.f32_from_bf16_bits(d["logits_bits"][: nreq * R])
    t0 = time.perf_counter()
    oracle.chain_spec_sampling(x, True, D, d["draft_tokens"][:nreq], logprobs=False,
                               **{k: d[k][:nreq] for k in keys})
    dt1 = time.perf_counter() - t0
    single = {"value": nreq * R / dt1, "unit": "rows/s", "cores": 1,
              "sample": f"first {nreq} requests ({nreq * R} rows), {dt1:.1f} s"}
    procs = max(1, os.cpu_count() or 1)
    step = -(-B // procs)
    tasks = [(np.ascontiguousarray(d["logits_bits"][b * R:min(B, b + step) * R]), D,
              np.ascontiguousarray(d["draft_tokens"][b:b + step]),
              {k: d[k][b:b + step] for k in keys}) for b in range(0, B, step)]
    with multiprocessing.get_context("spawn").Pool(len(tasks)) as pool:
        pool.map(_oracle_slice, [(t[0][:R], D, t[2][:1], {k: v[:1] for k, v in t[3].items()})
                                 for t in tasks])  # warm the workers (imports, builds)
        t0 = time.perf_counter()
        parts = pool.map(_oracle_slice, tasks)
        dtn = time.perf_counter() - t0
    ref = {k: np.concatenate([p[k] for p in parts]) for k in ("accepted_tokens", "accept_length",
                                                               "margin")}
    out = {"value": B * R / dtn, "unit": "rows/s", "cores": procs, "kind": "oracle",
           "sample": f"the whole step ({B} requests, {B * R} rows) in {len(tasks)} slices over "
                     f"{procs} processes, {dtn:.1f} s",
           "cpu_model": _cpu_model(), "single_core": single}
    if gpu_out is not None:
        ok = ref["margin"] > 1e-6
        acc, alen = gpu_out
        mism = int(((acc != ref["accepted_tokens"]).any(axis=1) | (alen != ref["accept_length"]))[ok].sum())
        out["parity"] = {"requests": int(B), "mismatches_outside_boundary": mism,
                         "boundary_requests": int((~ok).sum()), "boundary": "margin <= 1e-6"}
    return out


def run_reference(args):
    """The oracle, as it stands, timed on the host cores on the same workload: every step
    runs the whole verify step (all requests), the requests split in slices over one
    spawned process per core."""
    rank, _, world = dist_env()
    if world > 1 and rank != 0:
        return
    import multiprocessing

    import oracle

    oracle.build()
    d = main_workload(args.batch, args.knobs)
    B, D = d["B"], d["D"]
    R = D + 1
    keys = ("temperature", "top_k", "top_p", "seed", "offset")
    procs = max(1, os.cpu_count() or 1)
    step_n = -(-B // procs)
    tasks = [(np.ascontiguousarray(d["logits_bits"][b * R:min(B, b + step_n) * R]), D,
              np.ascontiguousarray(d["draft_tokens"][b:b + step_n]),
              {k: d[k][b:b + step_n] for k in keys}) for b in range(0, B, step_n)]
    with multiprocessing.get_context("spawn").Pool(len(tasks)) as pool:
        for _ in range(args.warmup):
            pool.map(_oracle_slice, tasks)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.map(_oracle_slice, tasks)
        dt = (time.perf_counter() - t0) / args.steps
    v = B * R / dt
    sample = (f"the whole step ({B} requests, {B * R} rows) each step, in {len(tasks)} slices "
              f"over {procs} processes")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if B == 512 else WORKLOAD.replace("B=512", f"B={B}"),
                   "batch": B, "D": D, "vocab": d["V"], "logits": "bf16"},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": procs, "kind": "oracle",
                         "sample": sample, "cpu_model": _cpu_model()},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_ours(args):
    import torch

    rank, local, world = dist_init("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__
    from speculative_decoding_verify_temp_gb300 import synth
    from speculative_decoding_verify_temp_gb300 import tsverify as tv

    __graft_entry__.build() if rank == 0 else None
    barrier()
    tv.load()
    peak, peak_kind = measured_peaks()

    d = main_workload(args.batch, args.knobs)
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    rows = B * R
    bits = np.ascontiguousarray(d["logits_bits"]).view(np.int16)
    logits = torch.from_numpy(bits).to(device).view(torch.bfloat16)
    drafts = torch.from_numpy(d["draft_tokens"]).to(device)
    T = torch.from_numpy(d["temperature"]).to(device)
    K = torch.from_numpy(d["top_k"]).to(device)
    P = torch.from_numpy(d["top_p"]).to(device)
    seed = torch.from_numpy(d["seed"]).to(device)
    off = torch.from_numpy(d["offset"]).to(device)
    ws = tv.make_workspace(B, R, V, device)
    outs = tv._chain_outputs(B, R, device, False, False)
    kw = dict(temperature=T, top_k=K, top_p=P, seed=seed, offset=off, workspace=ws, outputs=outs)

    def step():
        tv.chain_spec_sampling(logits, True, D, drafts, **kw)

    if args.legs_only:
        legs = run_legs(args, d, logits, device, tv, synth, peak)
        if rank == 0:
            print(json.dumps({"legs": legs}))
        return

    alg_bytes = rows * V * 2  # the logits, read once
    with ClockSampler(local) as clk:
        ms, pct = time_device(step, args.steps, args.warmup, device, per_step=True)
    clocks = clk.summary()
    gpu_out = (outs[0].cpu().numpy(), outs[1].cpu().numpy())  # the last timed step's
    value = world * rows / (ms / 1e3)
    achieved = alg_bytes / (ms / 1e3) / 1e9

    # end to end through the public API with host buffers
    pin_logits = torch.from_numpy(bits).pin_memory()
    pin_small = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                 for a in (d["draft_tokens"], d["temperature"], d["top_k"], d["top_p"],
                           d["seed"], d["offset"])]
    dev_small = [drafts, T, K, P, seed, off]
    host_acc = torch.empty((B, R), dtype=torch.int32).pin_memory()
    host_len = torch.empty((B,), dtype=torch.int32).pin_memory()
    h2d = pin_logits.numel() * 2 + sum(t.numel() * t.element_size() for t in pin_small)
    d2h = host_acc.numel() * 4 + host_len.numel() * 4

    def e2e_step():
        logits.view(torch.int16).copy_(pin_logits, non_blocking=True)
        for dst, src in zip(dev_small, pin_small):
            dst.copy_(src, non_blocking=True)
        r = tv.chain_spec_sampling(logits, True, D, drafts, **kw)
        host_acc.copy_(r["accepted_tokens"], non_blocking=True)
        host_len.copy_(r["accept_length"], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 10))
    ms_e2e = time_device(e2e_step, e2e_steps, 2, device)
    e2e = {"value": world * rows / (ms_e2e / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e}

    legs = {}
    if not args.no_legs:
        legs = run_legs(args, d, logits, device, tv, synth, peak)

    if rank != 0:
        return
    cpu = cpu_baseline(d, args.cpu_sample, gpu_out) if args.cpu_sample > 0 else None
    traffic = ncu_traffic("k_chain", "verify_step") if B == 512 else None
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "ms_per_step_percentiles": pct,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if B == 512 else WORKLOAD.replace("B=512", f"B={B}"),
                   "batch": B, "D": D, "vocab": V, "real_vocab": 200019,
                   "logits": "bf16", "greedy_requests": 0.25,
                   "top_k": "uniform {0,20,50,1000}", "top_p": "uniform {1.0,0.95,0.9}",
                   "temperature": "U[0.3,1.5]",
                   "l2": f"inputs {alg_bytes / 1e6:.0f} MB vs 129 MB L2 (no flush)",
                   "parallelism": f"replicas x{world}",
                   **({"knobs_override": args.knobs} if args.knobs else {})},
        "hbm_gbs": achieved, "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic,
                     "kernel": "k_chain<bf16> (the step: a one-CTA planning launch, it, then the one-thread-a-request chain writer)",
                     "timed": "the whole step (all three launches) with CUDA events",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "legs": legs,
    }
    print(json.dumps(line))


_POOL = None


def _oracle_pool():
    """One spawned process per host core for the oracle checks of the legs."""
    global _POOL
    if _POOL is None:
        import multiprocessing

        _POOL = multiprocessing.get_context("spawn").Pool(max(1, os.cpu_count() or 1))
    return _POOL


def _oracle_task(task):
    """One slice of rows or requests through the oracle (runs in a spawned process)."""
    import oracle
    from speculative_decoding_verify_temp_gb300 import synth

    kind, x, is_bits, args, kw = task
    x = synth.f32_from_bf16_bits(x) if is_bits else x
    if kind == "gumbel":
        return oracle.gumbel_max_sample(x, *args, **kw)
    if kind == "greedy":
        return oracle.verify_chain_greedy(x, *args, **kw)
    if kind == "sample":
        return oracle.sample_from_logits(x, *args, **kw)
    return oracle.chain_spec_sampling(x, *args, **kw)


def leg_parity(kind, x, is_bits, R, args_req, kw_req, gpu, extra=None):
    """Check a leg's outputs (from its last timed call) against the oracle over every
    request, in slices across the host cores: exact tokens and lengths on every request
    whose decision margin exceeds 1e-6; the others are counted as boundary requests.
    args_req / kw_req: per-request arrays (sliced) and scalars (kept) for the oracle."""
    B = x.shape[0] // R
    procs = max(1, os.cpu_count() or 1)
    step = -(-B // procs)

    def cut(v, b0, b1, per_row):
        if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] in (B, B * R):
            lo, hi = (b0 * R, b1 * R) if (per_row or v.shape[0] == B * R) else (b0, b1)
            return np.ascontiguousarray(v[lo:hi])
        return v

    tasks = []
    for b0 in range(0, B, step):
        b1 = min(B, b0 + step)
        xa = np.ascontiguousarray(x[b0 * R:b1 * R])
        a = [cut(v, b0, b1, False) for v in args_req]
        k = {n: cut(v, b0, b1, False) for n, v in kw_req.items()}
        if extra is not None:
            # draft-side rows: [B, D, V] or [B * D, V]
            k.update({n: np.ascontiguousarray(v[b0:b1] if v.shape[0] == B
                                              else v[b0 * (R - 1):b1 * (R - 1)])
                      for n, v in extra.items()})
        tasks.append((kind, xa, is_bits, a, k))
    parts = _oracle_pool().map(_oracle_task, tasks)
    if kind in ("gumbel", "sample"):
        if kind == "gumbel":
            want = np.concatenate([p[0] for p in parts])
            marg = np.concatenate([p[1] for p in parts])
        else:
            want = np.concatenate([p["tokens"] for p in parts])
            marg = np.concatenate([p["margin"] for p in parts])
        ok = marg > 1e-6
        mism = int((gpu[0] != want)[ok].sum())
        return {"rows": int(len(want)), "mismatches_outside_boundary": mism,
                "boundary_rows": int((~ok).sum()), "boundary": "margin <= 1e-6"}
    acc = np.concatenate([p["accepted_tokens"] for p in parts])
    alen = np.concatenate([p["accept_length"] for p in parts])
    if kind == "greedy":
        mism = int(((gpu[0] != acc).any(axis=1) | (gpu[1] != alen)).sum())
        return {"requests": int(B), "mismatches": mism}
    ok = np.concatenate([p["margin"] for p in parts]) > 1e-6
    mism = int((((gpu[0] != acc).any(axis=1)) | (gpu[1] != alen))[ok].sum())
    return {"requests": int(B), "mismatches_outside_boundary": mism,
            "boundary_requests": int((~ok).sum()), "boundary": "margin <= 1e-6"}


def run_legs(args, d, logits, device, tv, synth, peak):
    """The other calls, each on its own workload (mean device time per call), with the
    oracle's check of each leg's outputs (boundary counts per configuration) unless
    --no-parity."""
    import torch

    legs = {}
    steps, warm = max(5, args.steps), 3
    B, D, V = d["B"], d["D"], d["V"]
    R = D + 1
    rows = B * R
    parity = not args.no_parity
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # > the 129 MB L2

    def want(name):
        return args.leg is None or args.leg in name

    def rec(name, ms, nrows, nbytes, launches=1, **more):
        legs[name] = {"ms": ms, "rows_per_s": nrows / (ms / 1e3),
                      "hbm_gbs": nbytes / (ms / 1e3) / 1e9,
                      "frac_of_peak": nbytes / (ms / 1e3) / 1e9 / peak, "launches": launches}
        legs[name].update(more)

    def host(t):
        return t.cpu().numpy()

    bits = d["logits_bits"]
    drafts = torch.from_numpy(d["draft_tokens"]).to(device)
    Trow_np = np.repeat(d["temperature"], R).astype(np.float32)
    Trow = torch.from_numpy(Trow_np).to(device)
    seed = torch.from_numpy(d["seed"]).to(device)
    off = torch.from_numpy(d["offset"]).to(device)
    # greedy chain verification on the same logits (the greedy gate)
    name = "greedy_verify_B512_D3_V201088_bf16"
    if want(name):
        ws = tv.make_workspace(B, R, V, device)
        outs = tv._chain_outputs(B, R, device, False, False)
        ms = time_device(lambda: tv.verify_chain_greedy(logits, D, drafts, ws, outputs=outs),
                         steps, warm, device)
        rec(name, ms, rows, rows * V * 2)
        if parity:
            legs[name]["parity"] = leg_parity("greedy", bits, True, R, [D, d["draft_tokens"]], {},
                                              (host(outs[0]), host(outs[1])))
    # Gumbel-max on the same logits as 512 requests x 4 rows, greedy rows included
    name = "gumbel_B512_N4_V201088_bf16"
    if want(name):
        wsg = tv.make_workspace(B, R, V, device)
        tok = torch.empty(rows, dtype=torch.int32, device=device)
        ms = time_device(lambda: tv.gumbel_max_sample(logits, R, Trow, seed, off, wsg, out=tok),
                         steps, warm, device)
        alu = ncu_entry("k_gumbel", "gumbel_B512")
        rec(name, ms, rows, rows * V * 2, alu=alu)
        if parity:
            legs[name]["parity"] = leg_parity("gumbel", bits, True, R,
                                              [R, Trow_np, d["seed"], d["offset"]], {},
                                              (host(tok),))
    # the verify step with every output on (logprobs at temperature 1, accept_index)
    name = "verify_step_with_logprobs_B512_D3_V201088_bf16"
    if want(name):
        outs = tv._chain_outputs(B, R, device, True, True)
        kw = dict(temperature=torch.from_numpy(d["temperature"]).to(device),
                  top_k=torch.from_numpy(d["top_k"]).to(device),
                  top_p=torch.from_numpy(d["top_p"]).to(device), seed=seed, offset=off,
                  workspace=tv.make_workspace(B, R, V, device), outputs=outs)
        ms = time_device(lambda: tv.chain_spec_sampling(logits, True, D, drafts, **kw), steps,
                         warm, device)
        rec(name, ms, rows, rows * V * 2, launches=3)
        if parity:
            legs[name]["parity"] = leg_parity(
                "chain", bits, True, R, [True, D, d["draft_tokens"]],
                {k: d[k] for k in ("temperature", "top_k", "top_p", "seed", "offset")} |
                {"logprobs": False}, (host(outs[0]), host(outs[1])))
    # the Gumbel-max vocabulary sweep: V in {32000, 128256, 201088} x B in {1, 32, 512}, N = 4
    # (the 201088 logits are the step's; the others are generated by the same recipe)
    for Vs in (32000, 128256, 201088):
        if not want(f"gumbel_sweep_B1_N4_V{Vs}") and not want(f"gumbel_sweep_B32_N4_V{Vs}") \
                and not want(f"gumbel_sweep_B512_N4_V{Vs}"):
            continue
        if Vs == V:
            gl, Trs, gseed, goff = logits, Trow, seed, off
        else:
            gsw = synth.gumbel(B=512, N=4, V=Vs, real_vocab=min(Vs, 200019), want_f32=False)
            gl = torch.from_numpy(np.ascontiguousarray(gsw["logits_bits"]).view(np.int16)).to(
                device).view(torch.bfloat16)
            Trs = torch.from_numpy(gsw["temperature"]).to(device)
            gseed = torch.from_numpy(gsw["seed"]).to(device)
            goff = torch.from_numpy(gsw["offset"]).to(device)
        for Bs in (1, 32, 512):
            name = f"gumbel_sweep_B{Bs}_N4_V{Vs}_bf16"
            if not want(name):
                continue
            # the smaller batches take successive slices of the 2048-row buffer, call by
            # call, so that consecutive calls do not read the same rows
            nr = Bs * 4
            wss = tv.make_workspace(Bs, 4, Vs, device)
            toks = torch.empty(nr, dtype=torch.int32, device=device)
            nsl = 512 // Bs
            sl = [(gl[i * nr:(i + 1) * nr], Trs[i * nr:(i + 1) * nr], gseed[i * Bs:(i + 1) * Bs],
                   goff[i * Bs:(i + 1) * Bs]) for i in range(nsl)]
            cur = [0]

            def call():
                xs, ts, ss, os_ = sl[cur[0] % nsl]
                cur[0] += 1
                tv.gumbel_max_sample(xs, 4, ts, ss, os_, wss, out=toks)

            ms = time_device(call, max(steps, 50), warm, device)
            more = {}
            if Bs < 512:
                more["ms_l2_flushed"] = time_device(call, max(steps, 50), warm, device,
                                                    flush=flush)
            rec(name, ms, nr, nr * Vs * 2, **more)
        del gl
    # single-step sampling of the same logits (2048 rows, joint top-k/top-p order)
    kn_rows = {k: torch.from_numpy(np.repeat(d[k], R)).to(device)
               for k in ("temperature", "top_k", "top_p")}
    name = "sample_joint_R2048_V201088_bf16"
    if want(name):
        wss = tv.make_workspace(rows, 1, V, device)
        stok = torch.empty(rows, dtype=torch.int32, device=device)
        ms = time_device(lambda: tv.sample_from_logits(logits, R, **kn_rows, joint=True, seed=seed,
                                                       offset=off, workspace=wss, out=stok),
                         steps, warm, device)
        rec(name, ms, rows, rows * V * 2, launches=3)
        if parity:
            legs[name]["parity"] = leg_parity(
                "sample", bits, True, R, [R],
                {"temperature": Trow_np, "top_k": np.repeat(d["top_k"], R).astype(np.int32),
                 "top_p": np.repeat(d["top_p"], R).astype(np.float32), "joint": True,
                 "seed": d["seed"], "offset": d["offset"]}, (host(stok),))
    # draft-side sampling with the kept distributions stored (min_p on), 2048 rows
    name = "draft_sample_with_probs_R2048_V201088_bf16"
    if want(name):
        wss = tv.make_workspace(rows, 1, V, device)
        stok = torch.empty(rows, dtype=torch.int32, device=device)
        pbuf = torch.empty((rows, V), dtype=torch.float32, device=device)
        mp = torch.full((rows,), 0.01, dtype=torch.float32, device=device)
        ms = time_device(lambda: tv.sample_from_logits(logits, R, **kn_rows, min_p=mp, seed=seed,
                                                       offset=off, workspace=wss, out=stok,
                                                       probs=pbuf),
                         steps, warm, device)
        rec(name, ms, rows, rows * V * (2 + 4), launches=4)
        del pbuf
    # the verify step with min_p and relaxed acceptance thresholds
    name = "verify_step_min_p_relaxed_B512_D3_V201088_bf16"
    if want(name):
        outs = tv._chain_outputs(B, R, device, False, False)
        mpr = torch.full((B,), 0.01, dtype=torch.float32, device=device)
        kw = dict(temperature=torch.from_numpy(d["temperature"]).to(device),
                  top_k=torch.from_numpy(d["top_k"]).to(device),
                  top_p=torch.from_numpy(d["top_p"]).to(device), seed=seed, offset=off,
                  workspace=tv.make_workspace(B, R, V, device), outputs=outs, min_p=mpr,
                  threshold_single=0.9, threshold_acc=0.5)
        ms = time_device(lambda: tv.chain_spec_sampling(logits, True, D, drafts, **kw), steps,
                         warm, device)
        rec(name, ms, rows, rows * V * 2, launches=3)
    # ragged verification: windows of 1 to 4 rows of the step's logits
    name = "verify_ragged_B512_D3_V201088_bf16"
    if want(name):
        rng = np.random.default_rng(512)
        lens = rng.integers(1, D + 2, B)
        qo_np = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        sel = np.concatenate([np.arange(b * R, b * R + lens[b]) for b in range(B)])
        packed = logits[torch.from_numpy(sel).to(device)]
        qo = torch.from_numpy(qo_np).to(device)
        outs = tv._chain_outputs(B, R, device, False, False)
        kw = dict(temperature=torch.from_numpy(d["temperature"]).to(device),
                  top_k=torch.from_numpy(d["top_k"]).to(device),
                  top_p=torch.from_numpy(d["top_p"]).to(device), seed=seed, offset=off,
                  workspace=tv.make_workspace(B, R, V, device), outputs=outs, qo_indptr=qo)
        ms = time_device(lambda: tv.chain_spec_sampling(packed, True, D, drafts, **kw), steps,
                         warm, device)
        nrow = int(qo_np[-1])
        rec(name, ms, nrow, nrow * V * 2, launches=3)
        del packed
    # softmax with temperature, fp32 probabilities out
    name = "softmax_B512_R4_V201088_bf16"
    if want(name):
        out = torch.empty((rows, V), dtype=torch.float32, device=device)
        ms = time_device(lambda: tv.softmax_temp(logits, Trow, out=out), steps, warm, device)
        rec(name, ms, rows, rows * V * 6)
        del out
    # greedy verification, small batch (latency-bound; L2-resident unless flushed)
    name = "greedy_verify_B64_D3_V32000_bf16"
    if want(name):
        g = synth.greedy_verify()
        gl = torch.from_numpy(np.ascontiguousarray(g["logits_bits"]).view(np.int16)).to(
            device).view(torch.bfloat16)
        gd = torch.from_numpy(g["draft_tokens"]).to(device)
        gws = tv.make_workspace(g["B"], g["D"] + 1, g["V"], device)
        gouts = tv._chain_outputs(g["B"], g["D"] + 1, device, False, False)

        def gcall():
            tv.verify_chain_greedy(gl, g["D"], gd, gws, outputs=gouts)

        ms = time_device(gcall, max(50, steps), 10, device)
        msf = time_device(gcall, max(50, steps), 10, device, flush=flush)
        grows = g["B"] * (g["D"] + 1)
        rec(name, ms, grows, grows * g["V"] * 2, ms_l2_flushed=msf)
        if parity:
            legs[name]["parity"] = leg_parity("greedy", g["logits_bits"], True, g["D"] + 1,
                                              [g["D"], g["draft_tokens"]], {},
                                              (host(gouts[0]), host(gouts[1])))
    # target-only chain sampling, B=128 D=4 V=128256
    name = "target_only_B128_D4_V128256_bf16"
    if want(name):
        c = synth.target_only()
        cl = torch.from_numpy(np.ascontiguousarray(c["logits_bits"]).view(np.int16)).to(
            device).view(torch.bfloat16)
        couts = tv._chain_outputs(c["B"], c["D"] + 1, device, False, False)
        ca = dict(temperature=torch.from_numpy(c["temperature"]).to(device),
                  top_k=torch.from_numpy(c["top_k"]).to(device),
                  top_p=torch.from_numpy(c["top_p"]).to(device),
                  seed=torch.from_numpy(c["seed"]).to(device),
                  offset=torch.from_numpy(c["offset"]).to(device),
                  workspace=tv.make_workspace(c["B"], c["D"] + 1, c["V"], device), outputs=couts)
        cd = torch.from_numpy(c["draft_tokens"]).to(device)
        ms = time_device(lambda: tv.chain_spec_sampling(cl, True, c["D"], cd, **ca), steps, warm,
                         device)
        crows = c["B"] * (c["D"] + 1)
        rec(name, ms, crows, crows * c["V"] * 2, launches=3)
        if parity:
            legs[name]["parity"] = leg_parity(
                "chain", c["logits_bits"], True, c["D"] + 1, [True, c["D"], c["draft_tokens"]],
                {k: c[k] for k in ("temperature", "top_k", "top_p", "seed", "offset")} |
                {"logprobs": False}, (host(couts[0]), host(couts[1])))
        del cl
    # rejection sampling with draft probabilities, B=256 D=7 V=151936 (fp32 probs), and the
    # top-k/top-p renorm of the same probabilities with the target-only knob mix
    if want("rejection_B256_D7_V151936_f32") or want("renorm_R2048_V151936_f32"):
        r = synth.rejection()
        rp = torch.from_numpy(r["target_probs"]).to(device)
        rrows = r["B"] * (r["D"] + 1)
    name = "rejection_B256_D7_V151936_f32"
    if want(name):
        rq = torch.from_numpy(r["draft_probs"]).to(device)
        routs = tv._chain_outputs(r["B"], r["D"] + 1, device, False, True)
        ra = dict(draft_probs=rq, seed=torch.from_numpy(r["seed"]).to(device),
                  offset=torch.from_numpy(r["offset"]).to(device),
                  workspace=tv.make_workspace(r["B"], r["D"] + 1, r["V"], device), outputs=routs)
        rd = torch.from_numpy(r["draft_tokens"]).to(device)
        res = tv.chain_spec_sampling(rp, False, r["D"], rd, **ra)
        alen = res["accept_length"].cpu().numpy()
        # algorithmic bytes: the row the draw needs (p, plus q for a rejection) and the
        # accepted-prefix scalars
        need = sum((2 if L <= r["D"] else 1) for L in alen) * r["V"] * 4
        ms = time_device(lambda: tv.chain_spec_sampling(rp, False, r["D"], rd, **ra), steps, warm,
                         device)
        rec(name, ms, rrows, need)
        if parity:
            legs[name]["parity"] = leg_parity(
                "chain", r["target_probs"], False, r["D"] + 1, [False, r["D"], r["draft_tokens"]],
                {"seed": r["seed"], "offset": r["offset"], "logprobs": False},
                (host(routs[0]), host(routs[1])), extra={"draft_probs": r["draft_probs"]})
        del rq
    name = "renorm_R2048_V151936_f32"
    if want(name):
        rng = np.random.default_rng(1)
        kk = torch.from_numpy(rng.choice(np.array(synth.TOPK_CHOICES, np.int32), rrows)).to(device)
        pp = torch.from_numpy(rng.choice(np.array(synth.TOPP_CHOICES, np.float32), rrows)).to(
            device)
        ro = torch.empty_like(rp)
        ms = time_device(lambda: tv.topk_topp_renorm(rp, kk, pp, out=ro), steps, warm, device)
        rec(name, ms, rrows, rrows * r["V"] * 8)
    return legs


def main():
    args = parse()
    try:
        if args.impl == "reference":
            run_reference(args)
        else:
            run_ours(args)
    finally:
        if _POOL is not None:
            _POOL.close()
            _POOL.join()


if __name__ == "__main__":
    main()
