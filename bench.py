"""Benchmark of batched speculative-decoding verification on GB300.

One step = one spec_verify call over the whole batch (every row's statistics and filtering,
the draft gathers, the first-rejection scan and the residual / extra-token draws).  The
default workload is B=256 requests x k=4 drafts over V=128256 (bf16 Zipf-shaped logits,
top-k 50, top-p 0.9, a quarter greedy).  Inputs are synthetic and seeded; three device copies
of the two large inputs (0.85 GB each set) rotate between steps so no step reads inputs left
in L2 by the one before.

--scheme onehot times the one-hot-draft entry point instead (drafts = the argmax of each draft
row's q; every row is sampled and the matching prefix kept; q is not read).  --scheme lazy times
spec_verify_lazy, which reads no row after a request's first rejection.

Prints one JSON line (rank 0).  --impl reference times the float64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify rows/s and achieved HBM GB/s (% of GB300 roofline) vs CPU oracle"

# DRAM bytes (read + write) of one stream-kernel launch on the full batch, from the ncu capture
# summarised under profiles/ (a 160-request cut, scaled by rows).  Valid only for the kernel as
# captured; absent (null) otherwise.
TRAFFIC_STREAM_KERNEL = {"b256_k4_v128256_bf16_zipf": 335.3e6}
DEFAULT_WORKLOAD = "b256_k4_v128256_bf16_zipf"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def algorithmic_bytes(w, accept_len, onehot=False, lazy=False) -> dict:
    """Bytes the method must move for one call (see the design notes, 'Measurement').

    Every target row of every request (the one-pass design cannot skip rows before knowing
    where the rejection falls); one 32-byte sector of q per sampled draft (q(x_i)); at a
    rejected sampled row whose kept set is cut by top-k (0 < top_k < V), one 32-byte q sector
    per kept token (at most top_k: the residual max(0, p - q) is zero outside the kept set);
    at a rejected sampled row without top-k, the whole q row plus a re-read of the target row;
    small per-row/per-request I/O (8 B per row, 4 B per draft, 4 (k_max + 2) + 24 B per
    request).  The one-hot scheme reads no q: the target rows and the I/O only.  The lazy scheme
    needs only each request's rows up to the one where it stops (a_b + 1 rows, with a_b its
    accept length) and the q sectors of the drafts on that path; `rows_read` is what its two
    phases read: every row 0, then rows 1..k of the requests that kept draft 0.
    """
    esz = 2 if w.dtype == "bf16" else 4
    V = w.V
    nd = w.num_drafts.astype(np.int64)
    rows = int((nd + 1).sum())
    sampled = w.greedy == 0
    a = np.where(accept_len >= 0, np.minimum(accept_len, nd), nd).astype(np.int64)
    b_rows = (int((a + 1).sum()) if lazy else rows) * V * esz
    on_path = np.minimum(a + 1, nd) if lazy else nd
    b_q = 0 if onehot else int(on_path[sampled].sum()) * 32
    b_rej = 0
    for b in ([] if onehot else np.nonzero(sampled & (accept_len < nd) & (accept_len >= 0))[0]):
        K = int(w.top_k[b])
        if 0 < K < V:
            b_rej += 32 * K
        else:
            b_rej += V * esz + V * 4
    b_io = rows * 8 + int(nd.sum()) * 4 + w.B * (4 * (w.k_max + 2) + 24)
    total = b_rows + b_q + b_rej + b_io
    b_json = rows * V * esz + int(nd.sum()) * V * 4 + int(((accept_len < nd) & (accept_len >= 0)).sum()) * V * esz
    out = dict(total=total, rows=b_rows, q_sectors=b_q, rejected=b_rej, io=b_io, baseline_json_formula=b_json)
    if lazy:
        kept0 = (accept_len >= 1) & (nd >= 1)
        out["rows_read"] = int(w.B + nd[kept0].sum()) * V * esz
    return out


def launches_per_call(w, scheme: str) -> int:
    """Kernels one call launches: the workspace clear, the history prepass with a history, then
    the stream and select kernels (the lazy scheme: both for row 0, both for the queued rows,
    and the residual kernel; only the first pair when no request has drafts)."""
    n = 1 + (1 if getattr(w, "prior_offsets", None) is not None else 0)
    if scheme == "lazy":
        return n + (2 if int(w.num_drafts.sum()) == 0 else 5)
    return n + 2


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(workload: str, seconds_target: float = 12.0, max_requests: int = 256, onehot=False):
    """The float64 oracle on the host cores, on a bounded sample of the same workload: the
    first (up to) 256 requests, verified repeatedly until about 12 s of wall time."""
    import oracle
    import sv_workloads as W
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    sp = W.spec(workload)
    n = min(sp.B, max_requests)
    w = W.make(workload, requests=range(n))
    if onehot:
        W.with_argmax_drafts(w)
    rows = int((w.num_drafts.astype(np.int64) + 1).sum())
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.verify(w, threads=cores, onehot=onehot)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds_target or reps >= 1000:
            break
    return {"value": rows * reps / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {sp.B} requests ({rows} rows) x {reps} repetitions, float64 C oracle, "
                      f"{cores} threads, {dt:.1f} s"}


def max_over_ranks(ms: float, device=None) -> float:
    """The slowest rank's time: the job's time is the max over its ranks (replicas each time
    their own K steps; the whole job ends when the slowest does)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, steps: int, ms_max: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return units_per_rank * world * steps / (ms_max / 1e3)


def workload_config(sp, w, world: int, onehot=False, lazy=False) -> dict:
    """The `config` object of a JSON line: the workload by name and its shape and filters."""
    def one(a):
        u = np.unique(np.asarray(a))
        return u.item() if u.size == 1 else "mixed"
    extra = {"scheme": "one-hot drafts (argmax of q): every row sampled, matching prefix kept"} if onehot else {}
    if lazy:
        extra = {"scheme": "lazy: row 0 of every request, then rows 1..k of those that kept draft 0"}
    return {**extra, "workload": sp.name, "B": int(w.B), "k": int(sp.k_max), "V": int(sp.V), "logits": sp.dtype,
            "top_k": one(w.top_k), "top_p": round(float(one(w.top_p)), 4) if one(w.top_p) != "mixed" else "mixed",
            "greedy_share": round(float(np.mean(w.greedy != 0)), 4), "ragged_k": w.row_offsets is not None,
            "parallelism": f"replicas x{world}"}


def run_reference(args, budget_s: float = 150.0):
    """--impl reference: the float64 oracle on the host cores, timed per step.  A step is a
    bounded sample of the workload (a prefix of its requests) sized from a probe so that
    warm-up plus timed steps take about `budget_s`."""
    import oracle
    import sv_workloads as W
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    sp = W.spec(args.workload)
    n_probe = min(sp.B, max(2 * cores, 32))
    onehot = args.scheme == "onehot"
    mk = lambda req: W.with_argmax_drafts(W.make(args.workload, requests=req)) if onehot else \
        W.make(args.workload, requests=req)
    w = mk(range(n_probe))
    t0 = time.perf_counter()
    oracle.verify(w, threads=cores, onehot=onehot)
    t_req = (time.perf_counter() - t0) / n_probe
    n = int(max(1, min(sp.B, budget_s / ((args.steps + args.warmup) * max(t_req, 1e-6)))))
    if n != n_probe:
        w = mk(range(n))
    rows = int((w.num_drafts.astype(np.int64) + 1).sum())
    for _ in range(args.warmup):
        oracle.verify(w, threads=cores, onehot=onehot)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify(w, threads=cores, onehot=onehot)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(sp, W.make(args.workload) if n != sp.B else w, args.gpus, onehot),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                             "sample": f"first {n} of {sp.B} requests ({rows} rows) per step, float64 C oracle, "
                                       f"{cores} threads"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sv_workloads as W
    import speculative_decoding_verification_12_gb300 as sv
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch, bound_call

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.lib()

    sp = W.spec(args.workload)
    onehot = args.scheme == "onehot"
    lazy = args.scheme == "lazy"
    w = W.make(args.workload, requests=None if args.requests is None else list(range(args.requests)))
    if onehot:
        W.with_argmax_drafts(w)
    db = DeviceBatch.from_host(w, dev, want_pq=False)
    stream = torch.cuda.Stream(dev)
    # rotate enough copies that the logits one round of calls reads are 2.5x the L2: a call
    # then never finds its rows left in L2 by the calls before it
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 126 << 20)
    logit_bytes = db.target_logits.numel() * db.target_logits.element_size()
    n_copies = args.copies if args.copies > 0 else max(3, -(-int(2.5 * l2) // logit_bytes))
    copies = [(db.target_logits, db.draft_probs)]
    for _ in range(n_copies - 1):
        # the one-hot scheme reads no q: only the target logits rotate
        copies.append((db.target_logits.clone(), db.draft_probs if onehot else db.draft_probs.clone()))
    with torch.cuda.stream(stream):
        calls = [bound_call(db, stream, t, d, onehot=onehot, lazy=lazy) for t, d in copies]
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        calls[i % len(calls)]()
    barrier()
    acc = db.accept_len.cpu().numpy()
    out_tok = db.out_tokens.cpu().numpy()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    ev0.record(stream)
    for i in range(args.steps):
        calls[i % len(calls)]()
    ev1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, dev)
    rows = int((w.num_drafts.astype(np.int64) + 1).sum())
    drafts = int(w.num_drafts.sum())
    per_step_ms = ms_max / args.steps
    value = whole_job_rate(rows, world, args.steps, ms_max)

    nb = algorithmic_bytes(w, acc, onehot, lazy)
    peak, peak_kind = peaks()
    achieved = nb["total"] / (ms / args.steps / 1e3) / 1e9

    # The dominant kernel alone: the library records two events around the stream kernel of
    # each call (sv_set_phase_events).  That separates the two kernels (no PDL overlap), so it
    # is a pass of its own after the timed region.
    lib = sv.lib()
    phase = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(0 if lazy else args.phase_steps)]
    for a, b in phase:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    for i, (a, b) in enumerate(phase):
        lib.sv_set_phase_events(a.cuda_event, b.cuda_event)
        calls[i % len(calls)]()
    lib.sv_set_phase_events(None, None)
    torch.cuda.synchronize(dev)
    stream_ms = float(np.mean([a.elapsed_time(b) for a, b in phase])) if phase else float("nan")
    stream_gbs = nb["rows"] / (stream_ms / 1e3) / 1e9

    # end to end through the C ABI from pinned host buffers: H2D inputs, verify, D2H results
    host = {
        "tl": torch.from_numpy(np.ascontiguousarray(w.target_logits).view(np.int16) if w.dtype == "bf16"
                               else w.target_logits).pin_memory(),
        "dt": torch.from_numpy(w.draft_tokens).pin_memory(),
        "u": torch.from_numpy(w.uniforms).pin_memory(),
    }
    if not onehot:
        host["dp"] = torch.from_numpy(w.draft_probs).pin_memory()
    pins_out = (torch.empty_like(db.out_tokens, device="cpu").pin_memory(),
                torch.empty_like(db.accept_len, device="cpu").pin_memory())
    tl_dev = db.target_logits.view(torch.int16) if w.dtype == "bf16" else db.target_logits
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in pins_out)

    def e2e_step():
        with torch.cuda.stream(stream):
            tl_dev.copy_(host["tl"], non_blocking=True)
            if not onehot:
                db.draft_probs.copy_(host["dp"], non_blocking=True)
            db.draft_tokens.copy_(host["dt"], non_blocking=True)
            db.uniforms.copy_(host["u"], non_blocking=True)
            calls[0]()
            pins_out[0].copy_(db.out_tokens, non_blocking=True)
            pins_out[1].copy_(db.accept_len, non_blocking=True)

    e2e_value = None
    if args.e2e_steps > 0:
        for _ in range(2):
            e2e_step()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        barrier()
        e2e_value = whole_job_rate(rows, world, args.e2e_steps, max_over_ranks(e0.elapsed_time(e1), dev))
        assert np.array_equal(pins_out[1].numpy(), acc), "end-to-end results differ from the device-resident run"

    entry = {"accept": "spec_verify", "onehot": "spec_verify_onehot", "lazy": "spec_verify_lazy"}[args.scheme]
    call = {"achieved": achieved, "frac": achieved / peak, "bytes": nb["total"], "us": per_step_ms * 1e3,
            "what": f"whole {entry} call: " + ("clear_kernel, stream_kernel + select_kernel over every row 0, "
                                               "the same over the queued rows, resid_kernel (PDL chain)" if lazy else
                                               "clear_kernel + stream_kernel + select_kernel (PDL chain)")}
    if lazy:
        # the lazy call's kernels overlap in one programmatic chain; its roofline is the call's
        roofline = {"bound": "hbm", "kernel": "whole spec_verify_lazy call", "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind, "algorithmic_bytes": nb["total"],
                    "kernel_us": per_step_ms * 1e3, "timed": "CUDA events around whole calls on the launching stream",
                    "traffic": args.traffic, "traffic_unit": "bytes per call (ncu dram read+write)", "call": call}
    else:
        roofline = {"bound": "hbm", "kernel": f"stream_kernel<{sp.dtype}>", "achieved": stream_gbs,
                    "peak": peak, "unit": "GB/s", "frac": stream_gbs / peak, "peak_source": peak_kind,
                    "algorithmic_bytes": nb["rows"], "kernel_us": stream_ms * 1e3,
                    "timed": f"CUDA events recorded by the library around the stream kernel on its stream, "
                             f"mean of {args.phase_steps} calls",
                    "traffic": args.traffic if args.traffic is not None else
                    (TRAFFIC_STREAM_KERNEL.get(sp.name) if args.requests is None and not onehot else None),
                    "traffic_unit": "bytes per launch (ncu dram read+write)", "call": call}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per_step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(sp, w, world, onehot, lazy),
                           l2=f"{n_copies} rotating device copies of the inputs; the logits of one round "
                              f"({n_copies * logit_bytes / 1e6:.0f} MB) are {n_copies * logit_bytes / l2:.1f}x the "
                              f"{l2 / 1e6:.0f} MB L2"),
            "draft_tokens_per_s": whole_job_rate(drafts, world, args.steps, ms_max),
            "hbm_gbs": achieved,
            "accept": {"mean_accept_len": float(acc.mean()), "accept_rate": float(acc.sum() / max(drafts, 1)),
                       "tokens_per_step": float(acc.mean() + 1)},
            "bytes_per_step": nb,
            "roofline": roofline,
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            # every kernel one call launches (launches_per_call), times the timed calls
            "gpu_launches": launches_per_call(w, args.scheme) * args.steps,
            "clocks": clk,
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(args.workload, onehot=onehot)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--copies", type=int, default=0,
                    help="rotating input copies (0: enough that one round's logits are 2.5x the L2)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--phase-steps", type=int, default=200,
                    help="calls timed with events around the stream kernel alone")
    ap.add_argument("--requests", type=int, default=None,
                    help="verify only the first N requests of the workload (small cases for ncu captures)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes (read+write) per launch of the verify kernel, if captured")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scheme", default="accept", choices=["accept", "onehot", "lazy"],
                    help="accept: spec_verify (accept test against q); onehot: spec_verify_onehot; "
                         "lazy: spec_verify_lazy (no row after a request's first rejection is read)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
