#!/usr/bin/env python3
"""Benchmark of the verification pass: verified draft positions per second.

One step = one full pass of the hot path over one batch resident in HBM:
spec_verify (stochastic rule, residual/bonus draw, logit(q_max) features and
estimator confidences) followed by spec_estimator_update (one online step of
the acceptance estimator) -- the large-batch estimator workload,
B=256 sequences, K=8 draft positions, V=128256, bf16 logits, unless
--workload says otherwise.

Prints one JSON line (rank 0). With --impl reference the fp64 CPU oracle is
timed instead, on the host cores, each step a bounded sample of the workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  torchrun --nproc-per-node N bench.py --gpus N ...   (N independent replicas)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and achieved HBM GB/s vs ~8 TB/s peak (1 GB300)"
UNIT = "positions/s"
KERNEL_SOURCES = ("speculative_decoding_token_verify_gb300/csrc/spec_verify.cu",
                  "speculative_decoding_token_verify_gb300/csrc/spec_device.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "verify_kernel_traffic.txt")
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (~8 TB/s)
L2_BYTES = 129e6

# the other configurations of the verification pass, timed alone in the
# default run (spec_verify only, inputs resident): (workload name, mode)
CONFIG_POINTS = (
    ("tiny_B4_K4_V1024_f32", "stochastic"),
    ("tiny_B4_K4_V1024_f32", "greedy"),
    ("llama3vocab_B64_K5_V128256_bf16", "stochastic"),
    ("fly_B128_K15_V152064_bf16", "fly"),
    ("sweep_B32_K4_V32000_bf16", "stochastic"),
    ("sweep_B32_K8_V128256_bf16", "stochastic"),
    ("sweep_B128_K8_V128256_bf16", "stochastic"),
    ("sweep_B512_K8_V152064_bf16", "stochastic"),
    ("sweep_B128_K4_V152064_f32", "stochastic"),
    ("sweep_B1024_K8_V152064_f32", "stochastic"),
)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="estimator_B256_K8_V128256_bf16")
    ap.add_argument("--B", type=int, default=0, help="override the workload's batch size")
    ap.add_argument("--seed", type=int, default=1003)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--ngram", action="store_true",
                    help="also time prompt-lookup drafting (spec_ngram_draft) for this workload's B and K")
    ap.add_argument("--av", action="store_true",
                    help="also time adaptive-verification pruning (spec_av_budget) and the pruned verify")
    ap.add_argument("--temperature", action="store_true",
                    help="also time temperature-processed verification (spec_verify_temperature) on this "
                         "workload, inverse temperatures log-uniform on [0.5, 2]")
    ap.add_argument("--top-p", type=float, default=None, dest="top_p",
                    help="also time top-p (nucleus) processed verification (spec_verify_top_p) at this top_p "
                         "on this workload, inverse temperatures log-uniform on [0.5, 2]")
    ap.add_argument("--irls", action="store_true",
                    help="also time the IRLS refit entry points (spec_irls_*) on this workload's B, K")
    ap.add_argument("--confidence", action="store_true",
                    help="also time the draft-only confidence pass (spec_confidence) on this workload's draft rows")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration timings (C1, C2, C4 and six sweep points)")
    ap.add_argument("--sweep", action="store_true",
                    help="time spec_verify alone at every point of the throughput sweep (B x K x V x dtype, "
                         "stochastic) and print one JSON line per point instead of the step line")
    return ap.parse_args()


def get_workload(args):
    import workloads

    if args.workload in workloads.WORKLOADS:
        w = workloads.WORKLOADS[args.workload]
    else:
        sweep = {w.name: w for w in workloads.sweep()}
        if args.workload not in sweep:
            raise SystemExit(f"unknown workload {args.workload}")
        w = sweep[args.workload]
    if args.B:
        w = w.scaled(B=args.B, name=f"{w.name}@B{args.B}")
    return w


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ---------------------------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        # NCCL on GPU ranks; SPEC_DIST_BACKEND=gloo runs the same host logic
        # on CPU ranks (the tests do)
        backend = os.environ.get("SPEC_DIST_BACKEND", "nccl")
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def replica_throughput(world: int, steps: int, B: int, K: int, max_ms: float) -> float:
    """Whole-job verified positions/s of N replicas: every rank verifies its
    own B x K positions per step, and the slowest rank's time counts."""
    return world * steps * B * K / (max_ms / 1e3)


def max_over_ranks(pg, v: float, device=None) -> float:
    if pg is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled=True):
        self.proc = None
        self.gpu = gpu_index
        self.enabled = enabled

    def start(self):
        if not self.enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 reasons=dict(hw_slowdown=f[5], hw_thermal_slowdown=f[6],
                                              sw_thermal_slowdown=f[7], sw_power_cap=f[8])))
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r["power"] > 0.5 * max(r["power"] for r in rows)] or rows
        reasons = sorted({k for r in load for k, v in r["reasons"].items() if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_inputs(w, n_seq, seed):
    """A bounded sample: the first n_seq sequences of the workload, drawn on
    the CPU with the workload's recipe."""
    import workloads

    sub = w.scaled(B=n_seq)
    inp = workloads.make_inputs(sub, seed, "cpu")
    return dict(zt=workloads.to_numpy_logits(inp["zt"]), zd=workloads.to_numpy_logits(inp["zd"]),
                x=inp["x"].numpy(), u=inp["u"].numpy())


def oracle_step(w, s, nthreads):
    import numpy as np

    import oracle

    mode = {"stochastic": oracle.STOCHASTIC, "greedy": oracle.GREEDY, "fly": oracle.FLY}[w.mode]
    est = np.r_[1.0, np.zeros(w.K)] if w.with_confidence else None
    zd = s["zd"] if (w.mode == "stochastic" or w.with_confidence) else None
    r = oracle.verify(s["zt"], zd, s["x"], s["u"] if w.mode == "stochastic" else None, mode=mode,
                      fly_theta=w.fly_theta, fly_window=w.fly_window, est_params=est,
                      nthreads=nthreads)
    if w.with_confidence:
        oracle.estimator_update(r["feature"], r["accepted_len"], est, w.estimator_lr)
    return r


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, seed, target_s=1.0):
    """Time the oracle as it stands on all host cores over a bounded sample
    (about target_s seconds of wall time, i.e. cores * target_s of CPU work)."""
    import oracle

    oracle.build()
    cores = host_cores()
    probe = oracle_sample_inputs(w, 1, seed)
    t0 = time.perf_counter()
    oracle_step(w, probe, 1)
    t_seq = time.perf_counter() - t0
    n_seq = max(cores, int(round(target_s / max(t_seq, 1e-6))) * cores)
    n_seq = min(n_seq, w.B, 16 * cores)
    s = oracle_sample_inputs(w, n_seq, seed)
    t0 = time.perf_counter()
    oracle_step(w, s, cores)
    dt = time.perf_counter() - t0
    return {"value": n_seq * w.K / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {n_seq} of {w.B} sequences of {w.name} (fp64 C oracle, OpenMP over "
                      f"sequences, {cores} threads, {dt:.2f} s wall)"}


def step_config(w, world):
    """The `config` object of the step line, shared by both arms."""
    logit_bytes = w.logit_bytes(w.mode == "stochastic" or w.with_confidence)
    l2_note = ("inputs larger than L2 (%.2f GB of logits per step, L2 129 MB)" % (logit_bytes / 1e9)
               if logit_bytes > 2 * L2_BYTES else "L2 flushed between steps")
    return {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "logits": w.dtype,
            "mode": w.mode + ("+confidence+estimator_update" if w.with_confidence else ""),
            "l2": l2_note, "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, w, world, rank, pg):
    import oracle

    if rank != 0:
        return 0
    oracle.build()
    cores = host_cores()
    n_seq = min(w.B, cores)
    s = oracle_sample_inputs(w, n_seq, args.seed)
    for _ in range(args.warmup):
        oracle_step(w, s, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, s, cores)
    dt = time.perf_counter() - t0
    value = args.steps * n_seq * w.K / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": step_config(w, world),
        "sample": f"each step: the oracle's full step (verification, confidences, estimator update) on "
                  f"the first {n_seq} of {w.B} sequences of {w.name}",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: first {n_seq} of {w.B} sequences of {w.name}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def source_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def verify_kernel_name(w):
    """The verify kernel instance a default launch of this workload runs:
    verify_kernel<T, kTemp = 0, kRing>, the staging-buffer ring (kRing = 1)
    in the modes with no draw."""
    t = "__nv_bfloat16" if w.dtype == "bf16" else "float"
    return f"verify_kernel<{t}, 0, {0 if w.mode == 'stochastic' else 1}>"


def recorded_traffic(workload_name):
    """Per-launch DRAM bytes of the verify kernel on this workload from the
    committed ncu summary, if it was taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            kv = dict(line.strip().split("=", 1) for line in f if "=" in line and not line.startswith("#"))
    except OSError:
        return None
    if kv.get("source_sha256") != source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch." + workload_name])
    except (KeyError, ValueError):
        return None


def measured_hbm_peak():
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(mp["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback (6.8 TB/s, earlier GB300 measurement)"


def run_ours(args, w, world, rank, local, pg):
    import torch

    import speculative_decoding_token_verify_gb300 as sv
    import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    inp = workloads.make_inputs(w, args.seed + 7919 * rank, dev)
    with_draft = w.mode == "stochastic" or w.with_confidence
    zd = inp["zd"] if with_draft else None
    u = inp["u"] if w.mode == "stochastic" else None
    est0 = torch.tensor([1.0] + [0.0] * w.K, dtype=torch.float32, device=dev)
    est = est0.clone()
    ws = sv.Workspace(dev)
    out = {"out_tokens": torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev),
           "accepted_len": torch.empty((w.B,), dtype=torch.int32, device=dev)}
    if w.with_confidence:
        out["feature"] = torch.empty((w.B, w.K), dtype=torch.float32, device=dev)
        out["conf"] = torch.empty((w.B, w.K), dtype=torch.float32, device=dev)

    nvtx = torch.cuda.nvtx

    def step(zt_, zd_, x_, u_):
        nvtx.range_push("spec_verify")
        sv.verify(zt_, zd_, x_, u_, mode=w.mode, fly_theta=w.fly_theta, fly_window=w.fly_window,
                  est_params=est if w.with_confidence else None, out=out, workspace=ws,
                  want_feature=w.with_confidence, want_conf=w.with_confidence)
        nvtx.range_pop()
        if w.with_confidence:
            nvtx.range_push("spec_estimator_update")
            sv.estimator_update(out["feature"], out["accepted_len"], est, w.estimator_lr)
            nvtx.range_pop()

    launches_per_step = 2 if w.with_confidence else 1
    for _ in range(args.warmup):
        step(inp["zt"], zd, inp["x"], u)
    torch.cuda.synchronize(dev)

    logit_bytes = w.logit_bytes(with_draft)
    flush = None
    if logit_bytes <= 2 * L2_BYTES:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    clocks = ClockSampler(local, enabled=(rank == 0 and not args.no_clocks))
    clocks.start()
    ev_v = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    if flush is None:
        t_start.record(stream)
        for i in range(args.steps):
            ev_v[i][0].record(stream)
            step(inp["zt"], zd, inp["x"], u)
            ev_v[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = t_start.elapsed_time(t_end)
    else:
        total_ms = 0.0
        for i in range(args.steps):
            flush.add_(1)
            ev_v[i][0].record(stream)
            step(inp["zt"], zd, inp["x"], u)
            ev_v[i][1].record(stream)
        torch.cuda.synchronize(dev)
        total_ms = sum(a.elapsed_time(b) for a, b in ev_v)
    barrier(pg, dev)
    step_ms = [a.elapsed_time(b) for a, b in ev_v]
    total_ms = max_over_ranks(pg, total_ms, dev)

    # the dominant kernel alone: spec_verify's launches, same stream, same region
    verify_ms = []
    if w.with_confidence:
        ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(min(args.steps, 200))]
        for a, b in ev_k:
            a.record(stream)
            sv.verify(inp["zt"], zd, inp["x"], u, mode=w.mode, est_params=est, out=out, workspace=ws,
                      want_feature=True, want_conf=True)
            b.record(stream)
        torch.cuda.synchronize(dev)
        verify_ms = [a.elapsed_time(b) for a, b in ev_k]
    else:
        verify_ms = step_ms

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, inp, zd, u, est0, out, ws, dev, stream, step, pg)
    clk = clocks.stop()

    value = replica_throughput(world, args.steps, w.B, w.K, total_ms)
    kern_s = statistics.mean(verify_ms) / 1e3
    peak, peak_src = measured_hbm_peak()
    achieved = logit_bytes / kern_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": step_config(w, world),
        "hbm_gbs": logit_bytes * world * args.steps / (total_ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS, "traffic": recorded_traffic(w.name),
                     "kernel": verify_kernel_name(w),
                     "algorithmic_bytes_per_launch": logit_bytes,
                     "kernel_ms_mean": kern_s * 1e3, "kernel_ms_median": statistics.median(verify_ms),
                     "peak_source": peak_src, "frac_note": "of measured" if "measured" in peak_src
                     else "of fallback"},
        "gpu_launches": args.steps * launches_per_step,
        "e2e": e2e,
        "clocks": clk,
    }
    if args.irls and w.with_confidence:
        line["irls"] = time_irls(w, out, est, dev, stream)
    if args.ngram:
        line["ngram"] = time_ngram(w, dev, stream, args.seed)
    if args.av and w.with_confidence and w.mode == "stochastic":
        line["av"] = time_av(w, inp, zd, u, out, est, ws, dev, stream, peak)
    if args.temperature:
        line["temperature"] = time_temperature(w, args.seed, out, est, ws, dev, stream, peak, logit_bytes,
                                               kern_s * 1e3)
    if args.top_p is not None:
        line["top_p"] = time_temperature(w, args.seed, out, est, ws, dev, stream, peak, logit_bytes,
                                         kern_s * 1e3, top_p=args.top_p)
    if args.confidence and zd is not None:
        line["confidence"] = time_confidence(w, zd, est, dev, stream, peak)
    if not args.no_configs and world == 1:
        del inp
        torch.cuda.empty_cache()
        line["configs"] = time_configs(dev, stream, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.seed)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def device_us(fn, stream, reps):
    """Mean device time of fn() in microseconds over `reps` back-to-back
    calls. A short sleep kernel holds the stream while the host enqueues
    them, so the events bracket device work, not host issue gaps (these are
    launch-sized kernels)."""
    import torch

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(20_000_000)          # ~10 ms of device time, bounded
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps


def time_irls(w, out, est, dev, stream, round_steps=64, damping=16.0, reps=20):
    """Device time of the IRLS refit's two calls on this workload's features
    and labels: one spec_irls_accumulate per decoding step, one
    spec_irls_refit per round of `round_steps` steps (both CUDA events on the
    launching stream, after warm-up)."""
    import torch

    import speculative_decoding_token_verify_gb300 as sv

    st = sv.IrlsState(w.K, dev)
    params = est.clone()
    for _ in range(3):
        sv.irls_accumulate(out["feature"], out["accepted_len"], params, st)
        sv.irls_refit(st, params, damping)
    acc_us = device_us(lambda: sv.irls_accumulate(out["feature"], out["accepted_len"], params, st), stream,
                       round_steps)
    ref_us = device_us(lambda: sv.irls_refit(st, params, damping), stream, reps)
    return {"accumulate_us_per_step": acc_us, "refit_us_per_round": ref_us, "round_steps": round_steps,
            "damping": damping, "B": w.B, "K": w.K,
            "note": "launch-bound O(B*K) work; one CTA each"}


def time_ngram(w, dev, stream, seed, ld=4096, reps=50):
    """Device time of prompt-lookup drafting for this workload's B sequences
    of `ld` context tokens (synthetic: uniform tokens with a planted repeat
    of 4..40 tokens in every other sequence), n in [1, 4], K drafts."""
    import numpy as np
    import torch

    import speculative_decoding_token_verify_gb300 as sv

    rng = np.random.default_rng(seed + 17)
    ctx = rng.integers(0, w.V, (w.B, ld)).astype(np.int32)
    for b in range(0, w.B, 2):
        n = int(rng.integers(4, 41))
        a = int(rng.integers(0, ld // 2))
        ctx[b, ld - n:] = ctx[b, a:a + n]
    c = torch.tensor(ctx, device=dev)
    ln = torch.full((w.B,), ld, dtype=torch.int32, device=dev)
    d = sv.ngram_draft(c, ln, 1, 4, w.K)
    us = device_us(lambda: sv.ngram_draft(c, ln, 1, 4, w.K), stream, reps)
    return {"us": us, "B": w.B, "context": ld, "n": [1, 4], "K": w.K,
            "mean_draft_len": float(d["draft_len"].float().mean().item())}


def time_av(w, inp, zd, u, out, est, ws, dev, stream, peak, reps=50):
    """Device time of one adaptive-verification step's two calls: the budget
    (spec_av_budget on this step's confidences, with a synthetic cost table
    that grows by a third of a base step per B verified drafts) and the
    pruned verify it selects (spec_verify_ragged). The pruned verify reads
    only the rows it verifies: sum_b (2 K_b + 1) V s bytes."""
    import torch

    import speculative_decoding_token_verify_gb300 as sv

    N = w.B * w.K
    k = torch.arange(N + 1, dtype=torch.float32, device=dev)
    dcost = 0.01 * k / w.B
    vcost = 1.0 + 0.05 * k / w.B
    # confidences from a calibrated estimator (slope 0.5, intercepts 1.5, in
    # the range the pages report for fitted pairs) on this step's draft rows
    est_av = torch.tensor([0.5] + [1.5] * w.K, dtype=torch.float32, device=dev)
    _, conf = sv.confidence(zd, est_av)
    bud = sv.av_budget(conf, dcost, vcost)
    for _ in range(3):
        sv.av_budget(conf, dcost, vcost, stream=None)
        sv.verify(inp["zt"], zd, inp["x"], u, mode=w.mode, est_params=est, out=dict(out), workspace=ws,
                  want_feature=True, want_conf=True, draft_len=bud["draft_len"])
    budget_us = device_us(lambda: sv.av_budget(conf, dcost, vcost), stream, reps)
    o2 = dict(out)
    v_ms = device_us(lambda: sv.verify(inp["zt"], zd, inp["x"], u, mode=w.mode, est_params=est, out=o2,
                                       workspace=ws, want_feature=True, want_conf=True,
                                       draft_len=bud["draft_len"]), stream, reps) / 1e3
    dl = bud["draft_len"].cpu()
    es = 2 if w.dtype == "bf16" else 4
    pruned_bytes = int(((2 * dl.long() + 1) * w.V * es).sum())
    return {"budget": int(bud["budget"].item()), "drafts": N, "mean_draft_len": float(dl.float().mean()),
            "budget_us": budget_us,
            "pruned_verify_ms": v_ms, "pruned_bytes": pruned_bytes,
            "pruned_frac": pruned_bytes / (v_ms / 1e3) / 1e9 / peak,
            "cost_table": "draft 0.01 k/B, verify 1 + 0.05 k/B (synthetic)", "est": "omega 0.5, beta 1.5"}


def time_temperature(w, seed, out, est, ws, dev, stream, peak, logit_bytes, default_ms, reps=100, top_p=None):
    """Device time of one verification at per-sequence inverse temperatures
    (log-uniform on [0.5, 2]; drafts drawn from the temperature-processed q)
    and, with top_p, at that top-p (spec_verify_top_p: the nucleus pass and
    the verification launch), CUDA events on the launching stream over `reps`
    back-to-back calls; the inputs (same shapes and logits as the main line)
    are larger than L2."""
    import statistics as st

    import torch

    import speculative_decoding_token_verify_gb300 as sv
    import workloads

    wt = w.scaled(inv_temp_range=(0.5, 2.0))
    inp = workloads.make_inputs(wt, seed, dev)
    with_draft = w.mode == "stochastic" or w.with_confidence
    zd = inp["zd"] if with_draft else None
    u = inp["u"] if w.mode == "stochastic" else None
    o = dict(out)

    def call():
        sv.verify(inp["zt"], zd, inp["x"], u, mode=w.mode, fly_theta=w.fly_theta, fly_window=w.fly_window,
                  est_params=est if w.with_confidence else None, out=o, workspace=ws,
                  want_feature=w.with_confidence, want_conf=w.with_confidence, inv_temperature=inp["inv_temp"],
                  top_p=top_p)

    for _ in range(5):
        call()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = st.mean(ms)
    del inp
    res = {"verify_ms_mean": mean_ms, "verify_ms_median": st.median(ms),
           "frac": logit_bytes / (mean_ms / 1e3) / 1e9 / peak, "default_verify_ms_mean": default_ms,
           "inv_temperature": "log-uniform [0.5, 2] per sequence",
           "kernel": "verify_kernel<T, 1, 0> (temperature variant)"}
    if top_p is not None:
        res["top_p"] = top_p
        res["kernel"] = "nucleus_row_kernel<T> + verify_kernel<T, 2, 0> (precomputed rows)"
    return res


def time_confidence(w, zd, est, dev, stream, peak, reps=100):
    """Device time of spec_confidence (logit(q_max) features and
    confidences from the draft rows alone: B*K*V elements read once), CUDA
    events on the launching stream over back-to-back calls; the draft logits
    are larger than L2."""
    import statistics as st

    import torch

    import speculative_decoding_token_verify_gb300 as sv

    cws = sv.Workspace(dev)
    for _ in range(5):
        sv.confidence(zd, est, workspace=cws)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record(stream)
        sv.confidence(zd, est, workspace=cws)
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms = [a.elapsed_time(b) for a, b in ev]
    nbytes = zd.numel() * zd.element_size()
    mean_ms = st.mean(ms)
    return {"ms_mean": mean_ms, "ms_median": st.median(ms), "algorithmic_bytes": nbytes,
            "frac": nbytes / (mean_ms / 1e3) / 1e9 / peak, "kernel": "verify_kernel<T, 0, 1> (draft rows only, staging-buffer ring)"}


def time_configs(dev, stream, peak, reps=50):
    """spec_verify alone on each configuration of CONFIG_POINTS, inputs
    resident in HBM, CUDA events around each call on the launching stream
    (an L2 flush before each call where the logits are under twice the L2
    size). The tiny workload is launch-bound: its calls are timed back to back
    with the stream held while the host enqueues them (device time per
    call). Each entry: kernel time, GB/s, positions/s and the fractions of the
    measured and the nominal HBM bandwidth."""
    import torch

    import speculative_decoding_token_verify_gb300 as sv
    import workloads

    sweep = {w.name: w for w in workloads.sweep()}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = {}
    for k, (name, mode) in enumerate(CONFIG_POINTS):
        w = workloads.WORKLOADS.get(name) or sweep[name]
        inp = workloads.make_inputs(w, 1000 + k, dev)
        with_draft = mode == "stochastic"
        zd = inp["zd"] if with_draft else None
        u = inp["u"] if mode == "stochastic" else None
        ws = sv.Workspace(dev)
        out = {"out_tokens": torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev),
               "accepted_len": torch.empty((w.B,), dtype=torch.int32, device=dev)}
        nbytes = w.logit_bytes(with_draft)

        def call():
            sv.verify(inp["zt"], zd, inp["x"], u, mode=mode, fly_theta=w.fly_theta, fly_window=w.fly_window,
                      out=out, workspace=ws)

        for _ in range(5):
            call()
        torch.cuda.synchronize(dev)
        if nbytes < 4 << 20:
            us = device_us(call, stream, 200)
            ms = [us / 1e3]
            timing = "launch-bound: 200 back-to-back calls, device time per call"
        else:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            small = nbytes <= 2 * L2_BYTES
            for a, b in ev:
                if small:
                    flush.add_(1)
                a.record(stream)
                call()
                b.record(stream)
            torch.cuda.synchronize(dev)
            ms = [a.elapsed_time(b) for a, b in ev]
            timing = ("L2 flushed before each call" if small else "inputs larger than L2") + f", {reps} calls"
        mean_s = statistics.mean(ms) / 1e3
        gbs = nbytes / mean_s / 1e9
        t = "__nv_bfloat16" if w.dtype == "bf16" else "float"
        res[f"{name}:{mode}"] = {
            "B": w.B, "K": w.K, "V": w.V, "logits": w.dtype, "mode": mode,
            "rows": "target + draft" if with_draft else "target only",
            "kernel_ms_mean": mean_s * 1e3, "kernel_ms_median": statistics.median(ms),
            "positions_per_s": w.B * w.K / mean_s, "hbm_gbs": gbs, "algorithmic_bytes": nbytes,
            "frac": gbs / peak, "frac_nominal": gbs / NOMINAL_HBM_GBS,
            "kernel": f"verify_kernel<{t}, 0, {0 if mode == 'stochastic' else 1}>", "timing": timing,
            "status": sv.device_status(ws.buf)}
        del inp, zd, u, ws, out
        torch.cuda.empty_cache()
    return res


def run_sweep(args):
    """spec_verify alone at every sweep point, inputs resident in HBM: CUDA
    events around each call on the launching stream; an L2 flush (a write of
    256 MB) before each call where the logits are under twice the L2 size."""
    import torch

    import speculative_decoding_token_verify_gb300 as sv
    import workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_src = measured_hbm_peak()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(0, enabled=not args.no_clocks)
    clocks.start()
    lines = []
    for k, w in enumerate(workloads.sweep()):
        inp = workloads.make_inputs(w, 2000 + k, dev)
        ws = sv.Workspace(dev)
        out = {"out_tokens": torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev),
               "accepted_len": torch.empty((w.B,), dtype=torch.int32, device=dev)}
        logit_bytes = w.logit_bytes(True)
        small = logit_bytes <= 2 * 129e6

        def call():
            sv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], mode="stochastic", out=out, workspace=ws)

        for _ in range(max(args.warmup, 3)):
            call()
        reps = max(10, min(args.steps, 100))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            if small:
                flush.add_(1)
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = [a.elapsed_time(b) for a, b in ev]
        mean_s = statistics.mean(ms) / 1e3
        line = {"metric": METRIC, "workload": w.name, "B": w.B, "K": w.K, "V": w.V, "logits": w.dtype,
                "ms_mean": mean_s * 1e3, "ms_median": statistics.median(ms),
                "positions_per_s": w.B * w.K / mean_s, "hbm_gbs": logit_bytes / mean_s / 1e9,
                "frac": logit_bytes / mean_s / 1e9 / peak, "peak": peak,
                "algorithmic_bytes": logit_bytes,
                "l2": "flushed before each call" if small else "inputs larger than L2",
                "status": sv.device_status(ws.buf)}
        print(json.dumps(line), flush=True)
        lines.append(line)
        del inp, ws, out
        torch.cuda.empty_cache()
    clk = clocks.stop()
    print(json.dumps({"sweep_points": len(lines), "clocks": clk, "peak_source": peak_src}), flush=True)
    return 0


def run_e2e(args, w, inp, zd, u, est0, out, ws, dev, stream, step, pg):
    """Same metric through the public API with HOST inputs: every step copies
    its inputs from pinned host memory and reads its results back. The copy
    of step i+1's inputs (a copy stream, into the other of two device input
    sets) overlaps step i's verification and read-back (the launching
    stream); the host link, not the kernels, bounds this number."""
    import torch

    h_zt = inp["zt"].cpu().pin_memory()
    h_zd = zd.cpu().pin_memory() if zd is not None else None
    h_x = inp["x"].cpu().pin_memory()
    h_u = u.cpu().pin_memory() if u is not None else None
    sets = []
    for _ in range(2):
        sets.append((torch.empty_like(inp["zt"]), torch.empty_like(zd) if zd is not None else None,
                     torch.empty_like(inp["x"]), torch.empty_like(u) if u is not None else None))
    res = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()}
    h2d = sum(t.numel() * t.element_size() for t in (h_zt, h_zd, h_x, h_u) if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in res.values())
    steps = max(3, min(args.steps, 50))
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]
    for e in used:
        e.record(stream)

    def issue_copy(slot):
        d_zt, d_zd, d_x, d_u = sets[slot]
        copy_stream.wait_event(used[slot])      # the set's previous step is done with it
        with torch.cuda.stream(copy_stream):
            d_zt.copy_(h_zt, non_blocking=True)
            if d_zd is not None:
                d_zd.copy_(h_zd, non_blocking=True)
            d_x.copy_(h_x, non_blocking=True)
            if d_u is not None:
                d_u.copy_(h_u, non_blocking=True)
        copied[slot].record(copy_stream)

    def issue_compute(slot):
        stream.wait_event(copied[slot])
        step(*sets[slot])
        for k, t in res.items():
            t.copy_(out[k], non_blocking=True)
        used[slot].record(stream)

    def run(n):
        issue_copy(0)
        for i in range(n):
            if i + 1 < n:
                issue_copy((i + 1) % 2)
            issue_compute(i % 2)

    run(2)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    barrier(pg, dev)
    a.record(stream)
    copy_stream.wait_event(a)
    run(steps)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(pg, a.elapsed_time(b), dev)
    world = pg.get_world_size() if pg is not None else 1
    return {"value": replica_throughput(world, steps, w.B, w.K, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
            "overlap": "step i+1's host-to-device copy overlaps step i's kernels and read-back"}


def main():
    args = parse_args()
    if args.sweep:
        return run_sweep(args)
    w = get_workload(args)
    world, rank, local, pg = dist_setup(args)
    if world != args.gpus and rank == 0:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            return run_reference(args, w, world, rank, pg)
        return run_ours(args, w, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
