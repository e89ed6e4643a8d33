#!/usr/bin/env python3
"""Benchmark of the GB300 fused attention forward (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one fa_fwd call over the whole workload (inputs resident in HBM).
Metric: useful TFLOPS = 4*B*H*S^2*D / t, halved under the causal mask.  The
default workload is the training-size causal one (4 x 32 x 4096 x 128, bf16).
Under torchrun every rank runs its own replica of the workload (replicas only:
the path needs no exchange between GPUs); `value` is the FLOPs of all ranks
divided by the slowest rank's time.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on
bounded samples of the same workload, and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fa_inputs import WORKLOADS, make_workload  # noqa: E402

METRIC = "attention fwd TFLOPS (causal/non-causal) at 1 GB300; fraction of tensor peak"
UNIT = "TFLOPS"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash() -> str:
    """sha256 over the kernel and launcher sources (csrc/): identifies the build
    whose counters a profile summary holds.  The public header's comments do
    not change the kernel, so they do not void a summary."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "attention_fa_fwd_gb300", "csrc", "*")))
    for fn in files:
        h.update(os.path.basename(fn).encode())
        with open(fn, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu figures of this workload
    (profiles/fa_fwd_kernel_<workload>.traffic.json), or None when there are
    none or they were taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", f"fa_fwd_kernel_{workload}.traffic.json")
    try:
        with open(path, encoding="utf-8") as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != source_hash():
        return None
    try:
        return int(rec["traffic_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi samples (200 ms) of one GPU while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        return self.summary()

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        loaded = [r for r in self.rows if (num(r[8]) or 0) > 0] or self.rows
        if not loaded:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [num(r[0]) for r in loaded if num(r[0]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in loaded for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        power = [num(r[2]) for r in loaded if num(r[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(loaded[0][1]), "reasons": reasons,
                "power_w_max": max(power) if power else None, "samples": len(loaded)}


def oracle_rows_sample(w, q, k, v, n_rows, seed):
    """(heads, rows, useful FLOPs) of a sample of rows of the workload."""
    import numpy as np
    rng = np.random.default_rng(seed)
    BH, S = w.B * w.H, w.S
    heads = rng.integers(0, BH, n_rows)
    rows = rng.integers(0, S, n_rows)
    keys = (rows + 1) if w.causal else np.full(n_rows, S)
    flops = float(4.0 * w.D * keys.sum())     # QK^T and PV over the keys each row sees
    return heads, rows, flops


def time_oracle(w, q, k, v, budget_s: float, steps: int, seed: int = 0):
    """Run the fp64 oracle (row-by-row definition) on `steps` bounded samples;
    returns (TFLOPS, seconds per step, sample description, threads)."""
    import numpy as np
    import oracle
    from fa_inputs import to_f64
    nthreads = os.cpu_count() or 1
    # the oracle reads a few heads only: gather them once (exact fp64 widening)
    BH, S, D = w.B * w.H, w.S, w.D
    qf, kf, vf = (x.reshape(BH, S, D) for x in (q, k, v))
    # calibrate rows per step so one step takes about budget_s seconds
    n_rows = max(nthreads, 8)
    per_step = []
    tflops = []
    desc = None
    for step in range(steps + 1):
        heads, rows, flops = oracle_rows_sample(w, q, k, v, n_rows, seed + step)
        uh, inv = np.unique(heads, return_inverse=True)
        sel = torch.from_numpy(uh)
        sub = lambda x: to_f64(x[sel].unsqueeze(0))
        qs, ks, vs = sub(qf), sub(kf), sub(vf)
        t0 = time.perf_counter()
        oracle.attention_rows(qs, ks, vs, w.causal, w.scale, inv, rows, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if step == 0:
            # calibration step: resize the sample to the budget, not timed
            n_rows = max(nthreads, int(n_rows * budget_s / max(dt, 1e-3)))
            continue
        per_step.append(dt)
        tflops.append(flops / dt / 1e12)
        desc = (f"{n_rows} random (head, row) pairs of the {w.name} workload per step, "
                f"fp64 row-by-row definition, {nthreads} OpenMP threads")
    return statistics.median(tflops), statistics.median(per_step), desc, nthreads


def rescale_events(w, q, k, v, heads: int = 1, fa=None):
    """Re-bases of the lazy rescale: the kernel's own counts over the whole
    workload (its debug-statistics build, one extra pass), and the oracle's
    lazy-rescale recurrence (row level, P rounded to fp16, no overshoot) on the
    first `heads` heads at the pages' threshold 8 and the kernel's T."""
    import oracle
    from fa_inputs import to_f64
    BH, S, D = w.B * w.H, w.S, w.D
    kernel = None
    T = 15.0
    if fa is not None:
        _, _, _, counts, (T, over) = fa.debug_stats(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
        kernel = {"heads": BH, "warp_rescales": counts[0], "row_rebases": counts[1],
                  "rule": {"T": T, "overshoot": over}}
    qs, ks, vs = (to_f64(x.reshape(BH, S, D)[:heads].unsqueeze(0)) for x in (q, k, v))
    out = {}

    def run(t):
        out[t] = oracle.attention_lazy(qs, ks, vs, w.causal, w.scale, 128, t, "fp16", nthreads=heads)[2]

    ts = [8.0, T]
    th = [threading.Thread(target=run, args=(t,)) for t in ts]
    for t in th:
        t.start()
    for t in th:
        t.join()
    steps = out[ts[0]]["steps"]
    return {"kernel": kernel,
            "model": {"what": "oracle lazy-rescale recurrence, row level, no overshoot", "heads": heads,
                      "row_tile_steps": steps, "row_rebases": {f"T={t:g}": out[t]["rebases"] for t in ts}}}


def aggregate(ms_local: float, flops_per_rank: float, world: int, dist=None, device=None):
    """Max of the ranks' timed milliseconds and the whole-job TFLOPS over it
    (every rank ran `flops_per_rank`).  `dist` is torch.distributed or None."""
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if dist is not None and world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, flops_per_rank * world / (ms_max * 1e-3) / 1e12


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v = make_workload(w)
    budget = max(0.05, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    value, sec, desc, cores = time_oracle(w, q, k, v, budget, args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                   "causal": w.causal, "input_dtype": w.dtype},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Every workload of the target list, timed on the device in the same run.  The
# short ones are launch-bound, so each is timed for a fixed wall time instead of
# a fixed count; C1 runs both masks.
PER_CONFIG = [("C1", "tiny"), ("C1", "tiny_causal"), ("C2", "batch1_causal"), ("C3", "wide_noncausal"),
              ("C4", "train_causal"), ("C5", "stress_causal")]


def time_device_loop(step, stream, dev, steps):
    """Milliseconds per step over `steps` back-to-back steps (CUDA events on the
    launching stream, the device synchronised on both sides)."""
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps


L2_BYTES = 129 * 1000 * 1000   # GB300 L2


def time_flushed_steps(step, flush, stream, dev, steps):
    """Milliseconds per step with L2 flushed before every step: each step is
    bracketed by its own pair of CUDA events on the launching stream, the
    flush (a write of twice the L2's size) runs outside the pair."""
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for a, b in pairs:
        flush()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return statistics.fmean(a.elapsed_time(b) for a, b in pairs)


def per_config_lines(fa, dev, local, stream, peak_burst, peak_sustained, target_s):
    """Device time, TFLOPS and fraction of peak of every workload, each timed
    for about `target_s` seconds after a warm-up, with its own clock samples.
    Workloads whose tensors exceed the L2 run back to back; the others get an
    L2 flush before every step (their back-to-back time, inputs resident in
    L2, is reported beside it)."""
    out = {}
    flush_buf = None
    for tag, name in PER_CONFIG:
        w = WORKLOADS[name]
        q, k, v = make_workload(w)
        qd, kd, vd = (x.to(dev) for x in (q, k, v))
        od = torch.empty_like(qd)
        ld = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)

        def step():
            fa.fa_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=od, lse=ld, stream=stream)

        for _ in range(5):
            step()
        probe = time_device_loop(step, stream, dev, 10)
        resident = w.io_bytes() < L2_BYTES
        warm = None
        if resident:
            if flush_buf is None:
                flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
            flush = lambda: flush_buf.fill_(1)
            warm = time_device_loop(step, stream, dev, int(min(20000, max(20, 0.1e3 / max(probe, 1e-3)))))
            per_iter = time_flushed_steps(step, flush, stream, dev, 5) + 0.08   # + ~80 us of flush
            steps = int(min(5000, max(20, target_s * 1e3 / per_iter)))
        else:
            steps = int(min(200000, max(20, target_s * 1e3 / max(probe, 1e-3))))
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.25)
        if resident:
            ms = time_flushed_steps(step, flush, stream, dev, steps)
        else:
            ms = time_device_loop(step, stream, dev, steps)
        clocks = sampler.stop()
        status, site = fa.device_status(clear=True, stream=stream)
        if status != fa.FA_OK:
            raise SystemExit(f"{name}: in-kernel wait gave up at site {site:#x}")
        tflops = w.flops() / (ms * 1e-3) / 1e12
        out[name] = {"config": tag, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "causal": w.causal,
                     "dtype": w.dtype, "kind": w.kind, "steps": steps, "ms_per_step": round(ms, 6),
                     "tflops": round(tflops, 3), "frac_burst": round(tflops / peak_burst, 4),
                     "frac_sustained": round(tflops / peak_sustained, 4),
                     "l2": ("L2 flushed before every step (tensors %.1f MB fit in L2)" % (w.io_bytes() / 1e6))
                           if resident else ("tensors %.0f MB exceed the L2; back to back" % (w.io_bytes() / 1e6)),
                     "timed_s": round(ms * steps / 1e3, 3), "clocks": clocks}
        if warm is not None:
            out[name]["ms_per_step_l2_resident"] = round(warm, 6)
            out[name]["tflops_l2_resident"] = round(w.flops() / (warm * 1e-3) / 1e12, 3)
        del qd, kd, vd, od, ld
        torch.cuda.empty_cache()
    del flush_buf
    torch.cuda.empty_cache()
    return out


def e2e_leg(fa, w, q, k, v, qd, kd, vd, od, ld, stream, barrier, world, dist, dev, steps):
    """The metric through fa_fwd_hostio with pinned host buffers: every step
    copies q, k, v in and o, lse out around the pass."""
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(steps, 50))

    def e2e_step():
        fa.fa_fwd_hostio(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, causal=w.causal, scale=w.scale,
                         stream=stream)

    for _ in range(2):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    _, value = aggregate(e0.elapsed_time(e1) / e2e_steps, w.flops(), world, dist, dev)
    h2d = 3 * q.numel() * q.element_size()
    d2h = oh.numel() * oh.element_size() + lh.numel() * lh.element_size()
    return {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def run_ours(args, w):
    import attention_fa_fwd_gb300 as fa
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the kernel has no CPU path)")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    fa.build()
    dev = torch.device("cuda", local)
    q, k, v = make_workload(w, seed=rank)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    od = torch.empty_like(qd)
    ld = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)
    info = fa.launch_info(w.B, w.H, w.S, w.D, w.causal, qd.dtype)

    def step():
        fa.fa_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=od, lse=ld, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    status, site = fa.device_status(clear=True, stream=stream)
    if status != fa.FA_OK:
        raise SystemExit(f"in-kernel wait gave up at site {site:#x}")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    # best single step: a short loop of individually timed launches
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(min(50, args.steps))]
    for a, b in pairs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms_best = min(a.elapsed_time(b) for a, b in pairs)
    status, site = fa.device_status(clear=True, stream=stream)
    if status != fa.FA_OK:
        raise SystemExit(f"in-kernel wait gave up at site {site:#x}")
    flops = w.flops()
    ms_max, value = aggregate(ms, flops * args.steps, world, dist, dev)
    ms_step = ms_max / args.steps

    # end to end through the C ABI with host buffers: H2D of q, k, v, the
    # kernel, D2H of o and lse, every step
    e2e = None
    if not args.no_e2e:
        e2e = e2e_leg(fa, w, q, k, v, qd, kd, vd, od, ld, stream, barrier, world, dist, dev, args.steps)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    pk, pk_kind = peaks()
    burst = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    # a loop timed for half a second or more runs at the power-capped clock:
    # compare it with the sustained GEMM peak, a short burst with the burst peak
    if ms_max >= 500.0:
        peak, peak_kind = sustained, f"bf16 dense sustained ({pk_kind})"
    else:
        peak, peak_kind = burst, f"bf16 dense burst ({pk_kind})"
    traffic = args.traffic if args.traffic is not None else profiled_traffic(w.name)
    achieved = flops / (ms_step * 1e-3) / 1e12   # one launch per step on this stream
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "ms_per_step_best": round(ms_best, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "fp16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "causal": w.causal,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs (Q,K,V,O = %d MiB) exceed the 129 MB L2; no flush" %
                         (4 * q.numel() * q.element_size() >> 20),
                   "grid": info["grid"], "tiles_per_unit": info["tiles_per_unit"],
                   "units": info["units"]},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind, "timed_ms": round(ms_max, 1), "traffic": traffic},
        "e2e": e2e,
        "gpu_launches": args.steps * world,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        budget = 15.0
        cv, _, desc, cores = time_oracle(w, q, k, v, budget, 1)
        line["cpu_baseline"] = {"value": round(cv, 6), "unit": UNIT, "cores": cores,
                                "kind": "oracle", "sample": desc}
    elif not args.no_cpu_baseline:
        line["cpu_baseline"] = None
    if w.kind == "stress" and not args.no_cpu_baseline:
        line["rescale"] = rescale_events(w, q, k, v, fa=fa)
    if not args.no_per_config and world == 1:
        del qd, kd, vd, od, ld
        torch.cuda.empty_cache()
        line["per_config"] = per_config_lines(fa, dev, local, stream, burst, sustained, args.per_config_s)
        line["per_config_peaks"] = {"burst": burst, "sustained": sustained, "kind": pk_kind,
                                    "note": "fp16 workloads are compared with the bf16 dense peak "
                                            "(the same tensor rate; only bf16 was measured)"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="train_causal", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer leg (its chunked launches would mix into an ncu launch list)")
    ap.add_argument("--no-per-config", action="store_true", help="time only the selected workload")
    ap.add_argument("--per-config-s", type=float, default=0.5,
                    help="seconds each workload of the per-config table is timed for")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
