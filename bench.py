"""Benchmark: batched token sampling throughput on one GB300 (and N GPUs as independent row shards).

Workload (default): a decode batch of B=1024 rows x V=128,256 float32 logits ~ N(0, 2.5^2) with a
20-token head raised by +6; every row T=0.7, top_k=50, top_p=0.9, min_p=0.05, distinct seeds; the
step counter advances each iteration.  One step = one call of the sampler over the whole batch.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU oracle instead, on the
host cores, over a bounded sample of the same rows.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "rows/s & HBM GB/s (% of peak) at B=1024 V=128256 fp32; p50 us at B=1"
UNIT = "rows/s"
ROW_PARAM_BYTES = 4 + 4 + 4 + 4 + 8 + 4  # T, top_k, top_p, min_p, seed, token out
# The sources the streaming kernel (the dominant kernel of the decode step) and its launch plan are
# built from: a committed ncu traffic figure applies only while their hash is unchanged.
KERNEL_SOURCES = ["nucleus_token_sampler_gb300/csrc/tps_stream.cuh",
                  "nucleus_token_sampler_gb300/csrc/tps_common.cuh",
                  "nucleus_token_sampler_gb300/csrc/tps_device.cuh",
                  "nucleus_token_sampler_gb300/csrc/tps_kernels.h",
                  "nucleus_token_sampler_gb300/csrc/tps_k_stream_f32.cu",
                  "nucleus_token_sampler_gb300/csrc/tps_k_stream_bf16.cu",
                  "nucleus_token_sampler_gb300/csrc/tps_api.cu"]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--B", type=int, default=1024)
    ap.add_argument("--V", type=int, default=128256)
    ap.add_argument("--dtype", default="f32", choices=["f32", "bf16"])
    ap.add_argument("--workload", default="decode", choices=["decode", "sweep", "mixed", "ties_masked", "small"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-latency", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--kernel", default="auto", choices=["auto", "cluster", "stream"])
    ap.add_argument("--logprobs", type=int, default=-1, metavar="N",
                    help="also return the sampled token's processed log-probability and the top N (0..32) "
                         "in every step")
    ap.add_argument("--penalties", type=int, default=0, metavar="H",
                    help="run the penalty kernel (histories of up to H tokens per row) ahead of the sampler "
                         "in every step")
    ap.add_argument("--draw", default="race", choices=["race", "rejection", "spec"],
                    help="time the exponential-race sampler (default), the sort-free rejection draw, or speculative "
                         "acceptance of one draft token per row (draft = the step's logits plus noise)")
    ap.add_argument("--no-sustained", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="time the sweep grid (B x V x dtype, sweep workload) and print one JSON table instead")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank: int, world: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank samples its own rows (the batch is sharded by rows, no
    collective on the data path), timed by the slowest rank."""
    return rows_per_rank * world * steps / (total_ms / 1e3)


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def committed_traffic(workload_tag: str):
    """ncu DRAM bytes per launch for this kernel source and workload, if a capture was committed."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(workload_tag)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def make_workload(args, device, seed=0):
    from nucleus_token_sampler_gb300 import workloads
    dt = torch.float32 if args.dtype == "f32" else torch.bfloat16
    if args.workload == "decode":
        return workloads.make("decode", device=device, seed=seed, B=args.B, V=args.V, dtype=dt)
    if args.workload == "sweep":
        return workloads.make("sweep", device=device, seed=seed, B=args.B, V=args.V, dtype=dt)
    return workloads.make(args.workload, device=device, seed=seed)


def cpu_baseline(w, gpu=None, seconds=10.0, max_passes=16, chunk=128):
    """Time the float64 oracle on the host cores over a bounded sample of the workload: passes over
    the device workload's rows (copied to the host), pass q at step counter step + q, in chunks of
    `chunk` rows, until about `seconds` of oracle time or `max_passes` passes; rows/s.  With `gpu`
    (one GPU call's diagnostics on the same rows at the same step), the first pass's oracle outputs
    also check the GPU: tokens, kept counts, cutoffs and statuses outside the boundary band must
    match exactly, and the boundary rows are counted by kind."""
    import oracle
    o = oracle.default()
    cores = o.max_threads()
    B = w.B
    spent = 0.0
    done = 0
    outs = []
    chunks = []
    for q in range(max_passes):
        for c, r0 in enumerate(range(0, B, chunk)):
            r1 = min(B, r0 + chunk)
            if q == 0:  # host copies of the chunk, made once and outside the timed calls
                sel = lambda t: t[r0:r1].cpu().numpy()
                chunks.append((w.logits[r0:r1].double().cpu().numpy(), sel(w.temperature), sel(w.top_k),
                               sel(w.top_p), sel(w.min_p), sel(w.seed).astype(np.uint64)))
            z, T, k, p, m, sd = chunks[c]
            t0 = time.perf_counter()
            res = o.sample(z, T, k, p, m, sd, w.step + q, row_ids=np.arange(r0, r1))
            spent += time.perf_counter() - t0
            done += r1 - r0
            if q == 0:
                outs.append(res)
            if spent >= seconds and q > 0:
                break
        if spent >= seconds:
            break
    passes = q + 1
    # one core, on the first rows of the same workload
    n1 = min(16, B)
    z = w.logits[:n1].double().cpu().numpy()
    t0 = time.perf_counter()
    o.sample(z, w.temperature[:n1].cpu().numpy(), w.top_k[:n1].cpu().numpy(), w.top_p[:n1].cpu().numpy(),
             w.min_p[:n1].cpu().numpy(), w.seed[:n1].cpu().numpy().astype(np.uint64), w.step, row_ids=np.arange(n1),
             nthreads=1)
    one_core = n1 / (time.perf_counter() - t0)
    res = {"value": done / spent, "unit": "rows/s", "cores": cores, "kind": "oracle",
           "sample": f"{done} rows: {passes} pass(es) over the {B} rows of the same workload at successive step "
                     f"counters, float64 oracle, OpenMP over rows ({spent:.1f} s)",
           "one_core_rows_per_s": round(one_core, 1), "cpu": cpu_model()}
    if gpu is not None and outs:
        cat = lambda k: np.concatenate([x[k] for x in outs])
        ot, ok_, oc, os_, of = cat("token"), cat("kept"), cat("cutoff"), cat("status"), cat("flags")
        g = {k: v.cpu().numpy() for k, v in gpu.items()}
        band = (of & 3) != 0
        race = (of & 4) != 0
        chk = (os_ == 0) & ~band
        mism = int((chk & ~race & (g["token"] != ot)).sum() + (chk & (g["kept"] != ok_)).sum() +
                   (chk & (g["cutoff"].astype(np.float64) != oc)).sum() + (g["status"] != os_).sum())
        res["parity"] = {"rows_checked": int(len(ot)), "mismatches_outside_band": mism,
                         "topp_band_rows": int(((of & 1) != 0).sum()), "minp_band_rows": int(((of & 2) != 0).sum()),
                         "race_margin_rows": int(race.sum())}
    return res


def cpu_model() -> str:
    """The host CPU as the OS describes it (model name, or the Arm implementer/part codes)."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.processor() or platform.machine()
    for key in ("model name", "Model"):
        for line in info:
            if line.split(":")[0].strip() == key:
                return line.split(":", 1)[1].strip()
    parts = {}
    for line in info:
        k = line.split(":")[0].strip()
        if k in ("CPU implementer", "CPU part") and k not in parts:
            parts[k] = line.split(":", 1)[1].strip()
    return f"{platform.machine()} " + " ".join(f"{k.split()[-1]} {v}" for k, v in parts.items())


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    o = oracle.default()
    w = make_workload(args, "cpu")
    # each step: a bounded sample of rows (sized so the whole run stays within a few minutes)
    per_step = max(1, min(w.B, 16))
    times = []
    total_steps = args.warmup + args.steps
    for it in range(total_steps):
        rows = (np.arange(per_step) + it * per_step) % w.B
        t0 = time.perf_counter()
        o.sample(w.logits[rows].double().numpy(), w.temperature[rows].numpy(), w.top_k[rows].numpy(),
                 w.top_p[rows].numpy(), w.min_p[rows].numpy(), w.seed[rows].numpy().astype(np.uint64), it,
                 row_ids=rows)
        if it >= args.warmup:
            times.append(time.perf_counter() - t0)
    secs = sum(times)
    value = per_step * len(times) / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": o.max_threads(), "kind": "oracle",
                         "sample": f"{per_step} rows per step of the {w.B}-row workload, float64 oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def penalty_kernel_stats(pen, penalise, stream, B, V, es, calls=50):
    """The penalty kernel timed alone (CUDA events around a graph of `calls` launches) against its
    algorithmic bytes: each row's history entries (4 B), a read and a write of each distinct token's
    logit, and the row's four parameters."""
    n = pen.hist_len.long().cpu()
    h = pen.history.cpu()
    distinct = 0
    for b in range(B):
        row = h[b, : int(n[b])]
        distinct += int(torch.unique(row[(row >= 0) & (row < V)]).numel())
    alg = int(4 * n.sum().item() + 2 * es * distinct + 16 * B)
    # Device time: `calls` launches captured in one CUDA graph (back-to-back Python calls would time
    # the host instead).
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        penalise()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(calls):
                penalise()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / calls
    return {"history": int(pen.history.shape[1]), "kernel_us": round(us, 2), "algorithmic_bytes": alg,
            "distinct_tokens_per_row": round(distinct / B, 1), "gbs": round(alg / (us * 1e-6) / 1e9, 1),
            "note": "in place on the step's logits; timed alone from a CUDA graph replay, L2-warm (the "
                    "history and the touched lines fit L2)"}


L2_BYTES = 129e6  # GB300's L2


def in_bytes(w) -> int:
    return w.logits.numel() * w.logits.element_size()


def timed_steps(step, first, steps, stream, flush, dev):
    """Time `steps` calls step(first), step(first + 1), ... with CUDA events on `stream`.  The steps
    are enqueued behind a GPU spin, so the host's launch gaps are not timed.  flush=False: back to
    back, one event between steps (inputs larger than L2); flush=True: a 512 MB buffer is written
    between steps, each step timed alone.  Returns (per-step ms, total ms, host wall seconds)."""
    torch.cuda._sleep(int(min(200e6, 2e6 * steps)))
    if not flush:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        t0 = time.perf_counter()
        ev[0].record(stream)
        for i in range(steps):
            step(first + i)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
        return per, ev[0].elapsed_time(ev[-1]), wall
    scrub = torch.empty(128 << 20, dtype=torch.float32, device=dev)
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = time.perf_counter()
    for i in range(steps):
        scrub.fill_(float(i))
        ea[i].record(stream)
        step(first + i)
        eb[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    per = [ea[i].elapsed_time(eb[i]) for i in range(steps)]
    return per, sum(per), wall


def workload_config(args, w):
    """The workload as it was built (a named workload other than decode and sweep has its own B, V
    and dtype)."""
    dt = "f32" if w.logits.dtype == torch.float32 else "bf16"
    mb = in_bytes(w) / 1e6
    return {"workload": f"{args.workload}_b{w.B}_v{w.V}_{dt}", "B": w.B, "V": w.V,
            "logits_dtype": dt, "params": "T=0.7 top_k=50 top_p=0.9 min_p=0.05" if args.workload == "decode"
            else args.workload, "parallelism": "rows sharded over ranks (replicas, no collective)",
            "l2": ("inputs larger than L2 (no flush): %.0f MB of logits per step per GPU" % mb if in_bytes(w) > 2 * L2_BYTES
                   else "inputs within 2x L2 (%.0f MB of logits per step per GPU): a 512 MB buffer is written "
                        "between timed steps and each step is timed alone" % mb),
            "timing": "CUDA events on the launching stream around each step; the K steps are enqueued behind "
                      "a GPU spin so host launch gaps are not timed",
            **({"penalties": f"repetition/frequency/presence, histories of up to {args.penalties} tokens"}
               if args.penalties else {}),
            **({"logprobs": f"sampled token's processed log-probability and the top {args.logprobs}"}
               if args.logprobs >= 0 else {})}


def run_sweep(args):
    """The sweep grid: every B x V x dtype point of the sweep workload (top-p ~ U[.1, 1], T ~ U[.3, 2],
    no top-k, no min-p), timed like the main run (warm-up, then timed_steps: back to back for inputs
    larger than 2x L2, L2 scrubbed between steps otherwise) through the chosen kernel.  Prints one
    JSON object with a row per point."""
    import nucleus_token_sampler_gb300 as tps
    from nucleus_token_sampler_gb300 import workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    tps.load()
    peak, peak_kind = measured_peaks()
    rows = []
    for dt_name, dt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        es = 4 if dt == torch.float32 else 2
        for V in workloads.SWEEP_V:
            for B in workloads.SWEEP_B:
                w = workloads.make("sweep", device=dev, B=B, V=V, dtype=dt)
                out = {"token": torch.empty(B, dtype=torch.int32, device=dev)}

                def call(i):
                    tps.sample(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, i, out=out, kernel=args.kernel)

                for i in range(args.warmup):
                    call(i)
                torch.cuda.synchronize()
                flush = in_bytes(w) <= 2 * L2_BYTES
                per, total, _ = timed_steps(call, args.warmup, args.steps, torch.cuda.current_stream(dev), flush, dev)
                ms = total / args.steps
                alg = B * (V * es + ROW_PARAM_BYTES)
                gbs = alg / (ms / 1e3) / 1e9
                rows.append({"dtype": dt_name, "B": B, "V": V, "us_per_step": round(ms * 1e3, 2),
                             "rows_per_s": round(B / (ms / 1e3), 1), "gbs": round(gbs, 1),
                             "frac": round(gbs / peak, 4), "kernels": tps.kernels_per_call(dt, B, V, args.kernel),
                             "p50_us": round(statistics.median(per) * 1e3, 2),
                             "l2": "flushed between steps" if flush else "larger than 2x L2 (back to back)"})
                del w, out
                torch.cuda.empty_cache()
    print(json.dumps({"sweep": rows, "kernel": args.kernel, "steps": args.steps, "warmup": args.warmup,
                      "peak_gbs": peak, "peak_kind": peak_kind,
                      "workload": "sweep: logits ~ N(0, 2^2), top_p ~ U[.1, 1], T ~ U[.3, 2], no top-k, no min-p"}))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    import nucleus_token_sampler_gb300 as tps

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    tps.load()

    w = make_workload(args, dev, seed=rank)
    B, V = w.B, w.V
    es = w.logits.element_size()
    stream = torch.cuda.current_stream(dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    out = {"token": tok}
    lp_kw = {}
    if args.logprobs >= 0:
        n = args.logprobs
        out.update(logprob=torch.empty(B, dtype=torch.float32, device=dev),
                   top_idx=torch.empty((B, n), dtype=torch.int32, device=dev),
                   top_logprob=torch.empty((B, n), dtype=torch.float32, device=dev))
        lp_kw = {"want_logprob": True, "top_logprobs": n}
    pen = None
    if args.penalties:
        from nucleus_token_sampler_gb300 import workloads
        pen = workloads.penalty_inputs(B, V, args.penalties, device=dev, seed=rank)

    def penalise():
        tps.apply_penalties(w.logits, pen.history, pen.hist_len, repetition=pen.repetition,
                            frequency=pen.frequency, presence=pen.presence)

    spec = None
    if args.draw == "spec":
        # draft rows: the target's logits plus N(0, 0.5^2) noise, sampled by the draft's own parameters
        g = torch.Generator(device=dev).manual_seed(1234 + rank)
        zd = (w.logits.float() + 0.5 * torch.randn(w.logits.shape, generator=g, device=dev)).to(w.logits.dtype)
        dp = (torch.full_like(w.temperature, 0.9), torch.zeros_like(w.top_k), torch.full_like(w.top_p, 0.95),
              torch.full_like(w.min_p, 0.02))
        x = tps.sample(zd, *dp, w.seed + 7, 0)
        spec = (zd, dp, x)

    def step(i):
        if pen is not None:
            penalise()  # in place, as an engine does on each step's fresh logits
        if args.draw == "rejection":
            tps.sample_rejection(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, i)
        elif args.draw == "spec":
            tps.spec_accept(w.logits, spec[0], (w.temperature, w.top_k, w.top_p, w.min_p), spec[1], spec[2], w.seed, i)
        else:
            tps.sample(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, i, out=out, kernel=args.kernel,
                       **lp_kw)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    clocks = ClockSampler(local) if not args.no_clocks else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if clocks:  # the sampler starts while the GPU runs untimed steps, so its samples are under load
        clocks.start()
        t0 = time.perf_counter()
        i = 0
        while time.perf_counter() - t0 < 0.5:
            step(50_000 + i)
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
    per, total_ms, t_wall = timed_steps(step, args.warmup, args.steps, stream, in_bytes(w) <= 2 * L2_BYTES, dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_rows_per_s(B, world, args.steps, total_ms)

    # roofline of the step: the algorithmic bytes over the step's device time.  A step is one call,
    # which launches the scratch clear and the streaming kernel (and the cluster kernel behind it for
    # a split batch); the step time covers all of them, so this is a lower bound on the streaming
    # kernel's own throughput (its share of the step is in the committed ncu launch list).
    alg_bytes = B * ((2 if args.draw == "spec" else 1) * V * es + ROW_PARAM_BYTES)
    kern_ms = statistics.mean(per)
    achieved = alg_bytes / (kern_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    dt_name = "f32" if w.logits.dtype == torch.float32 else "bf16"
    tag = f"{args.workload}_b{B}_v{V}_{dt_name}" + (f"_pen{args.penalties}" if pen is not None else "") + (
        f"_lp{args.logprobs}" if args.logprobs >= 0 else "")
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
            "frac_of_8000": round(achieved / 8000.0, 4), "traffic": committed_traffic(tag),
            "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms_mean": round(kern_ms, 5),
            "kernel_ms_p50": round(statistics.median(per), 5), "kernel_ms_min": round(min(per), 5),
            "kernel_ms_max": round(max(per), 5)}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dt_name, "data": "synthetic",
            "config": workload_config(args, w), "roofline": roof,
            "gpu_launches": args.steps * (launches_per_step(args, tps, w) + (pen is not None)),
            "hbm_gbs": round(achieved, 1), "us_per_step": round(1e3 * ms_per_step, 2),
            "wall_s_timed": round(t_wall, 3), "cluster_size": tps.cluster_size(w.logits.dtype, B, V)}
    if clk:
        line["clocks"] = clk
    if pen is not None:
        line["penalties"] = penalty_kernel_stats(pen, penalise, stream, B, V, es)

    if args.draw != "race":
        line["config"]["draw"] = args.draw
    if rank == 0 and world == 1 and not args.no_sustained:
        line["sustained"] = sustained(args, step, stream, B, local)
    if rank == 0 and not args.no_latency:
        line["latency_b1"] = latency_b1(args, dev)
    if not args.no_e2e:
        line["e2e"] = e2e(args, w, dev, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gpu = None
        if args.draw == "race" and pen is None:  # the sampler's own answer on the same rows, same step
            gpu = tps.sample(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, w.step, diagnostics=True,
                             kernel=args.kernel)
            torch.cuda.synchronize()
        line["cpu_baseline"] = cpu_baseline(w, gpu)
        if "parity" in line["cpu_baseline"]:
            line["parity"] = line["cpu_baseline"]["parity"]
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def launches_per_step(args, tps, w):
    """Kernels one step launches (the library's own count for the sampler call)."""
    if args.draw in ("rejection", "spec"):
        return 1
    return tps.kernels_per_call(w.logits.dtype, w.B, w.V, args.kernel)


def sustained(args, step, stream, B, local, seconds=1.2):
    """At least a second of back-to-back steps (after the main timed region), timed with CUDA events
    on the launching stream, with the SM clock sampled by nvidia-smi during it; the samples are also
    binned by clock so a throttled stretch would show."""
    n = 50
    for i in range(n):
        step(10_000 + i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        step(10_000 + i)
    e1.record(stream)
    torch.cuda.synchronize()
    per = e0.elapsed_time(e1) / n
    steps = max(50, int(seconds * 1e3 / per))
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0.record(stream)
    for i in range(steps):
        step(20_000 + i)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    out = {"steps": steps, "seconds": round(ms / 1e3, 3), "ms_per_step": round(ms / steps, 5),
           "value": B * steps / (ms / 1e3), "unit": UNIT}
    if clk:
        out["clocks"] = clk
    return out


def latency_b1(args, dev, calls=300):
    """B=1 latency at the same V and dtype (the decode distribution), three ways:
    - graph: one call captured in a CUDA graph and replayed back to back; the interval between
      consecutive events is the device time of one call (launch to completion, no host gap);
    - in_graph: 20 calls captured in one graph, the replay's time per call (no graph launch per
      call: what the call costs inside a captured decode step);
    - isolated: event, Python call, event, synchronize -- includes the host-side marshalling of the
      call, i.e. what one unbatched request sees end to end on an idle GPU."""
    import nucleus_token_sampler_gb300 as tps
    from nucleus_token_sampler_gb300 import workloads
    dt = torch.float32 if args.dtype == "f32" else torch.bfloat16
    w = workloads.make("decode", device=dev, seed=7, B=1, V=args.V, dtype=dt)
    tok = {"token": torch.empty(1, dtype=torch.int32, device=dev)}
    s = torch.cuda.current_stream(dev)
    for i in range(20):
        tps.sample(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, i, out=tok)
    torch.cuda.synchronize()

    def pct(ts):
        ts = sorted(ts)
        return round(ts[len(ts) // 2], 2), round(ts[int(len(ts) * 0.9)], 2), round(ts[min(len(ts) - 1, int(len(ts) * 0.99))], 2)

    iso = []
    for i in range(calls):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        tps.sample(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, i, out=tok)
        b.record(s)
        b.synchronize()
        iso.append(a.elapsed_time(b) * 1e3)
    out = {"cluster_size": tps.cluster_size(dt, 1, args.V), "calls": calls}
    out["isolated_p50_us"], out["isolated_p90_us"], out["isolated_p99_us"] = pct(iso)
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                tps.sample(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, 12345, out=tok)
        s.wait_stream(side)
        for _ in range(20):
            g.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(calls + 1)]
        ev[0].record(s)
        for i in range(calls):
            g.replay()
            ev[i + 1].record(s)
        torch.cuda.synchronize()
        gt = [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(calls)]
        out["p50_us"], out["p90_us"], out["p99_us"] = pct(gt)
        out["method"] = "CUDA graph replays back to back; events between replays"
        # The same call inside a longer graph (as when a serving loop captures its whole decode step):
        # 20 calls per graph, the replay's time divided by 20; median of 15 replays.
        g20 = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            side.wait_stream(s)
            with torch.cuda.graph(g20, stream=side):
                for i in range(20):
                    tps.sample(w.logits, w.temperature, w.top_k, w.top_p, w.min_p, w.seed, 20000 + i, out=tok)
        s.wait_stream(side)
        for _ in range(3):
            g20.replay()
        torch.cuda.synchronize()
        per = []
        for _ in range(15):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            g20.replay()
            b.record(s)
            b.synchronize()
            per.append(a.elapsed_time(b) * 1e3 / 20)
        out["in_graph_us"] = round(sorted(per)[len(per) // 2], 2)
        out["in_graph_method"] = "20 calls captured in one CUDA graph; replay time / 20, median of 15 replays"
    except Exception as e:  # graph capture unavailable: report the isolated numbers only
        out["graph_error"] = str(e)[:200]
        out["p50_us"], out["p90_us"], out["p99_us"] = out["isolated_p50_us"], out["isolated_p90_us"], out["isolated_p99_us"]
        out["method"] = "isolated calls"
    return out


def e2e(args, w, dev, world, steps=None, nstreams=4):
    """Same metric through the public call with host buffers: per step, pinned host logits and
    parameters are copied to the device, the batch is sampled and the tokens are read back.  The
    logits copy is split by rows over `nstreams` copy streams (several DMA engines), and the device
    inputs are double-buffered so that one step's copy overlaps the previous step's sampling; every
    step still copies all of its inputs inside the timed region."""
    import nucleus_token_sampler_gb300 as tps
    steps = steps or max(3, min(args.steps, 20))
    B, V = w.B, w.V
    keys = ("logits", "temperature", "top_k", "top_p", "min_p", "seed")
    host = {k: getattr(w, k).cpu().pin_memory() for k in keys}
    bufs = [{k: torch.empty_like(getattr(w, k)) for k in keys} for _ in range(2)]
    tok_h = torch.empty(B, dtype=torch.int32).pin_memory()
    out = {"token": torch.empty(B, dtype=torch.int32, device=dev)}
    s = torch.cuda.current_stream(dev)
    copiers = [torch.cuda.Stream(dev) for _ in range(nstreams)]
    bounds = [B * c // nstreams for c in range(nstreams + 1)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = tok_h.numel() * 4
    freed = [None, None]  # per buffer: an event after the last sampling that read it

    def one(i, gate):
        db = bufs[i % 2]
        ready = []
        for c, st in enumerate(copiers):
            st.wait_event(gate)
            if freed[i % 2] is not None:
                st.wait_event(freed[i % 2])
            with torch.cuda.stream(st):
                r0, r1 = bounds[c], bounds[c + 1]
                db["logits"][r0:r1].copy_(host["logits"][r0:r1], non_blocking=True)
                if c == 0:
                    for k in keys[1:]:
                        db[k].copy_(host[k], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(st)
            ready.append(ev)
        for ev in ready:
            s.wait_event(ev)
        tps.sample(db["logits"], db["temperature"], db["top_k"], db["top_p"], db["min_p"], db["seed"], i, out=out)
        tok_h.copy_(out["token"], non_blocking=True)
        freed[i % 2] = torch.cuda.Event()
        freed[i % 2].record(s)

    start = torch.cuda.Event(enable_timing=True)
    start.record(s)
    for i in range(3):
        one(i, start)
    torch.cuda.synchronize()
    freed[0] = freed[1] = None
    if world > 1:
        torch.distributed.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s)
    for i in range(steps):
        one(i, a)  # no copy starts before the timed region does
    b.record(s)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": B * world * steps / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "copy_streams": nstreams,
            "h2d_gbs": round(h2d * steps / (ms / 1e3) / 1e9, 1)}


if __name__ == "__main__":
    sys.exit(main())
