#!/usr/bin/env python3
"""Benchmark of the fused MoE finalize + residual + RMSNorm path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
                    [--impl ours|reference] [--sweep] [--no-cpu-baseline]

One step = one call of the whole path (gather, FP32 weighted sum, residual
update, RMSNorm, bf16 store) over one batch of synthetic inputs already
resident in HBM.  The headline workload is the prefill configuration
(T=16384 tokens, H=4096, top-8, 128 experts, Zipf(1.2) routing); its inputs
(1.75 GB per call) are far larger than L2, and two input/output sets are
alternated so no step starts with its data in L2.

The metric is effective HBM bandwidth: algorithmic bytes per call
(T*k*H*2 + T*H*(4+4+2) + T*k*8) divided by the device time of a call.

Under torchrun each rank runs its own independent batch on its own GPU
(tokens are independent, so the path shards with no collective): weak
scaling, value = all ranks' bytes / the slowest rank's time.

--impl reference times the CPU oracle (the plain C reference) on the host
cores on a bounded sample of the same workload, in the same metric.
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

import workloads as W  # noqa: E402

METRIC = "effective HBM GB/s (% of GB300 peak) and µs/call vs tokens T, H=4096/8192, k=8"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = {
    "stream": ["moe_finalize_residual_rmsnorm_gb300/csrc/mfr_stream.cu",
               "moe_finalize_residual_rmsnorm_gb300/csrc/mfr_device.cuh"],
    "rows": ["moe_finalize_residual_rmsnorm_gb300/csrc/mfr_rows.cu",
             "moe_finalize_residual_rmsnorm_gb300/csrc/mfr_device.cuh"],
}
KERNEL_SOURCES["cluster"] = KERNEL_SOURCES["rows"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="prefill", choices=sorted(W.all_named()))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true",
                    help="also time the full decode and wide sweeps (graph, stream loop, warm L2, other outputs)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the compact sweep of the metric (decode T<=8 against its floor, wide H=8192, "
                         "stress), the other outputs and the producer pairs that the line carries by default")
    ap.add_argument("--variants", action="store_true",
                    help="time the other outputs on the headline workload even with --no-sweep")
    ap.add_argument("--pdl-pairs", action="store_true",
                    help="time producer -> finalize pairs even with --no-sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--variant", default="auto", choices=["auto", "rows", "stream", "cluster"])
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T of the workload (small cases for profiling)")
    ap.add_argument("--floor-probe", type=int, default=None, metavar="T",
                    help=argparse.SUPPRESS)   # internal: the launch floor of decode T in a fresh process
    ap.add_argument("--floor-device", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# --- distributed plumbing ---------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --- clocks -----------------------------------------------------------------------

class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout=10.0):
        """Blocks until nvidia-smi has printed its first sample."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        loaded = [v for v in sm if smax and v > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --- helpers ------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(variant: str):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[variant]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, variant: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload, {})
    if e.get("variant") != variant or e.get("kernel_hash") != kernel_source_hash(variant):
        return None
    return e.get("dram_bytes_per_launch")


def workload_config(wl) -> dict:
    """The workload keys of the JSON line's config, the same for both arms."""
    return {"workload": f"{wl.name}: T={wl.T} H={wl.H} k={wl.k} E={wl.E} routing={wl.routing}"
                        f"{'(s=%g)' % wl.zipf_s if wl.routing == 'zipf' else ''}",
            "tokens_per_gpu": wl.T, "hidden": wl.H, "top_k": wl.k, "experts": wl.E,
            "io": "bf16 expert rows and output, f32 residual in and out"}


def host_cpu() -> str:
    """The host CPU's name from /proc/cpuinfo (on Arm the implementer and part
    numbers, which lscpu maps to names such as Neoverse-V2 for 0x41/0xd4f)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
    except OSError:
        return os.uname().machine
    fields = {}
    for line in info:
        if ":" in line:
            key, _, val = line.partition(":")
            fields.setdefault(key.strip().lower(), val.strip())
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        return f"{os.uname().machine} implementer {fields.get('cpu implementer', '?')} part {fields['cpu part']}"
    return os.uname().machine


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# --- CPU oracle timing ------------------------------------------------------------------

def time_oracle(inp_host: dict, n_tokens: int, threads: int, rng_seed: int = 0):
    """Runs the oracle on n_tokens sampled tokens split over `threads` host
    threads (the C calls release the GIL).  Returns (seconds, tokens)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    T = inp_host["idx"].shape[0]
    rng = np.random.default_rng(rng_seed)
    if n_tokens <= T:
        tokens = np.sort(rng.choice(T, size=n_tokens, replace=False))
    else:   # more work than one pass: whole passes over the workload, each shuffled
        passes = -(-n_tokens // T)
        tokens = np.concatenate([rng.permutation(T) for _ in range(passes)])[:n_tokens]
    parts = [p for p in np.array_split(tokens, threads) if p.size]
    orc = oracle.default()

    def work(tk):
        return orc.finalize_residual_rmsnorm(inp_host["E"], inp_host["idx"], inp_host["w"], inp_host["res"],
                                             inp_host["gamma"], inp_host["eps"], tokens=tk)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        list(ex.map(work, parts))
    return time.perf_counter() - t0, int(tokens.size)


def host_copy(inp):
    def bits16(t):
        return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return {"E": bits16(inp["expert_out"]), "idx": inp["permuted_row_of"].cpu().numpy(),
            "w": inp["topk_weights"].cpu().numpy(), "res": inp["residual"].cpu().numpy(),
            "gamma": bits16(inp["gamma"]), "eps": inp["eps"]}


def calibrate_tokens(inp_host, T: int, target_s: float, cores: int) -> int:
    """Number of sampled tokens (repeating whole passes over the workload
    when one pass is quicker) the oracle processes in about target_s."""
    n = min(T, cores * 4)
    while True:
        dt, n = time_oracle(inp_host, n, cores, 1)
        if dt >= 0.3 * target_s:
            break
        n = int(n * min(16.0, max(2.0, 0.9 * target_s / max(dt, 1e-6))))
    return int(max(cores, n * target_s / max(dt, 1e-6)))


def cpu_baseline(inp_host, wl, target_s: float):
    cores = host_cores()
    n_tokens = calibrate_tokens(inp_host, wl.T, target_s, cores)
    dt, n = time_oracle(inp_host, n_tokens, cores, 2)
    gbs = W.algorithmic_bytes(n, wl.H, wl.k) / dt / 1e9
    # the same code on one thread, on a quarter of one thread's share of the sample
    dt1, n1 = time_oracle(inp_host, max(1, n // (4 * cores)), 1, 3)
    gbs1 = W.algorithmic_bytes(n1, wl.H, wl.k) / dt1 / 1e9
    return {"value": round(gbs, 4), "unit": UNIT, "cores": cores, "kind": "oracle", "cpu": host_cpu(),
            "sample": f"{n} tokens drawn from the {wl.T}-token workload (seeded; whole shuffled passes "
                      f"when more than {wl.T}), H={wl.H}, k={wl.k}, {dt:.2f} s wall, {cores} host threads",
            "single_thread": {"value": round(gbs1, 4), "unit": UNIT, "cores": 1,
                              "sample": f"{n1} tokens, {dt1:.2f} s wall, 1 host thread"}}


# --- the GPU arm -------------------------------------------------------------------------

def run_ours(args):
    import moe_finalize_residual_rmsnorm_gb300 as mfr

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    wl = W.by_name(args.workload).with_(seed=W.by_name(args.workload).seed + rank)
    if args.tokens:
        wl = wl.with_(T=args.tokens)
    T, H, k, R = wl.T, wl.H, wl.k, wl.R
    nbytes = W.algorithmic_bytes(T, H, k)

    mfr.load_library()
    variant = {"auto": mfr.VARIANT_AUTO, "rows": mfr.VARIANT_ROWS, "stream": mfr.VARIANT_STREAM,
               "cluster": mfr.VARIANT_CLUSTER}[args.variant]
    plan = mfr.Plan(T, H, k, R, enable_pdl=not args.no_pdl, variant=variant)
    info = plan.info()

    # two independent input/output sets, alternated every step
    sets = []
    for s in range(2):
        inp = W.make_inputs(wl.with_(seed=wl.seed * 2 + s), device)
        inp["residual_out"] = torch.empty_like(inp["residual"])
        inp["out"] = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        sets.append(inp)
    stream = torch.cuda.Stream(device)

    def step(i):
        d = sets[i & 1]
        plan.run(d["expert_out"], d["permuted_row_of"], d["topk_weights"], d["residual"], d["residual_out"],
                 d["gamma"], d["eps"], d["out"], stream, validate=False)

    torch.cuda.synchronize(device)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(device)

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        clocks.wait_first()
        barrier(dist, device)
        torch.cuda.synchronize(device)
        start.record(stream)
        for i in range(args.steps):
            step(i)
        stop.record(stream)
        stop.synchronize()
        torch.cuda.synchronize(device)
        barrier(dist, device)
    ms_local = start.elapsed_time(stop) / args.steps
    ms = max_over_ranks(dist, ms_local, device)
    if plan.get_status(stream) != 0:
        raise RuntimeError("the device status word reported an out-of-range index")

    value = nbytes * world / (ms * 1e-3) / 1e9
    achieved = nbytes / (ms_local * 1e-3) / 1e9
    peak, peak_kind = measured_peak()
    traffic = recorded_traffic(args.workload, info["variant_name"])

    # end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, plan, sets[0], nbytes, world, dist, device)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "us_per_call": round(ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {**workload_config(wl),
                   "bytes_per_call": nbytes, "variant": info["variant_name"], "grid": info["grid_x"],
                   "block": info["block"], "cluster": info["cluster"], "pdl": not args.no_pdl,
                   "l2": f"inputs larger than L2 ({nbytes / 1e9:.2f} GB/call) and 2 alternating input sets",
                   "parallelism": f"replicas x{world} (independent token batches)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic, "algorithmic_bytes": nbytes,
                     "kernel": {"rows": "rows_kernel", "cluster": "rows_kernel (cluster)",
                                "stream": "stream_kernel"}[info["variant_name"]]},
        "clocks": clocks.summary(),
        "gpu_launches": args.steps,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_sweep and not args.tokens:
        # per-GPU figures of the metric's other sizes: rank 0 alone measures them
        result["sweep"] = run_compact_sweep(mfr, device, args)
    if args.sweep:
        result["sweep_full"] = run_sweep(mfr, device, args)
    # the other outputs on the headline workload and the producer -> finalize
    # pairs ride on the default line too (rank 0), unless --no-sweep
    default_extras = rank == 0 and not args.no_sweep and not args.tokens
    if args.pdl_pairs or default_extras:
        result["pdl_pairs"] = run_pdl_pairs(mfr, device)
    if args.variants or default_extras:
        result["variants"] = run_variants(mfr, device, wl, sets, args)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(host_copy(sets[0]), wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        barrier(dist, device)      # the other ranks wait for rank 0's sweep and CPU baseline
        dist.destroy_process_group()


def run_e2e(args, plan, dev, nbytes, world, dist, device):
    """The same metric through the public C ABI with host buffers
    (moe_finalize_rmsnorm_run_host): every step copies all of its inputs from
    pinned host memory into a device workspace, runs the kernel and copies
    both outputs back.  Steps alternate between two streams and two
    workspaces, so one step's device-to-host copies run under the next
    step's host-to-device copies (each step still moves all of its bytes)."""
    import moe_finalize_residual_rmsnorm_gb300 as mfr
    host_in = {key: dev[key].cpu().pin_memory() for key in
               ("expert_out", "permuted_row_of", "topk_weights", "residual", "gamma")}
    host_in["eps"] = dev["eps"]
    host_out = [{"residual_out": torch.empty(dev["residual_out"].shape, dtype=torch.float32).pin_memory(),
                 "out": torch.empty(dev["out"].shape, dtype=torch.bfloat16).pin_memory()} for _ in range(2)]
    ws_bytes = plan.host_workspace_bytes()
    workspaces = [torch.empty(ws_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    streams = [torch.cuda.Stream(device) for _ in range(2)]
    steps = max(3, min(args.steps, 12))

    def step(i):
        return mfr.finalize_residual_rmsnorm_host(plan, host_in, host_out[i & 1], workspaces[i & 1], streams[i & 1])

    for i in range(2):
        step(i)
    torch.cuda.synchronize(device)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    start.record(streams[0])
    streams[1].wait_event(start)
    h2d = d2h = 0
    for i in range(steps):
        h2d, d2h = step(i)
    streams[0].wait_stream(streams[1])
    stop.record(streams[0])
    stop.synchronize()
    ms = max_over_ranks(dist, start.elapsed_time(stop) / steps, device)
    return {"value": round(nbytes * world / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4),
            "steps": steps, "api": "moe_finalize_rmsnorm_run_host (C ABI), pinned host buffers, 2 streams"}


def _quartiles(xs):
    q = np.percentile(np.asarray(xs, dtype=np.float64), [25, 50, 75])
    return float(q[1]), float(q[2] - q[0])


FLOOR_CALLS = 4096


def floor_graph_times(mfr, device, plan, replays, ncalls=FLOOR_CALLS):
    """Per-launch µs of `replays` replays of a CUDA graph of `ncalls` empty
    kernels with the plan's launch geometry (two untimed replays first)."""
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(ncalls):
                plan.launch_floor(stream)
        for _ in range(3):
            graph.replay()
        stream.synchronize()
        times = []
        for _ in range(replays):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3 / ncalls)
    del graph
    return times


def run_floor_probe(args):
    """--floor-probe T: the launch floor of the decode plan for T tokens,
    measured in this fresh process before any other work (printed as one
    JSON line)."""
    import moe_finalize_residual_rmsnorm_gb300 as mfr
    torch.cuda.set_device(args.floor_device)
    device = torch.device("cuda", args.floor_device)
    mfr.load_library()
    wl = W.decode(args.floor_probe)
    plan = mfr.Plan(wl.T, wl.H, wl.k, wl.R, enable_pdl=not args.no_pdl)
    times = floor_graph_times(mfr, device, plan, 25)
    med, iqr = _quartiles(times)
    print(json.dumps({"T": wl.T, "floor_us": med, "floor_iqr": iqr, "replays": len(times)}), flush=True)


def fresh_process_floors(device, tokens, args):
    """The launch floor of each decode size, each in a fresh process of its
    own.  An empty kernel's launch rate depends on the state of the process:
    in a fresh one a graph of 4096 empty 4-CTA launches runs 0.35 us per
    launch, and after other graphs of thousands of launches (even destroyed
    ones) or large calls have run in it, 0.53-0.59 us, on the same GPU
    (measured).  The fresh figure is the lower and the reproducible one, so
    it is the floor the decode target is computed on."""
    floors = {}
    for T in tokens:
        cmd = [sys.executable, os.path.abspath(__file__), "--floor-probe", str(T), "--floor-device", str(device.index)]
        if args.no_pdl:
            cmd.append("--no-pdl")
        try:
            out = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
            if out.returncode == 0:
                floors[T] = json.loads(out.stdout.strip().splitlines()[-1])
                continue
            why = out.stderr.strip().splitlines()[-1:] or [f"exit code {out.returncode}"]
        except (subprocess.TimeoutExpired, OSError, ValueError, IndexError) as e:
            why = [repr(e)]
        # the row then falls back to the floor measured in this process, and says so
        print(f"bench.py: fresh-process floor for T={T} not measured: {why[0][:200]}", file=sys.stderr)
    return floors


def decode_against_floor(mfr, device, wl, args, replays=25, ncalls=4096, floor=None):
    """One decode size: the call, its launch floor and its one-pass floors,
    measured in the same run.

    Every figure is a CUDA graph of `ncalls` launches on one stream, per
    launch, median and interquartile range over `replays` replays.  All use
    the plan's exact launch geometry and PDL attribute.
      floor_us     the empty kernel (moe_finalize_rmsnorm_launch_floor), the
                   launch floor the decode target is defined on, measured in a
                   fresh process (`floor`, from fresh_process_floors) when
                   given; floor_in_process_us is the same graph measured here,
                   alone and after two untimed replays (the first replay of an
                   empty-kernel graph after data-moving work runs up to 2.5x
                   slower), as context.
      us_per_call  the call, cycling through enough input/output sets to
                   exceed 3x L2 (each call reads cold data).
      load_floor_us, store_floor_us, pass_floor_us, pass_exchange_floor_us
                   the empty kernel plus only the call's loads, only its
                   stores, both, and both with one cluster barrier between
                   them, over the same cold input sets, no arithmetic
                   (moe_finalize_rmsnorm_launch_floor_work): the launch plus
                   one pass over the call's bytes, measured.
    The call and the four work floors are replayed in turn, `replays`
    rounds.  The SM clock is sampled throughout.  The target is
    us_per_call <= 2 * (floor_us + bytes / 8 TB/s) (vs_2x_floor);
    vs_2x_pass_floor compares with twice the measured one-pass floor."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nbytes = W.algorithmic_bytes(wl.T, wl.H, wl.k)
    nsets = int(min(ncalls, max(2, -(-3 * l2 // max(nbytes, 1)))))
    base = W.make_inputs(wl, device)
    T, H, k, R = wl.T, wl.H, wl.k, wl.R
    E = base["expert_out"].unsqueeze(0).expand(nsets, R, H).contiguous()
    idx = base["permuted_row_of"].unsqueeze(0).expand(nsets, T, k).contiguous()
    w = base["topk_weights"].unsqueeze(0).expand(nsets, T, k).contiguous()
    res = base["residual"].unsqueeze(0).expand(nsets, T, H).contiguous()
    rout = torch.empty_like(res)
    out = torch.empty((nsets, T, H), dtype=torch.bfloat16, device=device)
    g, eps = base["gamma"], base["eps"]
    plan = mfr.Plan(T, H, k, R, enable_pdl=not args.no_pdl)
    stream = torch.cuda.Stream(device)
    work = {"load": mfr.FLOOR_LOAD, "store": mfr.FLOOR_STORE, "pass": mfr.FLOOR_LOAD | mfr.FLOOR_STORE,
            "pass_exchange": mfr.FLOOR_LOAD | mfr.FLOOR_EXCHANGE | mfr.FLOOR_STORE}

    def capture(kind):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(ncalls):
                j = i % nsets
                if kind == "floor":
                    plan.launch_floor(stream)
                elif kind == "call":
                    plan.run(E[j], idx[j], w[j], res[j], rout[j], g, eps, out[j], stream, validate=False)
                else:
                    plan.launch_floor_work(work[kind], E[j], idx[j], res[j], rout[j], out[j], stream)
        graph.replay()
        stream.synchronize()
        return graph

    def timed(graph):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) * 1e3 / ncalls

    times = {kind: [] for kind in ("floor", "call", *work)}
    with ClockSampler(device.index) as clocks, torch.cuda.stream(stream):
        clocks.wait_first()
        floor_graph = capture("floor")
        for _ in range(2):
            timed(floor_graph)
        times["floor"] = [timed(floor_graph) for _ in range(replays)]
        del floor_graph
        graphs = {kind: capture(kind) for kind in ("call", *work)}
        for _ in range(replays):
            for kind, graph in graphs.items():
                times[kind].append(timed(graph))
        del graphs
    if plan.get_status(stream) != 0:
        raise RuntimeError(f"the device status word reported an error during {wl.name}")
    q = {kind: _quartiles(v) for kind, v in times.items()}
    us, ps = q["call"][0], q["pass"][0]
    fl_here, fl_here_iqr = q["floor"]
    fl, fl_iqr = (floor["floor_us"], floor["floor_iqr"]) if floor else (fl_here, fl_here_iqr)
    ck = clocks.summary()
    info = plan.info()
    del E, idx, w, res, rout, out, base
    torch.cuda.empty_cache()
    return {"workload": wl.name, "T": T, "H": H, "us_per_call": round(us, 3), "us_iqr": round(q["call"][1], 3),
            "floor_us": round(fl, 3), "floor_iqr": round(fl_iqr, 3),
            "floor_where": "fresh process" if floor else "this process",
            "vs_2x_floor": round(us / (2 * (fl + nbytes / 8e12 * 1e6)), 3),
            "floor_in_process_us": round(fl_here, 3),
            "load_floor_us": round(q["load"][0], 3), "store_floor_us": round(q["store"][0], 3),
            "pass_floor_us": round(ps, 3), "pass_floor_iqr": round(q["pass"][1], 3),
            "pass_exchange_floor_us": round(q["pass_exchange"][0], 3),
            "vs_2x_pass_floor": round(us / (2 * ps), 3),
            "sm_mhz": ck["sm_mhz"], "us_x_mhz": round(us * ck["sm_mhz"], 1) if ck["sm_mhz"] else None,
            "clock_reasons": ck["reasons"], "replays": replays, "graph_calls": ncalls, "sets": nsets,
            "variant": info["variant_name"], "cluster": info["cluster"]}


def bandwidth_row(mfr, device, wl, args, steps, peak, repeat_check=False):
    """µs/call, GB/s and fraction of the measured copy bandwidth for one
    workload, timed like the headline step (CUDA events around `steps`
    calls on one stream, captured in a CUDA graph and replayed three times
    when a call moves less than 256 MB; input/output sets rotate so that
    together they exceed 3x L2 and no call starts with its data in L2).  With
    repeat_check, two further calls into fresh buffers must reproduce the
    first call's outputs bit for bit."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    T, H, k, R = wl.T, wl.H, wl.k, wl.R
    nbytes = W.algorithmic_bytes(T, H, k)
    nsets = int(min(16, max(2, -(-3 * l2 // nbytes))))
    sets = []
    for s in range(nsets):
        d = W.make_inputs(wl.with_(seed=wl.seed * 16 + s), device) if s < 2 or nbytes > l2 else None
        if d is None:   # small calls: further sets are copies of the first two (what matters is the address)
            d = {key: (v.clone() if torch.is_tensor(v) else v) for key, v in sets[s % 2].items()
                 if key not in ("residual_out", "out")}
        d["residual_out"] = torch.empty_like(d["residual"])
        d["out"] = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        sets.append(d)
    plan = mfr.Plan(T, H, k, R, enable_pdl=not args.no_pdl)
    stream = torch.cuda.Stream(device)

    def step(i):
        d = sets[i % nsets]
        plan.run(d["expert_out"], d["permuted_row_of"], d["topk_weights"], d["residual"], d["residual_out"],
                 d["gamma"], d["eps"], d["out"], stream, validate=False)

    for i in range(max(3, nsets)):
        step(i)
    stream.synchronize()
    # calls shorter than a Python launch go through a CUDA graph, so the host
    # does not set the pace; larger calls are launched one by one
    graph = None
    if nbytes < (256 << 20):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for i in range(steps):
                    step(i)
            graph.replay()
        stream.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3 if graph is not None else 1
    with ClockSampler(device.index) as clocks, torch.cuda.stream(stream):
        clocks.wait_first()
        a.record(stream)
        for _ in range(reps):
            if graph is not None:
                graph.replay()     # on the current stream, which is `stream` here
            else:
                for i in range(steps):
                    step(i)
        b.record(stream)
        b.synchronize()
    us = a.elapsed_time(b) * 1e3 / (steps * reps)
    del graph
    info = plan.info()
    row = {"workload": wl.name, "T": T, "H": H, "us_per_call": round(us, 2),
           "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1), "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4),
           "bytes_per_call": nbytes, "steps": steps, "sets": nsets, "variant": info["variant_name"],
           "grid": info["grid_x"], "sm_mhz": clocks.summary()["sm_mhz"], "clock_reasons": clocks.summary()["reasons"]}
    if repeat_check:
        d = sets[0]
        step(0)
        stream.synchronize()
        ok = True
        for _ in range(2):
            r2, o2 = torch.empty_like(d["residual_out"]), torch.empty_like(d["out"])
            plan.run(d["expert_out"], d["permuted_row_of"], d["topk_weights"], d["residual"], r2, d["gamma"],
                     d["eps"], o2, stream, validate=False)
            stream.synchronize()
            ok = ok and torch.equal(r2.view(torch.int32), d["residual_out"].view(torch.int32)) and \
                torch.equal(o2.view(torch.int16), d["out"].view(torch.int16))
            del r2, o2
        row["bitwise_repeat"] = bool(ok)
    if plan.get_status(stream) != 0:
        raise RuntimeError(f"the device status word reported an error during {wl.name}")
    del sets
    torch.cuda.empty_cache()
    return row


def run_compact_sweep(mfr, device, args):
    """The metric's sweep in a form short enough for every run: decode
    T = 1, 2, 4, 8 at H = 4096 against the launch-plus-one-HBM-pass floor
    (decode_against_floor), the mid size T = 512 and T = 4096, 8192 at
    H = 8192, and the stress configuration T = 32768, H = 8192 with its
    bitwise-repeat check (bandwidth_row)."""
    peak, _ = measured_peak()
    t0 = time.perf_counter()
    floors = fresh_process_floors(device, (1, 2, 4, 8), args)
    decode = [decode_against_floor(mfr, device, W.decode(t), args, floor=floors.get(t)) for t in (1, 2, 4, 8)]
    bandwidth = [bandwidth_row(mfr, device, W.wide(512), args, 400, peak),
                 bandwidth_row(mfr, device, W.wide(4096), args, 60, peak),
                 bandwidth_row(mfr, device, W.wide(8192), args, 40, peak),
                 bandwidth_row(mfr, device, W.STRESS, args, 12, peak, repeat_check=True)]
    return {"decode": decode, "bandwidth": bandwidth, "peak_gbs": peak,
            "decode_target": "us_per_call <= 2 * (floor_us + bytes / 8 TB/s); floor_us: empty-kernel graph in a "
                             "fresh process; us_per_call: median of 25 graph replays of 4096 cold calls",
            "seconds": round(time.perf_counter() - t0, 1)}


def run_sweep(mfr, device, args):
    """µs/call and GB/s at each decode and wide size, with the plan the
    library picks, three ways:
      us_per_call  calls captured in a CUDA graph (a decode call is far
                   shorter than a Python launch), cycling through enough
                   input/output sets that together exceed 3x L2, so each call
                   reads cold data; median of 5 replays.  Graphs of small calls
                   hold 4096 calls, so every size is timed at the same
                   steady state.
      loop_us      the same calls launched one by one from Python through the C
                   ABI (pointers taken once), CUDA events around 200+ calls,
                   median of 5 batches; loop_vs_2x_floor is the decode target
                   on this loop and its floor (host-bound for small calls, so
                   it says little about the kernel: the graph figure does).
      warm_us      the graph over a single input set (inputs in L2; context only).
      other_outputs_us  at T <= 8, the plain finalize, NVFP4 and per-expert
                   RMSNorm outputs timed like us_per_call.
    The floor is the same graph (or loop) of empty kernels with the identical
    launch geometry and PDL attribute (moe_finalize_rmsnorm_launch_floor);
    the decode target is us_per_call <= 2 * (floor_us + bytes / 8 TB/s)."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    rows = []
    for wl in [W.decode(t) for t in W.DECODE_TOKENS] + [W.wide(t) for t in W.WIDE_TOKENS]:
        nbytes = W.algorithmic_bytes(wl.T, wl.H, wl.k)
        nsets = int(min(4096, max(2, -(-3 * l2 // max(nbytes, 1)))))
        base = W.make_inputs(wl, device)
        T, H, k, R = wl.T, wl.H, wl.k, wl.R
        E = base["expert_out"].unsqueeze(0).expand(nsets, R, H).contiguous()
        idx = base["permuted_row_of"].unsqueeze(0).expand(nsets, T, k).contiguous()
        w = base["topk_weights"].unsqueeze(0).expand(nsets, T, k).contiguous()
        res = base["residual"].unsqueeze(0).expand(nsets, T, H).contiguous()
        rout = torch.empty_like(res)
        out = torch.empty((nsets, T, H), dtype=torch.bfloat16, device=device)
        g = base["gamma"]
        plan = mfr.Plan(T, H, k, R, enable_pdl=not args.no_pdl)
        stream = torch.cuda.Stream(device)
        ncalls = max(nsets, 4096 if nbytes <= (16 << 20) else 64)

        def launch(i, floor, sets):
            if floor:
                plan.launch_floor(stream)
            else:
                j = i % sets
                plan.run(E[j], idx[j], w[j], res[j], rout[j], g, base["eps"], out[j], stream, validate=False)

        def graph_us(floor: bool, sets: int, reps=5):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(ncalls):
                    launch(i, floor, sets)
            graph.replay()
            stream.synchronize()
            times = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graph.replay()
                b.record(stream)
                b.synchronize()
                times.append(a.elapsed_time(b) * 1e3 / ncalls)
            del graph
            return float(np.median(times))

        # the stream loop goes through the C ABI with pointers taken once, so
        # it times the library's host path and the launch, not tensor indexing
        ptrs = [(E[j].data_ptr(), idx[j].data_ptr(), w[j].data_ptr(), res[j].data_ptr(), rout[j].data_ptr(),
                 g.data_ptr(), base["eps"], out[j].data_ptr(), stream.cuda_stream) for j in range(nsets)]

        def loop_us(floor: bool, batches=5):
            n = max(200, min(ncalls, 1000))
            run_ptrs, floor_fn, sh = plan.run_ptrs, plan.launch_floor, stream

            def batch():
                bad = 0
                for i in range(n):
                    if floor:
                        floor_fn(sh)
                    else:
                        bad |= run_ptrs(*ptrs[i % nsets])
                if bad:
                    raise RuntimeError(f"moe_finalize_rmsnorm_run failed during {wl.name}")
            batch()
            stream.synchronize()
            times = []
            for _ in range(batches):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                batch()
                b.record(stream)
                b.synchronize()
                times.append(a.elapsed_time(b) * 1e3 / n)
            return float(np.median(times))

        with torch.cuda.stream(stream):
            us = graph_us(False, nsets)
            floor_us = graph_us(True, nsets)
            warm = graph_us(False, 1)
            loop = loop_us(False)
            loop_floor = loop_us(True)
            # the other outputs at decode sizes, timed the same way (graph, cold sets)
            others = {}
            if T <= 8:
                q = torch.empty((nsets, T, H // 2), dtype=torch.uint8, device=device)
                sf = torch.empty((nsets, T, H // 16), dtype=torch.uint8, device=device)
                kinds = {
                    "finalize_only": (mfr.FinalizePlan(T, H, k, R, enable_pdl=not args.no_pdl),
                                      lambda pl, j: pl.run(E[j], idx[j], w[j], out[j], stream, validate=False)),
                    "nvfp4_epilogue": (mfr.Nvfp4Plan(T, H, k, R, enable_pdl=not args.no_pdl),
                                       lambda pl, j: pl.run(E[j], idx[j], w[j], res[j], rout[j], g, base["eps"],
                                                            448.0 * 6.0 / 16.0, q[j], sf[j], stream,
                                                            validate=False)),
                    "expert_rmsnorm": (mfr.ExpertNormPlan(T, H, k, R, enable_pdl=not args.no_pdl),
                                       lambda pl, j: pl.run(E[j], idx[j], w[j], g, base["eps"], out[j], stream,
                                                            validate=False)),
                }
                for name, (pl, call) in kinds.items():
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph, stream=stream):
                        for i in range(ncalls):
                            call(pl, i % nsets)
                    graph.replay()
                    stream.synchronize()
                    times = []
                    for _ in range(5):
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        graph.replay()
                        b.record(stream)
                        b.synchronize()
                        times.append(a.elapsed_time(b) * 1e3 / ncalls)
                    del graph
                    if pl.get_status(stream) != 0:
                        raise RuntimeError(f"the device status word reported an error during {wl.name} {name}")
                    others[name] = round(float(np.median(times)), 3)
                del q, sf
        info = plan.info()
        target = 2 * (floor_us + nbytes / 8e12 * 1e6)
        rows.append({"workload": wl.name, "T": T, "H": H, "us_per_call": round(us, 3),
                     "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1), "floor_us": round(floor_us, 3),
                     "vs_2x_floor": round(us / target, 3), "variant": info["variant_name"],
                     "cluster": info["cluster"], "sets": nsets, "graph_calls": ncalls,
                     "warm_us": round(warm, 3), "loop_us": round(loop, 3), "loop_floor_us": round(loop_floor, 3),
                     "loop_vs_2x_floor": round(loop / (2 * (loop_floor + nbytes / 8e12 * 1e6)), 3),
                     **({"other_outputs_us": others} if others else {})})
        if plan.get_status(stream) != 0:
            raise RuntimeError(f"the device status word reported an error during {wl.name}")
        del E, idx, w, res, rout, out, base
        torch.cuda.empty_cache()
    return rows


def run_variants(mfr, device, wl, sets, args):
    """The other outputs of the library on the headline workload, timed
    like the main step (two alternating input sets, CUDA events):
    plain finalize (bf16 sum, no residual or norm: k*H*2 + H*2 + k*8 bytes
    per token), the NVFP4 epilogue (residual + RMSNorm, output as E2M1
    codes + E4M3 block scales: k*H*2 + H*8 + H/2 + H/16 + k*8 bytes), the
    same with the scales in the tiled layout of block-scaled GEMMs, and the
    finalize with an RMSNorm per expert row (k*H*2 + H*2 + k*8 bytes)."""
    T, H, k, R = wl.T, wl.H, wl.k, wl.R
    steps = max(20, min(args.steps, 500))
    stream = torch.cuda.Stream(device)
    out = {}
    fin = mfr.FinalizePlan(T, H, k, R, enable_pdl=not args.no_pdl)
    fp4 = mfr.Nvfp4Plan(T, H, k, R, enable_pdl=not args.no_pdl)
    fp4t = mfr.Nvfp4Plan(T, H, k, R, enable_pdl=not args.no_pdl, sf_layout=mfr.SF_TILED_128x4)
    en = mfr.ExpertNormPlan(T, H, k, R, enable_pdl=not args.no_pdl)
    q = [torch.empty((T, H // 2), dtype=torch.uint8, device=device) for _ in range(2)]
    sf = [torch.empty((T, H // 16), dtype=torch.uint8, device=device) for _ in range(2)]
    sft = [torch.empty((fp4t.sf_bytes(),), dtype=torch.uint8, device=device) for _ in range(2)]
    s_enc = 448.0 * 6.0 / 16.0

    def fin_step(i):
        d = sets[i & 1]
        fin.run(d["expert_out"], d["permuted_row_of"], d["topk_weights"], d["out"], stream, validate=False)

    def fp4_step(i):
        d = sets[i & 1]
        fp4.run(d["expert_out"], d["permuted_row_of"], d["topk_weights"], d["residual"], d["residual_out"],
                d["gamma"], d["eps"], s_enc, q[i & 1], sf[i & 1], stream, validate=False)

    def fp4t_step(i):
        d = sets[i & 1]
        fp4t.run(d["expert_out"], d["permuted_row_of"], d["topk_weights"], d["residual"], d["residual_out"],
                 d["gamma"], d["eps"], s_enc, q[i & 1], sft[i & 1], stream, validate=False)

    def en_step(i):
        d = sets[i & 1]
        en.run(d["expert_out"], d["permuted_row_of"], d["topk_weights"], d["gamma"], d["eps"], d["out"], stream,
               validate=False)

    plans = {"finalize_only": fin, "nvfp4_epilogue": fp4, "nvfp4_epilogue_tiled_scales": fp4t, "expert_rmsnorm": en}
    for name, fn, nbytes in (("finalize_only", fin_step, T * (k * H * 2 + H * 2 + k * 8)),
                             ("nvfp4_epilogue", fp4_step, T * (k * H * 2 + H * 8 + H // 2 + H // 16 + k * 8)),
                             ("nvfp4_epilogue_tiled_scales", fp4t_step,
                              T * (k * H * 2 + H * 8 + H // 2 + H // 16 + k * 8)),
                             ("expert_rmsnorm", en_step, T * (k * H * 2 + H * 2 + k * 8))):
        for i in range(5):
            fn(i)
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            fn(i)
        b.record(stream)
        b.synchronize()
        us = a.elapsed_time(b) * 1e3 / steps
        out[name] = {"us_per_call": round(us, 2), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "bytes_per_call": int(nbytes), "steps": steps,
                     "variant": plans[name].info()["variant_name"]}
    if fin.get_status(stream) or fp4.get_status(stream) or fp4t.get_status(stream) or en.get_status(stream):
        raise RuntimeError("status word set while timing the variants")
    return out


def run_pdl_pairs(mfr, device):
    """µs per (producer -> finalize) pair in a CUDA graph, both kernels with
    and without programmatic dependent launch.  The stand-in producer waits,
    signals its dependents, stays busy for `busy` cycles (a GEMM's main loop),
    then writes expert_out; with PDL the finalize's launch and prologue hide
    behind it.  Every pair uses the same buffers: the producer rewrites
    expert_out before each finalize, and the residual is the same tensor in
    every pair (for small T it stays in L2)."""
    rows = []
    for wl in (W.decode(1), W.decode(8), W.decode(128), W.PREFILL):
        base = W.make_inputs(wl, device)
        T, H, k, R = wl.T, wl.H, wl.k, wl.R
        src = base["expert_out"].clone()
        rout = torch.empty_like(base["residual"])
        out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        n = 64 if T <= 128 else 8
        for busy in (0, 10000):
            rec = {"workload": wl.name, "T": T, "busy_cycles": busy}
            for pdl in (False, True):
                plan = mfr.Plan(T, H, k, R, enable_pdl=pdl)
                stream = torch.cuda.Stream(device)
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    with torch.cuda.graph(graph, stream=stream):
                        for _ in range(n):
                            mfr.bench_producer(src, base["expert_out"], busy_cycles=busy, enable_pdl=pdl,
                                               stream=stream)
                            plan.run(base["expert_out"], base["permuted_row_of"], base["topk_weights"],
                                     base["residual"], rout, base["gamma"], base["eps"], out, stream,
                                     validate=False)
                    graph.replay()
                    stream.synchronize()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for _ in range(3):
                        graph.replay()
                    b.record(stream)
                    b.synchronize()
                if plan.get_status(stream) != 0:
                    raise RuntimeError("status word set during the PDL pairs")
                rec["us_per_pair_pdl" if pdl else "us_per_pair_serial"] = round(a.elapsed_time(b) * 1e3 / (3 * n), 3)
            rec["speedup"] = round(rec["us_per_pair_serial"] / rec["us_per_pair_pdl"], 4)
            rows.append(rec)
        del base, src, rout, out
        torch.cuda.empty_cache()
    return rows


# --- the reference arm: the CPU oracle ------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = W.by_name(args.workload)
    inp = W.make_inputs(wl, "cpu")
    host = host_copy(inp)
    cores = host_cores()
    # the whole run (warm-up + timed steps) stays within ~150 s of oracle work
    # for any --steps / --warmup: each step gets an equal share, at least 20 ms
    total_budget = 150.0
    per_step = max(0.02, min(args.cpu_seconds, total_budget / max(1, args.steps + args.warmup)))
    n_tokens = calibrate_tokens(host, wl.T, per_step, cores)
    for i in range(args.warmup):
        time_oracle(host, n_tokens, cores, 100 + i)
    times = []
    for i in range(args.steps):
        dt, n = time_oracle(host, n_tokens, cores, 1000 + i)
        times.append(dt)
    s = sum(times) / len(times)
    gbs = W.algorithmic_bytes(n_tokens, wl.H, wl.k) / s / 1e9
    sample = (f"{n_tokens} of {wl.T} tokens per step (seeded samples), H={wl.H}, k={wl.k}, "
              f"{s:.2f} s per step, {cores} host threads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {**workload_config(wl), "bytes_per_call": W.algorithmic_bytes(wl.T, wl.H, wl.k)},
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": cores, "kind": "oracle", "cpu": host_cpu(),
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        print("bench.py: --warmup must be >= 3", file=sys.stderr)
        return 2
    if args.floor_probe is not None:
        run_floor_probe(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        if not torch.cuda.is_available():
            print("bench.py: no CUDA device", file=sys.stderr)
            return 1
        run_ours(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
