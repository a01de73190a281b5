"""Benchmark of the GB300 allreduce schedule engine.

One step = one allreduce call (ar_execute) over P virtual-rank buffers already
resident in HBM.  The default workload is the large gradient-sync point:
ring schedule, fused single pass, order-faithful, P = 8 ranks x 256 MiB of
fp32 per rank, op = sum.  Buffers (2 GiB) are far larger than the 129 MB L2,
so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--P 8] [--mib 256] [--dtype float32] [--algo ring]
                    [--form fused] [--order faithful] [--sweep out.jsonl]

Prints ONE JSON line (rank 0).  value = allreduced bytes (P x S per call,
summed over all ranks' GPUs) per second, in GB/s.  Under torchrun each rank
runs the same per-GPU workload on its own GPU (no data-path collective; the
only collective is the timing max over ranks).

--impl reference times the CPU oracle (the plain simulation that defines
the schedules' results) on a bounded sample of the same workload, on the
host cores, and prints the same line with "impl": "reference".
"""

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

NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
METRIC = "allreduced bytes/s (P x S per call)"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
# the kernel code and the lowering that fixes its launch shape (tiles, stages, stores)
KERNEL_SRC = [os.path.join(ROOT, "collective_reduction_gb300", "csrc", f)
              for f in ("kernels.cu", "device.cuh", "devprog.hpp", "lower.cpp", "lower.hpp")]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--P", type=int, default=8)
    ap.add_argument("--mib", type=float, default=256.0, help="MiB per rank")
    ap.add_argument("--dtype", default="float32", choices=["float32", "bfloat16", "int32"])
    ap.add_argument("--op", default="sum")
    ap.add_argument("--algo", default="ring")
    ap.add_argument("--form", default="fused")
    ap.add_argument("--order", default="faithful")
    ap.add_argument("--r", type=int, default=0)
    ap.add_argument("--k1", type=int, default=0)
    ap.add_argument("--phase", default="allreduce", choices=["allreduce", "reduce_scatter", "all_gather"],
                    help="the whole allreduce, or one half (ring, rh, generalized r = 0)")
    ap.add_argument("--jit", default="auto", choices=["auto", "on", "off"],
                    help="DAG programs as run-time compiled code (auto / on) or interpreted (off)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--offset", type=int, default=0,
                    help="place every rank buffer this many elements past a 256-byte boundary "
                         "(not a multiple of 16 bytes: the element-wise path)")
    ap.add_argument("--no-floor", action="store_true",
                    help="skip the config5_floor points timed after the headline")
    ap.add_argument("--sweep", default=None, help="write the size sweep as JSON lines to this file")
    ap.add_argument("--sweep-ps", default="2,8,16,64", help="rank counts of the size sweep (comma-separated)")
    ap.add_argument("--rows", default=None,
                    help="time every schedule at the bench size (fused and step), JSON lines to this file")
    ap.add_argument("--costmodel", default=None,
                    help="fit the step-form cost model and validate its step choice, JSON lines to this file")
    ap.add_argument("--configs", default=None,
                    help="time every schedule of the parity configurations, JSON lines to this file")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def esize(dtype):
    return 2 if dtype == "bfloat16" else 4


def workload_name(a):
    return (f"{a.algo} allreduce, {a.form} {a.order}, P={a.P} x {a.mib:g} MiB {a.dtype} per rank, "
            f"op={a.op}" + (f", r={a.r}" if a.algo == "generalized" else "")
            + (f", buffers offset by {a.offset} elements" if getattr(a, "offset", 0) else "")
            + (f", k1={a.k1}" if a.algo == "hybrid" else "")
            + (f", phase={a.phase}" if a.phase != "allreduce" else ""))


def dtype_tag(dtype):
    return {"float32": "f32", "bfloat16": "bf16", "int32": "int32"}[dtype]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash():
    """Hash of the kernel source with comments and blank lines removed, so a
    recorded ncu traffic figure stays valid across comment-only edits and is
    dropped as soon as the code changes."""
    import re
    src = ""
    for path in KERNEL_SRC:
        with open(path) as f:
            src += f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lines = [ln.split("//", 1)[0].rstrip() for ln in src.splitlines()]
    code = "\n".join(ln for ln in lines if ln.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def bulk_kernel_name(bits):
    """The kernel that runs a plan's aligned bulk items, from ar_plan_info.kernels."""
    for bit, name in ((16, "ar_word_kernel"), (32, "chain_word_kernel"), (64, "copy_kernel"), (128, "few_kernel"),
                      (1, "stream_kernel"), (8, "ar_dag_kernel"), (2, "staged_kernel")):
        if bits & bit:
            return name
    return "elementwise_kernel"


def recorded_traffic(P, mib, dtype, algo, form, order):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    summary is missing, is for another workload, or predates the kernel."""
    try:
        rec = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("kernel_sha256_16") != kernel_hash():
            return None
        key = f"P={P} mib={mib:g} dtype={dtype} algo={algo} form={form} order={order}"
        if rec.get("workload") != key:
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in self.rows:
            try:
                sm.append(float(row[0]))
                mx = float(row[1])
                for nm, v in zip(names, row[4:8]):
                    if v.strip().lower() == "active":
                        reasons.add(nm)
            except Exception:
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier_sync(world):
    import torch
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        torch.cuda.synchronize()


def max_over_ranks(x, world):
    """Largest value of x over all ranks (timing only; never on the data path)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(bytes_per_call, calls, world, max_ms):
    """Whole-job throughput: every rank's allreduced bytes over the slowest
    rank's timed region."""
    return bytes_per_call * calls * world / (max_ms / 1e3) / 1e9


def busbw_gbps(S, seconds, P):
    """Bus bandwidth of an allreduce of S bytes per rank over P ranks:
    algbw x 2(P-1)/P ("All-Reduce, in depth", Reading benchmarks)."""
    return S / seconds * 2 * (P - 1) / P / 1e9


def gather_sample(dev, P, n, K, chunks):
    """K elements from each of the schedule's `chunks` base chunks of every rank
    buffer, laid out so a ceil split of the sample into `chunks` parts puts
    each chunk's elements into the same part."""
    import numpy as np
    import torch
    size = -(-n // chunks)
    idx = []
    for c in range(chunks):
        lo, hi = min(n, c * size), min(n, (c + 1) * size)
        if hi - lo < K:
            raise ValueError("chunk shorter than the sample")
        idx.extend(np.linspace(lo, hi - 1, K).astype(np.int64).tolist())
    it = torch.tensor(idx, dtype=torch.int64, device="cuda")
    out = []
    for t in dev:
        s = t.index_select(0, it)
        if t.dtype == torch.bfloat16:
            out.append(s.view(torch.int16).cpu().numpy().view(np.uint16))
        else:
            out.append(s.cpu().numpy())
    return out, it


def base_chunks(a):
    if a.algo == "ahc":
        raise ValueError("the bench's sampled check covers ring / generalized / binomial / rd / rh")
    return a.P


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def oracle_repeat(job):
    """Pool worker: the oracle on one sample, repeated for `seconds` (at least
    once); returns (runs, seconds)."""
    algo, kw, op, dtype, sample, seconds = job
    import oracle
    from oracle.elementops import Arith
    t0 = time.perf_counter()
    runs = 0
    while True:
        oracle.run(algo, sample, Arith(op, dtype), **kw)
        runs += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return runs, time.perf_counter() - t0


def split_sample(sample, P, parts):
    """The per-chunk blocks of a gathered sample cut into `parts` samples,
    each keeping the chunk structure (a ceil split gives the same P chunks)."""
    import numpy as np
    K = sample[0].size // P // parts
    out = []
    for j in range(parts):
        out.append([np.ascontiguousarray(np.concatenate(
            [b[c * K * parts + j * K: c * K * parts + (j + 1) * K] for c in range(P)])) for b in sample])
    return out


def oracle_kw(a):
    kw = {"r": a.r} if a.algo == "generalized" else ({"k1": a.k1} if a.algo == "hybrid" else {})
    if a.phase != "allreduce":
        kw["phase"] = a.phase
    return kw


def cpu_baseline_and_check(a, sample_in, sample_out_engine, parts, timed=True):
    """The oracle, as it stands, timed on the host cores on a bounded sample
    of the workload: one sample per core, each in its own process (spawned),
    for half the time budget, after a single-process run on the first sample
    for the other half that also checks the engine's output there.  With
    timed=False only the check runs (one oracle run) and no baseline is
    returned."""
    import multiprocessing as mp

    import numpy as np
    subs = split_sample(sample_in, a.P, parts)
    outs = split_sample(sample_out_engine, a.P, parts) if sample_out_engine is not None else None
    kw = oracle_kw(a)
    import oracle
    from oracle.elementops import Arith
    res = oracle.run(a.algo, subs[0], Arith(a.op, a.dtype), **kw)
    ok = None
    if outs is not None and a.order == "faithful":
        def bits(x):
            x = np.ascontiguousarray(x)
            return x if x.dtype == np.uint16 else x.view(np.uint32)
        if a.phase == "reduce_scatter":
            # only the owners' chunks are defined after a reduce-scatter
            ok = all(np.array_equal(bits(res.bufs[r][lo:hi]), bits(outs[0][r][lo:hi]))
                     for r, lo, hi in res.info["owner"])
        else:
            ok = all(np.array_equal(bits(res.bufs[r]), bits(outs[0][r])) for r in range(a.P))
    if not timed:
        return None, ok
    half = a.cpu_seconds / 2
    nbytes = a.P * subs[0][0].size * esize(a.dtype)
    runs1, dt1 = oracle_repeat((a.algo, kw, a.op, a.dtype, subs[0], half))
    with mp.get_context("spawn").Pool(parts) as pool:
        done = pool.map(oracle_repeat, [(a.algo, kw, a.op, a.dtype, sub, half) for sub in subs])
    runs = sum(r for r, _ in done)
    wall = max(t for _, t in done)
    return {"value": nbytes * runs / wall / 1e9, "unit": "GB/s", "cores": parts, "kind": "oracle",
            "single_thread_value": nbytes * runs1 / dt1 / 1e9, "cpu_model": cpu_model(),
            "sample": f"{parts} samples of {subs[0][0].size} elements per rank ({subs[0][0].size // a.P} from "
                      f"each of the {a.P} chunks of the benchmark buffers), one per core in its own process: "
                      f"{runs} oracle runs in {wall:.1f} s (single process: {runs1} runs in {dt1:.1f} s)"}, ok


# The weakest points of the large-size target (the fused kernel at >= 64 MB per
# rank): the ring over the sweep's largest P and size, both dtypes, both orders.
FLOOR_POINTS = [(64, 256, "float32", "faithful"), (64, 256, "float32", "fp32acc"),
                (64, 256, "bfloat16", "faithful"), (64, 256, "bfloat16", "fp32acc")]


def config5_floor(stream, peak, steps=20, warmup=3):
    """Times each FLOOR_POINTS plan (fused ring) back to back with CUDA events
    on the launching stream, after checking it against the oracle on 512
    sampled elements of every chunk (bit for bit; fp32-accumulated within
    tolerance).  One dict per point."""
    import numpy as np
    import torch

    import ar_synth
    import collective_reduction_gb300 as ar
    import oracle
    from oracle.direct import direct_f64, normwise_rel_err
    from oracle.elementops import Arith, bf16_to_f32
    mods = (oracle, Arith, direct_f64, normwise_rel_err, bf16_to_f32)
    out = []
    for P, mib, dtype, order in FLOOR_POINTS:
        n = (mib << 20) // esize(dtype)
        if P * n * esize(dtype) * 1.1 > torch.cuda.mem_get_info()[0]:
            out.append({"P": P, "bytes_per_rank": mib << 20, "dtype": dtype, "order": order, "skipped": "memory"})
            continue
        dev = ar_synth.device_inputs(P, n, dtype, sigma=1e-3, seed=P)
        plan = ar.Plan(P, n, dtype, "sum", "ring", order=order)
        info = plan.info()
        sample_in, idx = gather_sample(dev, P, n, 512, P)
        plan.execute(dev, stream)
        plan.check()
        got = [t.index_select(0, idx) for t in dev]
        got = [g.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bfloat16" else g.cpu().numpy()
               for g in got]
        if order == "fp32acc":
            ref = direct_f64(sample_in, "sum", dtype)
            err = max(normwise_rel_err(bf16_to_f32(g) if dtype == "bfloat16" else g, ref) for g in got)
            ok = bool(err <= (1e-6 if dtype == "float32" else 4e-3))
        else:
            want = oracle.run("ring", sample_in, Arith("sum", dtype)).bufs
            ok = all(np.array_equal(np.ascontiguousarray(g).view(np.uint8), np.ascontiguousarray(w).view(np.uint8))
                     for g, w in zip(got, want))
        for _ in range(warmup):
            plan.execute(dev, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            plan.execute(dev, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        plan.check()
        ms = e0.elapsed_time(e1) / steps
        gbps = info["hbm_bytes"] / (ms / 1e3) / 1e9
        out.append({"P": P, "bytes_per_rank": mib << 20, "dtype": dtype, "form": "fused", "order": order,
                    "steps": steps, "ms_per_step": round(ms, 4), "allreduced_GBps": round(P * n * esize(dtype) / ms / 1e6, 1),
                    "achieved_hbm_GBps": round(gbps, 1), "frac": round(gbps / peak, 4),
                    "frac_of_nominal_7900": round(gbps / NOMINAL_HBM_GBS, 4),
                    "verified_sample_vs_oracle": ok})
        plan.close()
        del dev
        torch.cuda.empty_cache()
    return out


def run_ours(a):
    import numpy as np
    import torch

    import ar_synth
    import collective_reduction_gb300 as ar

    world, rank, local = dist_setup()
    es = esize(a.dtype)
    n = int(a.mib * (1 << 20)) // es
    S = n * es
    params = dict(form=a.form, order=a.order, jit=a.jit)
    if a.phase != "allreduce":
        params["phase"] = a.phase
    if a.algo == "generalized":
        params["r"] = a.r
    if a.algo == "hybrid":
        params["k1"] = a.k1
    if a.dtype == "int32":
        dev = [torch.randint(-1000, 1001, (n,), dtype=torch.int32, device="cuda",
                             generator=torch.Generator("cuda").manual_seed(r)) for r in range(a.P)]
    else:
        dev = ar_synth.device_inputs(a.P, n, a.dtype, sigma=1e-3, seed=rank)
    if a.offset:
        shifted = []
        for t in dev:
            big = torch.empty(n + a.offset, dtype=t.dtype, device="cuda")
            big[a.offset:].copy_(t)
            shifted.append(big[a.offset:])
        dev = shifted
    plan = ar.Plan(a.P, n, a.dtype, a.op, a.algo, **params)
    info = plan.info()
    stream = torch.cuda.current_stream()

    # sampled check + CPU baseline (rank 0 only): sample before the first call
    parts = host_cores() if rank == 0 else 1
    sample_k = 1 << 17 if a.dtype != "bfloat16" else 1 << 18
    sample_k = max(1, min(sample_k // a.P, n // a.P // parts))
    sample_in, idx = (None, None)
    if rank == 0:
        sample_in, idx = gather_sample(dev, a.P, n, sample_k * parts, base_chunks(a))
    plan.execute(dev, stream)
    plan.check()
    sample_out = None
    if rank == 0:
        sample_out = []
        for t in dev:
            s = t.index_select(0, idx)
            sample_out.append(s.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16
                              else s.cpu().numpy())

    for _ in range(a.warmup):
        plan.execute(dev, stream)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier_sync(world)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # back-to-back calls with no event between them (an event between two
    # launches would stop the second from starting while the first drains)
    t_start.record(stream)
    for i in range(a.steps):
        plan.execute(dev, stream)
    t_end.record(stream)
    barrier_sync(world)
    clk = clocks.stop()
    plan.check()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world)
    # the kernels' average duration per step, from the same CUDA events
    # (on the launching stream) over the timed region: every launch of the
    # region is this plan's
    kernel_ms = total_ms / a.steps

    bytes_per_call = a.P * S
    value = whole_job_gbps(bytes_per_call, a.steps, world, total_ms)
    peak, peak_kind = measured_peak()
    alg_bytes = info["hbm_bytes"]
    achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
    traffic = recorded_traffic(a.P, a.mib, a.dtype, a.algo, a.form, a.order)

    # end to end through the C ABI with pinned host buffers
    host = [torch.empty(n, dtype=dev[0].dtype).pin_memory() for _ in range(a.P)]
    for h, d in zip(host, dev):
        h.copy_(d)
    plan.execute_host(host, dev, stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(a.e2e_steps):
        plan.execute_host(host, dev, stream)
    e2e_s = (time.perf_counter() - t0) / a.e2e_steps
    e2e_s = max_over_ranks(e2e_s, world)
    plan.check()

    # the weakest large-size points, timed after the headline's region with
    # its buffers released
    floor = None
    if not a.no_floor:
        del host
        plan.close()
        del dev
        torch.cuda.empty_cache()
        floor = config5_floor(stream, peak)

    # the CPU baseline is timed at N = 1 only (with N ranks on one host the
    # host cores are shared); rank 0 still checks its sample against the oracle
    cpu, verified = (None, None)
    if rank == 0:
        cpu, verified = cpu_baseline_and_check(a, sample_in, sample_out, parts, timed=world == 1)

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": round(total_ms / a.steps, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_tag(a.dtype),
        "data": "synthetic",
        "config": {"workload": workload_name(a), "P": a.P, "bytes_per_rank": S, "elements_per_rank": n,
                   "algo": a.algo, "form": a.form, "order": a.order, "op": a.op, "phase": a.phase,
                   "l2": "inputs larger than L2 (P x S = %.1f GiB vs 129 MB)" % (a.P * S / 2 ** 30),
                   "busbw_GBps": round(busbw_gbps(S, total_ms / a.steps / 1e3, a.P), 2),
                   "algbw_GBps": round(S / (total_ms / a.steps / 1e3) / 1e9, 2),
                   "parallelism": f"replicas{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal_7900": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": alg_bytes,
                     "kernel_ms": round(kernel_ms, 6),
                     "kernel": bulk_kernel_name(info["kernels"])},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_gbps(bytes_per_call, 1, world, e2e_s * 1e3), 3), "unit": "GB/s",
                "h2d_bytes_per_step": bytes_per_call, "d2h_bytes_per_step": bytes_per_call},
        "clocks": clk,
        "gpu_launches": info["launches"] * a.steps,
        "verified_sample_vs_oracle": verified,
    }
    if floor is not None:
        line["config5_floor"] = floor
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------ reference arm

_REF_BUFS = None


def _reference_init(P, n, dtype, dist):
    """Pool worker start-up: this worker's own seeded sample of the workload."""
    global _REF_BUFS
    import ar_synth
    _REF_BUFS = ar_synth.rank_inputs(P, n, dtype, dist, sigma=1e-3, seed=os.getpid())


def _reference_step(job):
    algo, kw, op, dtype = job
    import oracle
    from oracle.elementops import Arith
    oracle.run(algo, _REF_BUFS, Arith(op, dtype), **kw)
    return True


def run_reference(a):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import multiprocessing as mp
    # bounded sample of the workload: up to 2^20 elements per rank per core
    # (chunk structure kept: a ceil split of the sample gives the same P
    # chunks), one sample per core, each in its own (spawned) process; a step
    # is one oracle run on every core's sample
    cores = host_cores()
    n = max(a.P, min(int(a.mib * (1 << 20)) // esize(a.dtype), 1 << 20) // a.P * a.P)
    dist = "uniform_int" if a.dtype == "int32" else "normal"
    job = (a.algo, oracle_kw(a), a.op, a.dtype)
    with mp.get_context("spawn").Pool(cores, initializer=_reference_init, initargs=(a.P, n, a.dtype, dist)) as pool:
        for _ in range(a.warmup):
            pool.map(_reference_step, [job] * cores, chunksize=1)
        times = []
        for _ in range(a.steps):
            t0 = time.perf_counter()
            pool.map(_reference_step, [job] * cores, chunksize=1)
            times.append(time.perf_counter() - t0)
    total = sum(times)
    nbytes = a.P * n * esize(a.dtype) * cores
    value = nbytes * a.steps / total / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(total / a.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_tag(a.dtype), "data": "synthetic",
        "config": {"workload": workload_name(a), "P": a.P, "bytes_per_rank": int(a.mib * (1 << 20)),
                   "algo": a.algo, "form": a.form, "order": a.order, "op": a.op, "phase": a.phase,
                   "sample_elements_per_rank": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{cores} samples (one per core, each in its own process) of {n} elements "
                                   f"per rank (of {int(a.mib * (1 << 20)) // esize(a.dtype)}); a step is one "
                                   f"oracle run on every sample"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- sweep

def sweep_check(ar, oracle_mods, plan, dev, P, n, dtype, order):
    """Runs the plan once on dev and checks the result against the oracle:
    every element when P x n <= 2^24, else 2^12 elements sampled from each of
    the P chunks (bit for bit; fp32-accumulated within tolerance)."""
    import numpy as np
    import torch
    oracle, Arith, direct_f64, normwise_rel_err, bf16_to_f32 = oracle_mods
    full = P * n <= (1 << 24)
    K = n // P if full else min(1 << 12, n // P)
    if full:
        idx = None
        sample_in = [t.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bfloat16" else t.cpu().numpy()
                     for t in dev]
    else:
        sample_in, idx = gather_sample(dev, P, n, K, P)
    plan.execute(dev)
    plan.check()
    got = [t if idx is None else t.index_select(0, idx) for t in dev]
    got = [g.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bfloat16" else g.cpu().numpy() for g in got]
    if order == "fp32acc":
        ref = direct_f64(sample_in, "sum", dtype)
        err = max(normwise_rel_err(bf16_to_f32(g) if dtype == "bfloat16" else g, ref) for g in got)
        return bool(err <= (1e-6 if dtype == "float32" else 4e-3)), full, None
    t0 = time.perf_counter()
    want = oracle.run("ring", sample_in, Arith("sum", dtype)).bufs
    oracle_s = time.perf_counter() - t0

    def bits(x):
        x = np.ascontiguousarray(x)
        return x if x.dtype == np.uint16 else x.view(np.uint32)
    return all(np.array_equal(bits(g), bits(w)) for g, w in zip(got, want)), full, oracle_s


def run_sweep(a, path):
    """Configuration 5: ring fused (faithful, fp32acc) and ring step form over
    P in {2, 8, 16, 64} and 1 KiB .. 256 MiB per rank, fp32 and bf16; one
    JSON line per point.  Every point is first checked against the oracle
    (sweep_check).  Points up to 64 KiB are timed as a CUDA graph of 100
    calls."""
    import torch

    import ar_synth
    import collective_reduction_gb300 as ar
    import oracle
    from oracle.direct import direct_f64, normwise_rel_err
    from oracle.elementops import Arith, bf16_to_f32
    oracle_mods = (oracle, Arith, direct_f64, normwise_rel_err, bf16_to_f32)
    torch.cuda.set_device(0)
    free = torch.cuda.mem_get_info()[0]
    peak, _ = measured_peak()
    with open(path, "w") as out:
        for dtype in ("float32", "bfloat16"):
            for P in [int(p) for p in a.sweep_ps.split(",")]:
                for lg in range(10, 29):
                    S = 1 << lg
                    if P * S * 1.2 > free:
                        continue
                    n = S // esize(dtype)
                    dev = ar_synth.device_inputs(P, n, dtype, sigma=1e-3, seed=P)
                    for form, order in (("fused", "faithful"), ("fused", "fp32acc"), ("step", "faithful")):
                        plan = ar.Plan(P, n, dtype, "sum", "ring", form=form, order=order)
                        info = plan.info()
                        fresh = ar_synth.device_inputs(P, n, dtype, sigma=1e-3, seed=P + 1)
                        ok, full, oracle_s = sweep_check(ar, oracle_mods, plan, fresh, P, n, dtype, order)
                        del fresh
                        for _ in range(5):  # 5 warm-up calls
                            plan.execute(dev)
                        torch.cuda.synchronize()
                        if S <= 65536:
                            g = torch.cuda.CUDAGraph()
                            s = torch.cuda.Stream()
                            s.wait_stream(torch.cuda.current_stream())
                            with torch.cuda.stream(s):
                                with torch.cuda.graph(g, stream=s):
                                    for _ in range(100):
                                        plan.execute(dev)
                            torch.cuda.synchronize()
                            reps = []
                            for _ in range(5):
                                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                                e0.record()
                                g.replay()
                                e1.record()
                                torch.cuda.synchronize()
                                reps.append(e0.elapsed_time(e1) / 100)
                            ms = statistics.median(reps)
                            del g
                        else:
                            reps = []
                            for _ in range(5):
                                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                                e0.record()
                                for _ in range(10):
                                    plan.execute(dev)
                                e1.record()
                                torch.cuda.synchronize()
                                reps.append(e0.elapsed_time(e1) / 10)
                            ms = statistics.median(reps)
                        plan.check()
                        row = {"dtype": dtype, "P": P, "bytes_per_rank": S, "form": form, "order": order,
                               "ms": ms, "allreduced_GBps": P * S / (ms / 1e3) / 1e9,
                               "busbw_GBps": S / (ms / 1e3) * 2 * (P - 1) / P / 1e9,
                               "hbm_GBps": info["hbm_bytes"] / (ms / 1e3) / 1e9,
                               "frac_of_measured": info["hbm_bytes"] / (ms / 1e3) / 1e9 / peak,
                               "launches": info["launches"], "verified": ok,
                               "checked": "every element" if full else "2^12 sampled elements per chunk"}
                        if full and oracle_s:  # the oracle timed on the whole point (NumPy, one process)
                            row["oracle_GBps"] = P * S / oracle_s / 1e9
                        out.write(json.dumps(row) + "\n")
                        out.flush()
                        plan.close()
                    del dev
                    torch.cuda.empty_cache()


def config_cases():
    """The schedules of the four parity configurations, each in every form,
    then the widened ones: RD / RH / hybrid on a non-power-of-two P through
    the preparation and finalization rounds, the pipelined chain, and the
    reduce-scatter and all-gather halves on their own."""
    cases = []
    for form in ("fused", "step"):
        cases.append(("config1", 3, 1024, "int32", "sum", "ring", {"form": form}, ("uniform_int", 1.0)))
    for op in ("sum", "max"):
        for algo, kw in [("rh", {}), ("rd", {}), ("binomial", {})] + [("hybrid", {"k1": k}) for k in range(4)]:
            for form in ("fused", "step"):
                cases.append(("config2", 8, 1 << 20, "float32", op, algo, dict(kw, form=form), ("normal", 1.0)))
    for P in (7, 12):
        L = (P - 1).bit_length()
        for n in (106, 1 << 20):
            for r in range(L + 1):
                for form in ("fused", "step"):
                    cases.append(("config3", P, n, "float32", "sum", "generalized", {"r": r, "form": form},
                                  ("normal", 1e-2)))
    for kw in ({"form": "fused"}, {"form": "fused", "order": "fp32acc"}, {"form": "step"}):
        cases.append(("config4", 5, 1 << 24, "bfloat16", "sum", "ahc", dict(kw, group_sizes=[2, 3]),
                      ("normal", 1e-3)))
    for algo, kw in (("rd", {}), ("rh", {}), ("hybrid", {"k1": 1})):
        for form in ("fused", "step"):
            cases.append(("fold_p12", 12, 1 << 20, "float32", "sum", algo, dict(kw, form=form), ("normal", 1.0)))
    for m in (1, 16):
        for form in ("fused", "step"):
            cases.append(("pipeline_p8", 8, 1 << 20, "bfloat16", "sum", "pipeline", {"blocks": m, "form": form},
                          ("normal", 1e-2)))
    for phase in ("reduce_scatter", "all_gather"):
        for algo, kw in (("ring", {}), ("rh", {}), ("generalized", {})):
            for form in ("fused", "step"):
                cases.append(("halves_p8", 8, 1 << 24, "float32", "sum", algo, dict(kw, form=form, phase=phase),
                              ("normal", 1.0)))
    return cases


def run_configs(a, path):
    """Times every schedule of configurations 1-4 on the GPU (10 back-to-back
    calls, median of 5 CUDA-event measurements, launch overhead included) and
    the oracle on the same inputs on the host, and checks the GPU result
    against the oracle's bit for bit (fp32-accumulate: within tolerance)."""
    import numpy as np
    import torch

    import ar_synth
    import collective_reduction_gb300 as ar
    import oracle
    from oracle.direct import direct_f64, normwise_rel_err
    from oracle.elementops import Arith, bf16_to_f32
    torch.cuda.set_device(0)
    peak, _ = measured_peak()
    inputs = {}
    with open(path, "w") as out:
        for cfg, P, n, dtype, op, algo, kw, (dist, sigma) in config_cases():
            key = (P, n, dtype, dist, sigma)
            if key not in inputs:
                inputs = {key: ar_synth.rank_inputs(P, n, dtype, dist, sigma=sigma)}
            host = inputs[key]
            tdt = {"int32": torch.int32, "float32": torch.float32, "bfloat16": torch.int16}[dtype]
            dev0 = [torch.from_numpy(h.view(np.int16) if dtype == "bfloat16" else h).to("cuda") for h in host]
            dev = [t.clone() for t in dev0]
            if dtype == "bfloat16":
                dev = [t.view(torch.bfloat16) for t in dev]
            plan = ar.Plan(P, n, dtype, op, algo, **kw)
            info = plan.info()
            plan.execute(dev)
            torch.cuda.synchronize()
            plan.check()
            got = [t.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bfloat16" else t.cpu().numpy()
                   for t in dev]
            okw = {k: v for k, v in kw.items() if k in ("r", "k1", "group_sizes", "blocks", "phase")}
            t0 = time.perf_counter()
            want = oracle.run(algo, host, Arith(op, dtype), **okw)
            oracle_s = time.perf_counter() - t0
            if kw.get("order") == "fp32acc":
                ref = direct_f64(host, op, dtype)
                err = max(normwise_rel_err(bf16_to_f32(g) if dtype == "bfloat16" else g, ref) for g in got)
                ok = err <= (1e-6 if dtype == "float32" else 4e-3)
            else:
                def bits(x):
                    x = np.ascontiguousarray(x)
                    return x if x.dtype == np.uint16 else x.view(np.uint32)
                if kw.get("phase") == "reduce_scatter":
                    # only the owners' chunks are defined after a reduce-scatter
                    ok = all(np.array_equal(bits(got[r][lo:hi]), bits(want.bufs[r][lo:hi]))
                             for r, lo, hi in want.info["owner"])
                else:
                    ok = all(np.array_equal(bits(g), bits(w)) for g, w in zip(got, want.bufs))
            for _ in range(3):
                plan.execute(dev)
            torch.cuda.synchronize()
            ts = []
            for _ in range(5):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(10):
                    plan.execute(dev)
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / 10)
            plan.check()
            ms = statistics.median(ts)
            S = n * esize(dtype)
            row = {"config": cfg, "P": P, "n": n, "dtype": dtype, "op": op, "algo": algo,
                   "params": {k: v for k, v in kw.items()}, "verified": bool(ok),
                   "steps": info["steps"], "launches": info["launches"], "us_per_call": round(ms * 1e3, 2),
                   "allreduced_GBps": round(P * S / (ms / 1e3) / 1e9, 2),
                   "hbm_bytes_per_call": info["hbm_bytes"],
                   "hbm_GBps": round(info["hbm_bytes"] / (ms / 1e3) / 1e9, 1),
                   "frac_of_measured": round(info["hbm_bytes"] / (ms / 1e3) / 1e9 / peak, 4),
                   "oracle_s": round(oracle_s, 4),
                   "oracle_GBps": round(P * S / oracle_s / 1e9, 4)}
            out.write(json.dumps(row) + "\n")
            out.flush()
            plan.close()


def time_plan(plan, dev, reps=5, calls=20):
    """Median over reps of the mean CUDA-event time of `calls` back-to-back
    executes (after 5 warm-up calls), in microseconds."""
    import torch
    for _ in range(5):
        plan.execute(dev)
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(calls):
            plan.execute(dev)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / calls)
    plan.check()
    return statistics.median(ts)


def row_cases():
    """(row, P, op, algo, params, sample chunks): every schedule at P = 8,
    then rank-specific DAG programs (the generalized schedule with removed
    steps at P = 7, recursive doubling for max)."""
    out = []
    for algo, kw, chunks, row in (("ring", {}, 8, "a3/a4 ring RS+AG"),
                                  ("binomial", {}, 1, "a5/a6 binomial reduce+broadcast"),
                                  ("rh", {}, 8, "a7 RH"), ("rd", {}, 1, "a8 RD"),
                                  ("generalized", {"r": 0}, 8, "a9/a10 generalized r=0"),
                                  ("generalized", {"r": 1}, 8, "a9/a10 generalized r=1"),
                                  ("generalized", {"r": 3}, 8, "a9 generalized r=L"),
                                  ("hybrid", {"k1": 1}, 8, "a11 hybrid k1=1"),
                                  ("ahc", {"group_sizes": [4, 4]}, 8, "a12-a14 AHC {4,4}"),
                                  ("pipeline", {"blocks": 4}, 4, "f4 pipelined chain m=4")):
        for form in ("fused", "step"):
            out.append((row, 8, "sum", algo, dict(kw, form=form), chunks))
    for algo in ("ring", "rh"):
        for phase in ("reduce_scatter", "all_gather"):
            out.append((f"f2 {phase}", 8, "sum", algo, {"form": "fused", "phase": phase}, 8))
    out.append(("a15 fp32acc", 8, "sum", "ring", {"form": "fused", "order": "fp32acc"}, 8))
    out.append(("a15 fp32acc", 8, "sum", "ahc", {"form": "fused", "order": "fp32acc", "group_sizes": [4, 4]}, 8))
    for r in (1, 3):
        for form in ("fused", "step"):
            out.append((f"a9 generalized P=7 r={r}", 7, "sum", "generalized", {"r": r, "form": form}, 7))
    out.append(("a8 RD max (rank-specific)", 8, "max", "rd", {"form": "fused"}, 1))
    return out


def run_rows(a, path):
    """Every schedule of the hot path at the bench size, P = 8 x 256 MiB per
    rank (fp32 and bf16, sum): median of 5 CUDA-event timings of 10
    back-to-back calls, HBM GB/s from the plan's algorithmic bytes, the
    fraction of the measured copy peak, and the oracle's verdict on a sample
    of the result (2^14 elements from each base chunk, bit for bit;
    fp32-accumulated results within the normwise tolerance)."""
    import numpy as np
    import torch

    import ar_synth
    import collective_reduction_gb300 as ar
    import oracle
    from oracle.direct import direct_f64, normwise_rel_err
    from oracle.elementops import Arith, bf16_to_f32
    torch.cuda.set_device(0)
    peak, _ = measured_peak()
    K = 1 << 14

    def bits(x):
        x = np.ascontiguousarray(x)
        return x if x.dtype == np.uint16 else x.view(np.uint32)

    with open(path, "w") as out:
        for dtype in ("float32", "bfloat16"):
            n = (256 << 20) // esize(dtype)
            src = ar_synth.device_inputs(8, n, dtype, sigma=1e-2, seed=3)
            for row, P, op, algo, kw, chunks in row_cases():
                dev = [t.clone() for t in src[:P]]
                sample_in, idx = gather_sample(dev, P, n, K, chunks)
                plan = ar.Plan(P, n, dtype, op, algo, **kw)
                info = plan.info()
                plan.execute(dev)
                plan.check()
                got = [t.index_select(0, idx) for t in dev]
                got = [g.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bfloat16" else g.cpu().numpy()
                       for g in got]
                okw = {k: v for k, v in kw.items() if k in ("r", "k1", "group_sizes", "blocks", "phase")}
                if kw.get("order") == "fp32acc":
                    ref = direct_f64(sample_in, op, dtype)
                    err = max(normwise_rel_err(bf16_to_f32(g) if dtype == "bfloat16" else g, ref) for g in got)
                    ok = err <= (1e-6 if dtype == "float32" else 4e-3)
                else:
                    want = oracle.run(algo, sample_in, Arith(op, dtype), **okw)
                    if kw.get("phase") == "reduce_scatter":
                        ok = all(np.array_equal(bits(got[r][lo:hi]), bits(want.bufs[r][lo:hi]))
                                 for r, lo, hi in want.info["owner"])
                    else:
                        ok = all(np.array_equal(bits(g), bits(w)) for g, w in zip(got, want.bufs))
                us = time_plan(plan, dev, reps=5, calls=10)
                gbps = info["hbm_bytes"] / (us / 1e6) / 1e9
                out.write(json.dumps({
                    "row": row, "algo": algo, "op": op, "params": kw, "dtype": dtype, "P": P,
                    "bytes_per_rank": n * esize(dtype),
                    "verified": bool(ok), "steps": info["steps"], "launches": info["launches"],
                    "kernels": info["kernels"], "us_per_call": round(us, 2), "hbm_bytes": info["hbm_bytes"],
                    "hbm_GBps": round(gbps, 1), "frac_of_measured": round(gbps / peak, 4),
                    "allreduced_GBps": round(P * n * esize(dtype) / (us / 1e6) / 1e9, 1)}) + "\n")
                out.flush()
                plan.close()
                del dev
            del src
            torch.cuda.empty_cache()


def run_costmodel(a, path):
    """The step-form cost model ("A Generalization of the Allreduce
    Operation", eqs. 36-37) on this GPU.  Fit: alpha per round, beta per byte
    sent, gamma per byte combined (bytes over all ranks) and delta per
    message by non-negative least squares on relative error, over step-form
    ring, binomial, RD, the bandwidth-optimal and the latency-optimal
    generalized plans (the latter's rounds are many small messages) and the
    ring's reduce-scatter (combines) and all-gather (copies) halves, which
    tell beta and gamma apart, at P in {4, 16, 63} and 2 KiB .. 64 MiB per
    rank.  Validation: at P in {7, 12, 31, 63} and 1 KiB .. 16 MiB per
    rank, every candidate the selection weighs is timed; the measured best r
    of the generalized schedule is set against eq. (37)'s r, and the
    selection's pick against the fastest candidate."""
    import numpy as np
    import torch
    from scipy.optimize import nnls

    import ar_synth
    import collective_reduction_gb300 as ar
    torch.cuda.set_device(0)
    dtype = "float32"

    def counters(info):
        return [info["steps"], info["sent_bytes_total"], info["combines"] * esize(dtype), info["messages"]]

    rows = []
    with open(path, "w") as out:
        for P in (4, 16, 63):
            for lg in range(11, 27, 3):
                S = 1 << lg
                n = S // esize(dtype)
                dev = ar_synth.device_inputs(P, n, dtype, sigma=1e-3, seed=P)
                L = (P - 1).bit_length()
                for algo, kw in (("ring", {}), ("binomial", {}), ("rd", {}), ("generalized", {"r": 0}),
                                 ("generalized", {"r": L}),
                                 ("ring", {"phase": "reduce_scatter"}), ("ring", {"phase": "all_gather"})):
                    plan = ar.Plan(P, n, dtype, "sum", algo, form="step", **kw)
                    us = time_plan(plan, dev)
                    c = counters(plan.info())
                    rows.append((c, us))
                    out.write(json.dumps({"phase": "fit", "P": P, "S": S, "algo": algo, "params": kw,
                                          "steps": c[0], "sent_bytes_total": c[1], "combined_bytes": c[2],
                                          "messages": c[3], "us": round(us, 3)}) + "\n")
                    plan.close()
                del dev
                torch.cuda.empty_cache()
        A = np.array([[x / t for x in c] for c, t in rows])
        coef, _ = nnls(A, np.ones(len(rows)))
        alpha, beta, gamma, delta = (float(x) for x in coef)
        pred = A @ coef
        fit = {"phase": "model", "alpha_us": alpha, "beta_us_per_byte": beta, "gamma_us_per_byte": gamma,
               "delta_us_per_message": delta,
               "rel_rms": float(np.sqrt(np.mean((pred - 1.0) ** 2))), "rel_max": float(np.max(np.abs(pred - 1.0))),
               "points": len(rows)}
        out.write(json.dumps(fit) + "\n")
        out.flush()
        model = ar.CostModel(alpha, beta, gamma, delta)
        for P in (7, 12, 31, 63):
            L = (P - 1).bit_length()
            Lp = (1 << (P.bit_length() - 1)).bit_length() - 1
            cands = [("ring", {}), ("binomial", {}), ("rd", {}), ("rh", {})]
            cands += [("hybrid", {"k1": k}) for k in range(Lp + 1)]
            cands += [("generalized", {"r": r}) for r in range(L + 1)]
            for lg in range(10, 25, 2):
                S = 1 << lg
                n = S // esize(dtype)
                dev = ar_synth.device_inputs(P, n, dtype, sigma=1e-3, seed=P)
                meas = {}
                for algo, kw in cands:
                    plan = ar.Plan(P, n, dtype, "sum", algo, form="step", **kw)
                    meas[(algo, json.dumps(kw, sort_keys=True))] = time_plan(plan, dev)
                    plan.close()
                gen = {r: meas[("generalized", json.dumps({"r": r}))] for r in range(L + 1)}
                best_r = min(gen, key=gen.get)
                r37 = ar.optimal_r(P, S, model)
                sel_algo, sel_params, sel_pred = ar.select(P, n, dtype, "sum", model)
                sel_kw = {k: sel_params[k] for k in ("r", "k1") if
                          (k == "r" and sel_algo == "generalized") or (k == "k1" and sel_algo == "hybrid")}
                sel_us = meas[(sel_algo, json.dumps(sel_kw, sort_keys=True))]
                best_key = min(meas, key=meas.get)
                out.write(json.dumps({
                    "phase": "validate", "P": P, "S": S,
                    "generalized_us_by_r": {str(r): round(t, 3) for r, t in gen.items()},
                    "best_r_measured": best_r, "eq37_r": r37,
                    "eq37_loss": round(gen[r37] / gen[best_r], 4),
                    "select": [sel_algo, sel_kw], "select_us": round(sel_us, 3),
                    "select_predicted_us": round(sel_pred, 3),
                    "fastest": [best_key[0], json.loads(best_key[1])], "fastest_us": round(meas[best_key], 3),
                    "select_loss": round(sel_us / meas[best_key], 4),
                    "candidates_us": {f"{k[0]} {k[1]}": round(t, 3) for k, t in meas.items()}}) + "\n")
                out.flush()
                del dev
                torch.cuda.empty_cache()
        # the pipelined chain's block count: the page's optimal m (BSP runtime
        # (T_start + n/m T_byte)(p + m - 2)), with a round's T_start = alpha +
        # (P - 1) delta and a block byte's T_byte = (P - 1)(beta + gamma),
        # against the measured best over a geometric range of m
        for P in (8, 16):
            for lg in (18, 22, 26):
                S = 1 << lg
                n = S // esize(dtype)
                dev = ar_synth.device_inputs(P, n, dtype, sigma=1e-3, seed=P)
                t_start = alpha + (P - 1) * delta
                t_byte = (P - 1) * (beta + gamma)
                m_pred = int(min(4096, max(1, round((S * (P - 2) * t_byte / t_start) ** 0.5))))
                times = {}
                for m in sorted({1, 2, 4, 8, 16, 32, 64, 128, 256, m_pred}):
                    plan = ar.Plan(P, n, dtype, "sum", "pipeline", form="step", blocks=m)
                    times[m] = time_plan(plan, dev)
                    plan.close()
                best = min(times, key=times.get)
                out.write(json.dumps({"phase": "pipeline", "P": P, "S": S, "m_pred": m_pred, "m_best": best,
                                      "pred_loss": round(times[m_pred] / times[best], 4),
                                      "times_us": {str(k): round(v, 3) for k, v in times.items()}}) + "\n")
                out.flush()
                del dev
                torch.cuda.empty_cache()


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
        return
    if a.sweep:
        run_sweep(a, a.sweep)
        return
    if a.configs:
        run_configs(a, a.configs)
        return
    if a.costmodel:
        run_costmodel(a, a.costmodel)
        return
    if a.rows:
        run_rows(a, a.rows)
        return
    run_ours(a)


if __name__ == "__main__":
    main()
