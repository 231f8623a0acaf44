"""Benchmark of the fused ZeRO optimizer step on GB300.

One step = one pass of the whole path over one batch of synthetic gradients: rank-ordered
reduce-scatter of the M bf16 gradient replicas, global-norm clip, AdamW on every owner's
fp32 shard, all-gather of the bf16 parameters. Default workload: the 4B dense-transformer
parameter set (4,092,982,400 params, M = 4, ZeRO-3, clip 1.0).

Prints ONE JSON line (rank 0). Usage:
    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload tiny|gpt2s|1p3b|ragged|4b] [--impl ours|reference]
Multi-GPU: launched by torchrun, one process per GPU. By default every rank runs its own
emulated job (weak scaling, no data-path collective); the barrier and the max-over-ranks
timing use torch.distributed. With --shard the N processes form one job of M = N ranks,
each holding only its shard, with NCCL collectives between them (strong scaling); with
--shard --emulate-ranks one process runs every rank's kernels of such a job on one GPU.
Other modes: --mode stream (ZeRO-2 per-bucket streaming), --mode gather (ZeRO-3 per-bucket
gathers with prefetch), --graph (captured steps), --impl reference (the CPU oracle).
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "params/s and achieved HBM GB/s (% of GB300 peak) per fused ZeRO step"
KERNEL_SRCS = [os.path.join(ROOT, "zero_gradient_reduce_scatter_gb300", "csrc", f)
               for f in ("zero_kernels.cu", "zero_internal.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
VENDOR_HBM_GBS = 7900.0  # GB300 HBM3e nominal, for context beside the measured copy peak
MIB = 1024 * 1024
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=None, choices=["tiny", "gpt2s", "1p3b", "ragged", "4b"],
                    help="default: 4b (the 4B dense set) for --mode step and gather, gpt2s for --mode stream")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="step and stream modes: capture one step (scalars from a device schedule) in a CUDA "
                         "graph and time its replays; gather mode: capture one prefetched sweep; the roofline "
                         "then covers the whole step or sweep")
    ap.add_argument("--cpu-procs", type=int, default=0,
                    help="oracle processes for the CPU baseline and the reference arm (0 = one per host core)")
    ap.add_argument("--ghat-mode", default="auto", choices=["auto", "materialize", "recompute"])
    ap.add_argument("--mode", choices=["step", "stream", "gather"], default="step",
                    help="step: the fused ZeRO step (default); stream: ZeRO-2 per-bucket streaming (one fused "
                         "pass per bucket, or every bucket's reduce-scatter then one update: --stream-form); "
                         "gather: ZeRO-3 per-bucket parameter all-gather with prefetch")
    ap.add_argument("--emulate-ranks", action="store_true",
                    help="with --shard on one GPU: the workload's M ranks as M rank contexts in this one process, "
                         "each holding only its shard, with device copies in place of the collectives (timed "
                         "apart); all ranks' kernels run one after another and move the emulated step's bytes")
    ap.add_argument("--ranks", type=int, default=0,
                    help="with --shard --emulate-ranks: this many ranks instead of the workload's M")
    ap.add_argument("--shard", action="store_true",
                    help="process-per-rank mode: the job's M ranks are the N processes (one per GPU, NCCL), "
                         "each holding only its shard; the workload's tensors, stage, clipping and buckets "
                         "with M = N. Strong scaling: the whole job steps the workload's parameters once")
    ap.add_argument("--stream-form", default="auto", choices=["auto", "fused", "reduce-apply"],
                    help="--mode stream: one fused pass per bucket (no clipping) or reduce-scatter of every "
                         "bucket then one update (auto: fused when the workload does not clip)")
    ap.add_argument("--groups", type=int, default=1,
                    help="hybrid sharding: split the workload's M ranks into this many groups (state "
                         "sharded over M / groups ranks, replicated across groups)")
    ap.add_argument("--overlap", default="buckets", choices=["none", "launch", "buckets"],
                    help="--mode stream and gather: programmatic launch overlap of the per-bucket "
                         "kernels (zero_set_launch_overlap); the roofline then covers the whole step or sweep")
    ap.add_argument("--prefetch-buffers", type=int, default=4,
                    help="--mode gather: transient buffers of the prefetch (buckets gathered ahead + 1)")
    ap.add_argument("--bucket-mib", type=float, default=25.0,
                    help="bucket size for --mode gather when the workload has none")
    ap.add_argument("--max-params", type=int, default=0,
                    help="keep only the workload's leading tensors up to this many parameters (a small "
                         "case of the same kernels, for profiling); 0 = the whole workload")
    return ap.parse_args()


def workload(args):
    import workloads as W
    w = W.workload(args.workload or "4b")
    if args.max_params and args.max_params < w.N:
        keep, total = [], 0
        for n in w.numel:
            if total + n > args.max_params:
                if not keep:
                    keep.append(args.max_params)
                break
            keep.append(n)
            total += n
        w = W.small_variant(w, tuple(keep), name=f"{w.name}; leading {sum(keep):,} parameters only")
    return w


# ------------------------------------------------------------------------------------------
# distributed plumbing (timing only: barrier + max over ranks)
# ------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, use_cuda, timeout_s: float | None = None):
    """Process group for the barrier and the max-over-ranks timing (no data-path collective).
    A rank that never joins makes the others fail after timeout_s instead of waiting forever."""
    if world <= 1:
        return None
    import datetime

    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    kw = {"timeout": datetime.timedelta(seconds=timeout_s)} if timeout_s else {}
    dist.init_process_group("nccl" if use_cuda else "gloo", **kw)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "100"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "power_w_max": max(power),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------
# byte accounting
# ------------------------------------------------------------------------------------------
def alg_bytes_per_param(M: int) -> int:
    """Algorithmic bytes per parameter of one step: read M bf16 gradients and fp32 master,
    m, v; write fp32 master, m, v and the bf16 parameter."""
    return 2 * M + 26


def real_bytes_per_param(M: int, clip: bool, ghat_mode: str) -> int:
    """Bytes the step actually moves per parameter: one fused pass without clipping; with
    clipping either the gradients are read twice (4M + 26) or the fp32 average is written
    and read back (2M + 34)."""
    if not clip:
        return 2 * M + 26
    return 2 * M + 34 if ghat_mode == "materialize" else 4 * M + 26


def kernel_alg_bytes_per_lane(kernel: str, M: int, write_ghat: bool) -> int:
    return {"rs_adamw": 2 * M + 26, "adamw": 4 + 26, "rs_norm": 2 * M + (4 if write_ghat else 0),
            "gather": 4, "norm_final": 0}[kernel]


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha() -> str:
    """Hash of the kernel sources (the kernels and the header that holds their launch shapes
    and cache policies) with comments and blank space removed: an ncu traffic figure counts
    only while the code is unchanged."""
    import re
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str, workload_key: str):
    """dram bytes per launch from the committed ncu summary, if taken on this kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            tab = json.load(f)
        e = tab[f"{workload_key}:{kernel_key}"]
        if e.get("kernel_src_sha") != kernel_sha() or e.get("workload") != workload_key:
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample of the workload
# ------------------------------------------------------------------------------------------
def _oracle_sample(w, seed_step):
    """Inputs of one oracle sample: a 4 Mi-parameter slice of the workload with its M, stage,
    clip and gradient recipe (gradients drawn for step `seed_step`)."""
    import numpy as np
    import torch

    import oracle as O
    import workloads as W

    lanes = 1 << 22
    sample = W.small_variant(w, (lanes,), steps=1)
    p = O.plan(sample.numel, sample.M, sample.bucket_bytes)
    st = O.init_state(p, sample.stage, W.master_init(sample, "cpu").numpy())
    oh = O.hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 clip=w.clip is not None, max_grad_norm=w.clip or 1.0)
    sig = np.array([float(W.sigmas(w)[0])])
    grads = []
    for r in range(sample.M):
        g = torch.zeros(p.npad, dtype=torch.bfloat16)
        W.fill_grads(sample, r, seed_step, g, [0], sig)
        grads.append(g.view(torch.int16).numpy().view(np.uint16))
    return O, p, st, grads, oh


def _oracle_windows(w, worker, windows, seconds, barrier=None):
    """(parameters stepped, seconds) for each of `windows` timed windows of whole oracle steps."""
    O, p, st, grads, oh = _oracle_sample(w, worker)
    out = []
    for _ in range(windows):
        if barrier is not None:
            barrier.wait(timeout=600)
        done, t0 = 0, time.perf_counter()
        while True:
            O.zero_step(p, st, grads, oh)
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds or done >= 10000:
                break
        out.append((done * p.N, el))
    return out


def _oracle_proc(w, worker, windows, seconds, barrier, q):
    import torch
    torch.set_num_threads(1)
    try:
        q.put((worker, _oracle_windows(w, worker, windows, seconds, barrier)))
    except BaseException as e:  # reported to the parent, which raises
        if barrier is not None:
            barrier.abort()
        q.put((worker, repr(e)))


def oracle_rates(w, procs, windows, seconds):
    """Aggregate params/s of `procs` concurrent single-threaded oracle processes (spawned), each
    on its own slice of the workload, per timed window: all parameters stepped in the window
    over the longest of the processes' window times. One process runs in this one."""
    if procs <= 1:
        res = [_oracle_windows(w, 0, windows, seconds)]
    else:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        bar, q = ctx.Barrier(procs), ctx.Queue()
        ps = [ctx.Process(target=_oracle_proc, args=(w, k, windows, seconds, bar, q)) for k in range(procs)]
        for p in ps:
            p.start()
        try:
            got = dict(q.get(timeout=900) for _ in ps)
        finally:
            for p in ps:
                p.join(timeout=60)
                if p.is_alive():
                    p.kill()
        bad = [v for v in got.values() if isinstance(v, str)]
        if bad:
            raise RuntimeError(f"oracle process failed: {bad[0]}")
        res = list(got.values())
    return [sum(r[i][0] for r in res) / max(r[i][1] for r in res) for i in range(windows)]


def copy_rate(pairs, stream) -> float:
    """GB/s of plain copies dst.copy_(src) of every (dst, src) pair, back to back on `stream`
    (best of two passes, CUDA events)."""
    import torch
    best = 0.0
    nbytes = sum(src.numel() * src.element_size() for _, src in pairs)
    for _ in range(2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
            e1.record(stream)
        e1.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return best


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_baseline(w, procs=0):
    """The oracle as it stands on the host cores: one process per core (each single-threaded, on
    its own 4 Mi-parameter slice, ~1.5 s), plus one process alone (~4 s) for the per-core rate."""
    procs = procs or host_cores()
    single = oracle_rates(w, 1, 1, 4.0)[0]
    multi = oracle_rates(w, procs, 1, 1.5)[0] if procs > 1 else single
    desc = (f"oracle steps of 4,194,304-parameter slices of the workload (M={w.M}, ZeRO-{w.stage}, "
            f"clip {'on' if w.clip else 'off'}): {procs} single-threaded processes for ~1.5 s, "
            f"and one alone for ~4 s (single_thread_value)")
    return {"value": multi, "unit": "params/s", "cores": procs, "kind": "oracle", "single_thread_value": single,
            "sample": desc}


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch

    import workloads as W
    import zero_gradient_reduce_scatter_gb300 as zg
    from zero_gradient_reduce_scatter_gb300 import _build

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, True)
    if not os.path.exists(_build.LIB_PATH):
        if rank == 0:
            _build.build()
        barrier(dist, device)

    w = workload(args)
    gather = "fused"
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, device), bucket_bytes=w.bucket_bytes,
                           gather=gather, groups=args.groups)
    sig = W.sigmas(w)
    grads = opt.new_grad_buffers()
    for r in range(w.M):
        W.fill_grads(w, r, 0, grads[r], opt.tensor_offsets, sig)
    h = zg.Hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 clip=w.clip is not None, max_grad_norm=w.clip or 1.0, ghat_mode=args.ghat_mode)
    clip = w.clip is not None
    ghat_mode = args.ghat_mode
    if ghat_mode == "auto":
        ghat_mode = ("materialize" if (w.M > 4 and opt.ghat is not None) else "recompute") if clip else "none"
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    graph, launches_per_step = None, 0
    if args.graph:
        # the step's scalars come from a device schedule, so one captured step replays as the
        # next step each time; an eager scheduled step first counts the launches of a step
        if args.warmup + args.steps + 1 > zg.ZERO_MAX_SCHEDULE:
            raise SystemExit(f"--graph: at most {zg.ZERO_MAX_SCHEDULE - 1} warm-up and timed steps")
        opt.set_schedule([h] * (args.warmup + args.steps + 1))
        opt.set_timing(True)
        opt.kernel_times()
        opt.step_scheduled(grads)
        launches_per_step = int(sum(c for _, c in opt.kernel_times().values()))
        opt.set_timing(False)
        graph = torch.cuda.CUDAGraph()
        gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            opt.step_scheduled(grads)

        def one_step():
            graph.replay()
    else:
        def one_step():
            opt.step(grads, h)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if opt.sync_status() != 0:
        raise SystemExit("warm-up step saw a non-finite gradient norm")

    # ---- timed region: K steps, device events, per-kernel events inside the library ----
    opt.set_timing(True)
    opt.kernel_times()  # reset
    barrier(dist, device)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        one_step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(dist, device)
    ms_total = ev[0].elapsed_time(ev[-1])
    per_step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    step_ms = step_stats(per_step_ms, dist, device)
    ktimes = opt.kernel_times()
    opt.set_timing(False)
    ms_total_max = max_over_ranks(dist, ms_total, device)

    n = w.N
    ms_per_step = ms_total_max / args.steps
    value = world * n * args.steps / (ms_total_max / 1e3)
    alg_b = alg_bytes_per_param(w.M) * n
    gbs_alg = alg_b / (ms_per_step / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    peak_source = f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback"
    lanes = opt.sizes["npad"]
    if graph is not None:
        # replays run no per-launch events: the roofline covers the whole step
        launches = launches_per_step * args.steps
        roofline = {"bound": "hbm", "kernel": "whole step (CUDA graph replay)", "achieved": round(gbs_alg, 1),
                    "peak": peak, "unit": "GB/s", "frac": round(gbs_alg / peak, 4), "traffic": None,
                    "peak_source": peak_source, "alg_bytes_per_launch": alg_b, "avg_launch_ms": round(ms_per_step, 4),
                    "launches_per_step": launches_per_step}
    else:
        launches = int(sum(c for _, c in ktimes.values()))
        # dominant kernel (largest share of the timed region)
        dom = max((k for k in ktimes if ktimes[k][1] > 0), key=lambda k: ktimes[k][0])
        dom_ms = ktimes[dom][0] / ktimes[dom][1]
        dom_bytes = kernel_alg_bytes_per_lane(dom, w.M, ghat_mode == "materialize") * lanes
        achieved = dom_bytes / (dom_ms / 1e3) / 1e9
        variant = {"rs_adamw": "rs_adamw_scaled" if clip and ghat_mode != "materialize" else "rs_adamw_plain",
                   "adamw": "adamw", "rs_norm": "rs_norm_write" if ghat_mode == "materialize" else "rs_norm_only",
                   "gather": "gather", "norm_final": "norm_final"}[dom]
        workload_key = (args.workload or "4b") + (f"-max{args.max_params}" if args.max_params else "")
        traffic = ncu_traffic(variant, workload_key)
        roofline = {"bound": "hbm", "kernel": variant, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": peak_source,
                    "alg_bytes_per_launch": dom_bytes, "avg_launch_ms": round(dom_ms, 4),
                    "kernel_share": {k: round(v[0] / max(ms_total, 1e-9), 4) for k, v in ktimes.items() if v[1]}}
    if graph is not None:
        if opt.sync_status() != 0:
            raise SystemExit("a replayed step found no schedule entry or a non-finite norm")
        opt.set_schedule(None)  # the host-buffer steps below take host scalars

    # ---- end to end through the C ABI with host buffers (pinned) -----------------------
    e2e = None
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    one_fits = local_world * (2 * opt.sizes["npad"] + 2 * n) <= 0.6 * host_mem_available()
    one_fits = max_over_ranks(dist, 0.0 if one_fits else 1.0, device) == 0.0  # all ranks agree
    if not args.no_e2e and not one_fits:
        e2e = {"skipped": f"{local_world} ranks x {(2 * opt.sizes['npad'] + 2 * n) / 1e9:.1f} GB of pinned host "
                          f"memory would exceed 60% of the host's available memory"}
    if not args.no_e2e and one_fits:
        # Through the public host-buffer call: every step copies the M pinned host gradients in
        # (on a copy stream, into one of two device sets in turn, so step k+1's copies run
        # while step k computes) and copies the bf16 parameters back to pinned host memory.
        # Two streams are involved, so the region is timed by the host clock between device
        # synchronisations.
        # Host memory: every rank on the node pins its M replicas. When they would not fit,
        # one pinned replica is the source of all M copies (the same bytes move every step).
        rep_bytes = 2 * opt.sizes["npad"]
        distinct = local_world * (w.M * rep_bytes + 2 * n) <= 0.6 * host_mem_available()
        distinct = max_over_ranks(dist, 0.0 if distinct else 1.0, device) == 0.0
        srcs = [torch.empty(opt.sizes["npad"], dtype=torch.bfloat16, pin_memory=True)
                for _ in range(w.M if distinct else 1)]
        for i, hs in enumerate(srcs):
            hs.copy_(grads[i])
        host_grads = srcs if distinct else srcs * w.M
        host_params = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
        sets = [grads, opt.new_grad_buffers()]
        copy_stream = torch.cuda.Stream(device=device)
        for i in range(2):  # warm-up, both device sets
            opt.step_host_overlapped(host_grads, sets[i], host_params, h, copy_stream)
        torch.cuda.synchronize()
        # the host link's rate right now, by plain copies of the same bytes: pinned host-to-
        # device bandwidth on a shared host varies over minutes, and it bounds this number
        h2d_gbs = copy_rate([(sets[0][r], host_grads[r]) for r in range(w.M)], copy_stream)
        d2h_gbs = copy_rate([(host_params, opt.params())], copy_stream)
        barrier(dist, device)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
        t0 = time.perf_counter()
        marks[0].record(stream)
        for i in range(args.e2e_steps):
            opt.step_host_overlapped(host_grads, sets[i % 2], host_params, h, copy_stream)
            marks[i + 1].record(stream)  # after the step's parameters reached the host
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3, device)
        e2e_step_ms = [round(marks[i].elapsed_time(marks[i + 1]), 2) for i in range(args.e2e_steps)]
        h2d_after = copy_rate([(sets[0][r], host_grads[r]) for r in range(w.M)], copy_stream)
        h2d_bytes = sum(g.numel() * 2 for g in host_grads)
        e2e = {"value": world * n * args.e2e_steps / (e2e_ms / 1e3), "unit": "params/s",
               "ms_per_step": e2e_ms / args.e2e_steps, "ms_per_step_median": statistics.median(e2e_step_ms),
               "call": "zero_step_host_overlapped",
               "h2d_bytes_per_step": sum(g.numel() * 2 for g in host_grads), "d2h_bytes_per_step": n * 2,
               "host_gradients": (f"{w.M} pinned replicas" if distinct else
                                  f"one pinned replica copied to all {w.M} device buffers (host memory)"),
               "h2d_copy_gbs": round(h2d_gbs, 1), "d2h_copy_gbs": round(d2h_gbs, 1),
               "h2d_copy_gbs_after": round(h2d_after, 1), "step_ms": e2e_step_ms,
               "copy_floor_ms": round(h2d_bytes / h2d_gbs / 1e6, 2),
               "copy_floor_ms_after": round(h2d_bytes / h2d_after / 1e6, 2)}
        del host_grads, host_params, sets, srcs

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_procs)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": step_ms["median"],
            "ms_per_step_min": step_ms["min"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name + (f"; hybrid sharding: {args.groups} groups of {w.M // args.groups}"
                                             if args.groups > 1 else ""), "params": n, "M": w.M, "stage": w.stage,
                       "clip": w.clip, "bucket_bytes": w.bucket_bytes, "gather": gather, "ghat_mode": ghat_mode,
                       "padded_lanes": lanes,
                       "l2": l2_note(opt.sizes["bytes_grad_each"] * w.M + 12 * lanes),
                       "cuda_graph": bool(args.graph),
                       "parallelism": f"{world} independent emulated jobs (one per GPU)"},
            "gbs_alg": round(gbs_alg, 1), "alg_bytes_per_param": alg_bytes_per_param(w.M),
            "frac_of_peak_alg": round(gbs_alg / peak, 4),
            **target_stats(per_step_ms, alg_b, peak, dist, device),
            "real_bytes_per_param": real_bytes_per_param(w.M, clip, ghat_mode),
            "gbs_real": round(real_bytes_per_param(w.M, clip, ghat_mode) * n / (ms_per_step / 1e3) / 1e9, 1),
            "frac_of_peak_real": round(real_bytes_per_param(w.M, clip, ghat_mode) * n / (ms_per_step / 1e3) / 1e9
                                       / peak, 4),
            "frac_of_vendor_hbm_alg": round(gbs_alg / VENDOR_HBM_GBS, 4),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
        }
        print_line(line)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores, a bounded sample per step
# ------------------------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = workload(args)
    procs = args.cpu_procs or host_cores()
    rates = oracle_rates(w, procs, args.warmup + args.steps, 2.0)
    timed = rates[args.warmup:] or rates[-1:]
    rate = statistics.median(timed)
    sample = (f"per step, ~2 s of oracle steps on 4,194,304-parameter slices of the workload (M={w.M}, "
              f"ZeRO-{w.stage}, clip {'on' if w.clip else 'off'}) in {procs} single-threaded processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "params/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.N / rate * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "params": w.N, "M": w.M, "stage": w.stage, "clip": w.clip},
        "cpu_baseline": {"value": rate, "unit": "params/s", "cores": procs, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print_line(line)


def _timed_region(fn, steps, stream, dist, device):
    import torch
    barrier(dist, device)
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(dist, device)
    step_ms = step_stats([ev[i].elapsed_time(ev[i + 1]) for i in range(steps)], dist, device)
    return max_over_ranks(dist, ev[0].elapsed_time(ev[-1]), device), clk, step_ms


def host_mem_available() -> int:
    """MemAvailable of this host in bytes (0 if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def l2_note(input_bytes):
    """How the timed steps relate to L2 (inputs larger than L2 need no flush between steps)."""
    if input_bytes > L2_BYTES:
        return f"inputs {input_bytes / 1e9:.2f} GB > L2 {L2_BYTES / 1e6:.0f} MB; no flush"
    return (f"inputs {input_bytes / 1e6:.3f} MB fit in L2 {L2_BYTES / 1e6:.0f} MB and are not flushed: "
            f"a latency figure for a launch-bound step, not a bandwidth one")


TARGET_FRAC_ALG = 0.80  # the step's bandwidth target: this fraction of the measured HBM peak


def target_stats(per_step_ms, alg_bytes, peak, dist, device):
    """How the individual timed steps stand against the bandwidth target: each step's fraction
    of the peak under the algorithmic bytes (a rank's step counts at its own time; with several
    ranks the count is the smallest over ranks), and how many steps reach the target."""
    fr = [alg_bytes / (t / 1e3) / 1e9 / peak for t in per_step_ms]
    hits = sum(f >= TARGET_FRAC_ALG for f in fr)
    if dist is not None:
        hits = int(-max_over_ranks(dist, -float(hits), device))
    return {"target_frac_alg": TARGET_FRAC_ALG, "steps_at_or_above_target": int(hits),
            "step_frac_alg": {"min": round(min(fr), 4), "median": round(statistics.median(fr), 4),
                              "max": round(max(fr), 4)}}


def step_stats(ms, dist, device):
    """Median and minimum of the per-step times (CUDA events between steps), each the max over
    ranks."""
    return {"median": round(max_over_ranks(dist, statistics.median(ms), device), 4),
            "min": round(max_over_ranks(dist, min(ms), device), 4)}


def run_stream(args):
    """ZeRO-2 per-bucket streaming, every bucket from its own buffers in backward order.
    Without clipping (form "fused"): zero_step_bucket reduce-scatters and updates each bucket
    in one pass, 2M + 26 bytes per parameter. With clipping (form "reduce-apply"): every bucket
    reduce-scattered into the averaged gradient (zero_reduce_bucket), then one zero_apply,
    the bytes of the materialized clipped step, 2M + 34 per parameter."""
    import torch

    import workloads as W
    import zero_gradient_reduce_scatter_gb300 as zg

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, True)
    args.workload = args.workload or "gpt2s"
    w = workload(args)
    form = args.stream_form
    if form == "auto":
        form = "fused" if w.clip is None else "reduce-apply"
    if form == "fused" and w.clip is not None:
        raise SystemExit("--stream-form fused needs a workload without clipping")
    fused = form == "fused"
    opt = zg.ZeroOptimizer(w.numel, w.M, w.stage, W.master_init(w, device), bucket_bytes=w.bucket_bytes,
                           ghat_buffer=not fused, groups=args.groups)
    full = opt.new_grad_buffers()
    sig = W.sigmas(w)
    for r in range(w.M):
        W.fill_grads(w, r, 0, full[r], opt.tensor_offsets, sig)
    nb = len(opt.buckets)
    slices = [[g[opt.buckets[b][0]:opt.buckets[b][0] + opt.bucket_lanes(b)] for g in full] for b in range(nb)]
    h = zg.Hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                 clip=w.clip is not None, max_grad_norm=w.clip or 1.0)
    stream = torch.cuda.current_stream()

    def eager_step(scheduled=False):
        if fused:
            for b in reversed(range(nb)):
                if scheduled:
                    opt.step_bucket_scheduled(b, slices[b])
                else:
                    opt.step_bucket(b, slices[b], h)
            return
        for b in reversed(range(nb)):
            opt.reduce_bucket(b, slices[b])
        if scheduled:
            opt.apply_scheduled()
        else:
            opt.apply(h)

    step, launches_per_step = eager_step, 0
    overlapped = not args.graph and args.overlap != "none"
    if overlapped:
        # the buckets' slices exist before the step and its calls run back to back on one
        # stream, as the "buckets" mode requires; per-launch events would bracket launches
        # that overlap, so one eager step counts the launches and the region runs untimed
        opt.set_launch_overlap(args.overlap)
        opt.set_timing(True)
        opt.kernel_times()
        eager_step()
        launches_per_step = int(sum(c for _, c in opt.kernel_times().values()))
        opt.set_timing(False)
    if args.graph:  # one captured step (scalars from a device schedule), replayed
        if args.warmup + args.steps + 1 > zg.ZERO_MAX_SCHEDULE:
            raise SystemExit(f"--graph: at most {zg.ZERO_MAX_SCHEDULE - 1} warm-up and timed steps")
        opt.set_schedule([h] * (args.warmup + args.steps + 1))
        opt.set_timing(True)
        opt.kernel_times()
        eager_step(True)
        launches_per_step = int(sum(c for _, c in opt.kernel_times().values()))
        opt.set_timing(False)
        graph = torch.cuda.CUDAGraph()
        gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            eager_step(True)
        step = graph.replay

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if opt.sync_status() != 0:
        raise SystemExit("warm-up step failed")
    opt.set_timing(not overlapped)
    opt.kernel_times()
    ms, clk, step_ms = _timed_region(step, args.steps, stream, dist, device)
    kt = opt.kernel_times()
    if args.graph and opt.sync_status() != 0:
        raise SystemExit("a replayed step found no schedule entry")
    if overlapped and opt.sync_status() != 0:
        raise SystemExit("an overlapped step failed")
    n, lanes = w.N, opt.sizes["npad"]
    peak, kind = hbm_peak()
    ms_step = ms / args.steps
    if args.graph:  # replays run no per-launch events: the roofline covers the whole step
        real_b = 2 * w.M + (26 if fused else 34)
        dom_name, dom_bytes, dom_ms = "whole step (CUDA graph replay)", real_b * w.N, ms_step
        kt = {"all": (ms, launches_per_step * args.steps)}
    elif overlapped:  # launches overlap: the roofline covers the whole step
        real_b = 2 * w.M + (26 if fused else 34)
        dom_name, dom_bytes, dom_ms = f"whole step ({args.overlap}-overlapped bucket launches)", real_b * lanes, ms_step
        kt = {"all": (ms, launches_per_step * args.steps)}
    elif fused:  # per step: one fused launch per bucket
        real_b = 2 * w.M + 26
        dom, dom_name = "rs_adamw", "rs_adamw_plain (all buckets)"
        dom_bytes, dom_ms = real_b * lanes, kt["rs_adamw"][0] / args.steps
    else:
        real_b = 2 * w.M + 34
        rs_ms = kt["rs_norm"][0] / args.steps
        up_ms = kt["adamw"][0] / kt["adamw"][1]
        dom = "adamw" if kt["adamw"][0] >= kt["rs_norm"][0] else "rs_norm"
        dom_name = "adamw" if dom == "adamw" else "rs_norm_write (all buckets)"
        dom_bytes, dom_ms = (30 * lanes, up_ms) if dom == "adamw" else ((2 * w.M + 4) * lanes, rs_ms)
    if rank == 0:
        print_line({
            "metric": METRIC + " (ZeRO-2 per-bucket streaming)", "mode": "stream", "value": world * n * args.steps / (ms / 1e3),
            "unit": "params/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_median": step_ms["median"], "ms_per_step_min": step_ms["min"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name + (f"; hybrid sharding: {args.groups} groups of {w.M // args.groups}"
                                             if args.groups > 1 else ""), "params": n, "M": w.M, "stage": w.stage, "buckets": nb,
                       "bucket_bytes": w.bucket_bytes, "clip": w.clip, "form": form, "cuda_graph": bool(args.graph),
                       "launch_overlap": args.overlap if overlapped else "none"},
            "gbs_alg": round(alg_bytes_per_param(w.M) * n / (ms_step / 1e3) / 1e9, 1),
            "frac_of_peak_alg": round(alg_bytes_per_param(w.M) * n / (ms_step / 1e3) / 1e9 / peak, 4),
            "real_bytes_per_param": real_b,
            "frac_of_peak_real": round(real_b * n / (ms_step / 1e3) / 1e9 / peak, 4),
            "roofline": {"bound": "hbm", "kernel": dom_name,
                         "achieved": round(dom_bytes / (dom_ms / 1e3) / 1e9, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(dom_bytes / (dom_ms / 1e3) / 1e9 / peak, 4), "traffic": None,
                         "peak_source": kind, "kernel_share": {k: round(v[0] / ms, 4) for k, v in kt.items() if v[1]}},
            "gpu_launches": int(sum(c for _, c in kt.values())), "clocks": clk})
    if dist is not None:
        dist.destroy_process_group()


def run_gather(args):
    """ZeRO-3 per-module gather: every bucket's bf16 parameters all-gathered from the padded
    shards into a transient buffer, the next bucket prefetched on a side stream; 4 bytes
    per parameter (2 read, 2 written)."""
    import dataclasses

    import torch

    import workloads as W
    import zero_gradient_reduce_scatter_gb300 as zg

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = dist_init(world, True)
    w = workload(args)
    if w.bucket_bytes == 0:
        w = dataclasses.replace(w, bucket_bytes=int(args.bucket_mib * MIB))
    opt = zg.ZeroOptimizer(w.numel, w.M, 3, W.master_init(w, device), bucket_bytes=w.bucket_bytes, gather="shards")
    nb = len(opt.buckets)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=device)
    order = list(range(nb))

    def sweep():
        for _b, _params in opt.prefetched_buckets(order, stream=stream, side_stream=side,
                                                  buffers=args.prefetch_buffers):
            pass

    opt.set_launch_overlap(args.overlap)
    graph = None
    if args.graph:
        # one sweep captured in a CUDA graph: the prefetch's cross-stream event waits become
        # graph edges; each replay gathers the shards as they are then
        sweep()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        cap_side = torch.cuda.Stream(device=device)
        gc.collect()  # collect garbage (CUDA objects) now, not inside the global-mode capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            for _b, _params in opt.prefetched_buckets(order, stream=torch.cuda.current_stream(), side_stream=cap_side,
                                                      buffers=args.prefetch_buffers):
                pass
        sweep = graph.replay
    for _ in range(args.warmup):
        sweep()
    torch.cuda.synchronize()
    # the two buffers' gathers run on two side streams and overlap one another (and, with
    # launch overlap, their launches too): per-launch events would bracket concurrent
    # launches, so the region runs untimed and the roofline covers the whole sweep
    opt.set_timing(False)
    ms, clk, step_ms = _timed_region(sweep, args.steps, stream, dist, device)
    n = w.N
    peak, kind = hbm_peak()
    g_ms, g_cnt = ms, nb * args.steps
    achieved = 4 * n * args.steps / (g_ms / 1e3) / 1e9
    if rank == 0:
        print_line({
            "metric": "params/s and achieved HBM GB/s of the ZeRO-3 per-bucket parameter all-gather", "mode": "gather",
            "value": world * n * args.steps / (ms / 1e3), "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "ms_per_step_median": step_ms["median"],
            "ms_per_step_min": step_ms["min"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "params": n, "M": w.M, "stage": 3, "buckets": nb,
                       "bucket_bytes": w.bucket_bytes,
                       "prefetch": f"{args.prefetch_buffers - 1} bucket(s) ahead, {args.prefetch_buffers} transient "
                                   "buffers, a side stream per buffer",
                       "launch_overlap": args.overlap, "cuda_graph": graph is not None},
            "roofline": {"bound": "hbm", "kernel": "gather (whole sweep" + (", CUDA graph replay" if graph is not None
                                                                         else f", {args.overlap} launch overlap") + ")",
                         "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None, "peak_source": kind,
                         "alg_bytes_per_param": 4, "avg_launch_ms": round(g_ms / max(g_cnt, 1), 4)},
            "gpu_launches": int(g_cnt), "clocks": clk})
    if dist is not None:
        dist.destroy_process_group()


def print_line(line: dict):
    """The one JSON line. C-level stdout of the libraries (NCCL prints its version there) is
    flushed first, so that the line is the last one the process writes."""
    import ctypes
    try:
        ctypes.CDLL(None).fflush(None)
    except (OSError, AttributeError):
        pass
    sys.stdout.write(json.dumps(line) + "\n")
    sys.stdout.flush()


def run_shard(args):
    """Process-per-rank ZeRO step: N processes (torchrun, one per GPU, NCCL; N = 1 runs a job of
    one rank) form one job of M = N ranks over the workload's tensors. Per step every rank
    exchanges its gradient's bucket slices with the others (all-to-all), sums its shard's
    slices in rank order and updates it (the library's kernels), and all-gathers the bf16
    parameters; with clipping one fp64 per rank is all-gathered in between. The timed region
    holds the collectives and the kernels: the job steps w.N parameters per step."""
    import datetime
    import socket

    import torch
    import torch.distributed as tdist

    import workloads as W
    import zero_gradient_reduce_scatter_gb300 as zg
    from zero_gradient_reduce_scatter_gb300 import _build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    if world == 1 and "MASTER_PORT" not in os.environ:
        s = socket.socket()
        s.bind(("127.0.0.1", 0))
        os.environ["MASTER_PORT"] = str(s.getsockname()[1])
        s.close()
    tdist.init_process_group("nccl", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=600),
                             device_id=device)
    dist = tdist if world > 1 else None
    if not os.path.exists(_build.LIB_PATH):
        if rank == 0:
            _build.build()
        tdist.barrier(device_ids=[local])
    w0 = workload(args)
    w = W.small_variant(w0, w0.numel, name=w0.name, M=world)
    opt = zg.ShardedZeroOptimizer(w.numel, w.stage, W.master_init(w, device), bucket_bytes=w.bucket_bytes,
                                  full_params=True)
    grad = opt.new_grad_buffer()
    W.fill_grads(w, rank, 0, grad, opt.tensor_offsets)
    clip = w.clip is not None
    h = zg.Hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, clip=clip,
                 max_grad_norm=w.clip or 1.0, ghat_mode=args.ghat_mode)
    ghat_mode = args.ghat_mode
    if ghat_mode == "auto":
        ghat_mode = ("materialize" if (w.M > 4 and opt.ghat is not None) else "recompute") if clip else "none"
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        opt.step(grad, h)
    torch.cuda.synchronize()
    if opt.sync_status() != 0:
        raise SystemExit("warm-up step saw a non-finite gradient norm")
    # the step itself, with no per-launch events
    ms_total, clk, step_ms = _timed_region(lambda: opt.step(grad, h), args.steps, stream, dist, device)
    # then the same steps with every kernel launch bracketed by events
    opt.set_timing(True)
    opt.kernel_times()
    _timed_region(lambda: opt.step(grad, h), args.steps, stream, dist, device)
    kt = opt.kernel_times()
    opt.set_timing(False)
    n, L = w.N, opt.sizes["shard_len"]
    ms_per_step = ms_total / args.steps
    peak, peak_kind = hbm_peak()
    # each kernel kind covers the rank's shard once per step (in one launch per bucket where
    # it reads the exchanged slices): the dominant kernel's algorithmic bytes per step over
    # its time per step
    dom = max((k for k in kt if kt[k][1] > 0), key=lambda k: kt[k][0])
    dom_step_bytes = kernel_alg_bytes_per_lane(dom, w.M, ghat_mode == "materialize") * L
    dom_ms = kt[dom][0] / args.steps
    dom_launches = kt[dom][1] / args.steps
    achieved = dom_step_bytes / (dom_ms / 1e3) / 1e9
    kernel_ms = sum(v[0] for v in kt.values()) / args.steps

    e2e = None
    # every rank on the node pins its gradient and its parameters (2 B per padded lane each)
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    e2e_fits = local_world * 4 * opt.sizes["npad"] <= 0.6 * host_mem_available()
    e2e_fits = max_over_ranks(dist, 0.0 if e2e_fits else 1.0, device) == 0.0  # all ranks agree
    if not args.no_e2e and not e2e_fits:
        e2e = {"skipped": f"{local_world} ranks x {4 * opt.sizes['npad'] / 1e9:.1f} GB of pinned host memory "
                          f"would exceed 60% of the host's available memory"}
    if not args.no_e2e and e2e_fits:
        # the rank's gradient from pinned host memory in (on a copy stream, into two device
        # buffers in turn, so the next step's copy overlaps this step), the parameters out
        host_g = torch.empty(opt.sizes["npad"], dtype=torch.bfloat16, pin_memory=True)
        host_g.copy_(grad)
        host_p = torch.empty(opt.sizes["npad"], dtype=torch.bfloat16, pin_memory=True)
        bufs = [grad, opt.new_grad_buffer()]
        copy_stream = torch.cuda.Stream(device=device)
        turn = [0]
        last = 2 + args.e2e_steps  # two warm-up calls, then the timed ones

        def e2e_step():
            opt.step_host_overlapped(host_g, bufs[turn[0] % 2], host_p, h, copy_stream)
            turn[0] += 1
            if turn[0] == last:  # the last parameter copy to host inside the timed region
                stream.wait_event(opt.params_copied)

        for _ in range(2):
            e2e_step()
        e_ms, _, e_stats = _timed_region(e2e_step, args.e2e_steps, stream, dist, device)
        gbytes = 2 * opt.sizes["npad"]
        h2d_gbs = copy_rate([(bufs[0], host_g)], copy_stream)
        d2h_gbs = copy_rate([(host_p, opt.params())], copy_stream)
        e2e = {"value": n / (e_ms / args.e2e_steps / 1e3), "unit": "params/s", "ms_per_step": e_ms / args.e2e_steps,
               "ms_per_step_median": e_stats["median"], "call": "ShardedZeroOptimizer.step_host_overlapped",
               "h2d_bytes_per_step": gbytes * world, "d2h_bytes_per_step": gbytes * world,
               "h2d_copy_gbs_after": round(h2d_gbs, 1), "d2h_copy_gbs_after": round(d2h_gbs, 1),
               "copy_floor_ms_after": round(gbytes / min(h2d_gbs, d2h_gbs) / 1e6, 2)}
        del bufs
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_procs)
    if rank == 0:
        line = {
            "metric": METRIC, "value": n / (ms_per_step / 1e3), "unit": "params/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "ms_per_step_median": step_ms["median"], "ms_per_step_min": step_ms["min"], "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w0.name + f"; process per rank: M = {world}", "params": n, "M": world,
                       "stage": w.stage, "clip": w.clip, "bucket_bytes": w.bucket_bytes, "ghat_mode": ghat_mode,
                       "padded_lanes": opt.sizes["npad"], "shard_lanes": L,
                       "l2": l2_note(opt.sizes["bytes_grad_each"] * 2 + 12 * L),
                       "parallelism": (f"zero-dp{world}: one process per GPU, state sharded over {world} ranks "
                                       f"(NCCL all-to-all of bf16 bucket slices, rank-ordered fp32 sum at the owner, "
                                       f"bf16 all-gather)") if world > 1 else
                                      ("zero-dp1: one process, the whole state on one GPU (the exchange and the "
                                       "all-gather of one rank are identities: the kernels read the gradient in "
                                       "place, the full parameters are the bf16 shard)")},
            "kernel_ms_per_step": round(kernel_ms, 4),
            "collective_ms_per_step": round(ms_per_step - kernel_ms, 4),
            "kernel_timing": "a second pass of the same steps, each kernel launch bracketed by events",
            "frac_of_peak_alg_kernels": round(alg_bytes_per_param(w.M) * L / (kernel_ms / 1e3) / 1e9 / peak, 4),
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(dom, f"{args.workload or '4b'}-shard-m{world}")
                         if not args.max_params else None,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                         "alg_bytes_per_launch": dom_step_bytes / max(dom_launches, 1),
                         "avg_launch_ms": round(dom_ms / max(dom_launches, 1), 4),
                         "launches_per_step": dom_launches},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(sum(v[1] for v in kt.values())), "clocks": clk,
        }
        print_line(line)
    opt.close()
    tdist.destroy_process_group()


def run_shard_emulated(args):
    """The process-per-rank step of the workload's M ranks on one GPU, measured: M rank contexts
    (zero_config.sharded) in this process, each with only its shard of the state, its own
    exchange buffer and full-parameter buffer. The collectives are device copies in the
    exchange layout (all-to-all of every bucket's slices, the sums in rank order, the all-gather
    of bf16 shards), timed apart from the kernels. One step runs every rank's library calls one
    after another: the kernels' time per step is the sum over ranks, and their bytes are the
    emulated step's, (2M+26) per lane plus the clipped forms' extra pass."""
    import ctypes

    import torch

    import workloads as W
    import zero_gradient_reduce_scatter_gb300 as zg
    from zero_gradient_reduce_scatter_gb300 import _build

    world, rank, local = dist_env()
    if world != 1:
        raise SystemExit("--emulate-ranks runs on one GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if not os.path.exists(_build.LIB_PATH):
        _build.build()
    w = workload(args)
    if args.ranks:
        w = W.small_variant(w, w.numel, name=w.name + f" (as {args.ranks} ranks)", M=args.ranks)
    M, lib, sh = w.M, zg._lib(), zg._stream_handle(None)
    G = max(1, args.groups)
    if M % G:
        raise SystemExit(f"{M} ranks do not split into {G} groups")
    K = M // G  # owners of one copy of the state (the layout is planned for them)
    _, buckets = zg.layout(w.numel, M, w.stage, w.bucket_bytes, groups=G)
    sz = zg.plan(w.numel, M, w.stage, w.bucket_bytes, groups=G, rank=0)
    L, npad = sz["shard_len"], sz["npad"]
    clip = w.clip is not None
    h = zg.Hyper(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, clip=clip,
                 max_grad_norm=w.clip or 1.0, ghat_mode=args.ghat_mode)
    ghat = M > 4
    mi = W.master_init(w, device)
    ranks = []
    for r in range(M):
        b = {k: torch.empty(L, dtype=torch.float32, device=device) for k in ("master", "m", "v")}
        b["ghat"] = torch.empty(L, dtype=torch.float32, device=device) if ghat else None
        b["shards"] = torch.empty(L, dtype=torch.bfloat16, device=device)
        b["full"] = torch.empty(npad, dtype=torch.bfloat16, device=device)
        b["scratch"] = torch.empty(sz["bytes_scratch"], dtype=torch.uint8, device=device)
        b["recv"] = torch.empty(npad, dtype=torch.bfloat16, device=device)
        b["sumsq"] = torch.zeros(1, dtype=torch.float64, device=device)
        b["sums"] = torch.zeros(K, dtype=torch.float64, device=device)
        if G > 1:
            b["part"] = torch.empty(L, dtype=torch.float32, device=device)
            b["parts"] = torch.empty(G * L, dtype=torch.float32, device=device)
        b["grp"], b["k"] = divmod(r, K)
        bufs = zg.Buffers(b["master"].data_ptr(), b["m"].data_ptr(), b["v"].data_ptr(),
                          b["ghat"].data_ptr() if ghat else None, b["full"].data_ptr(), b["shards"].data_ptr(),
                          b["scratch"].data_ptr())
        ctx = ctypes.c_void_p()
        cfg = zg.Config(M, w.stage, w.bucket_bytes, 0, G if G > 1 else 0, 1, r)
        zg._check(lib.zero_init(ctypes.byref(ctx), ctypes.byref(cfg), ctypes.cast(zg._i64_array(w.numel), ctypes.c_void_p),
                                len(w.numel), ctypes.byref(bufs), mi.data_ptr(), sh), "zero_init")
        b["ctx"] = ctx
        ranks.append(b)
    del mi
    toff, _ = zg.layout(w.numel, M, w.stage, w.bucket_bytes, groups=G)
    grads = [torch.zeros(npad, dtype=torch.bfloat16, device=device) for _ in range(M)]
    sig = W.sigmas(w)
    for r in range(M):
        W.fill_grads(w, r, 0, grads[r], toff, sig)
    bases = [0]
    for bk in buckets:
        bases.append(bases[-1] + bk[2])

    # the collectives, as device copies (the exchange and the all-gather inside each group,
    # the group partials of a shard across the groups, the sums inside the group)
    def exchange():
        for b in ranks:
            for off, _n, S, _ in buckets:
                for q in range(K):
                    src = grads[b["grp"] * K + q]
                    b["recv"][off + q * S: off + (q + 1) * S].copy_(src[off + b["k"] * S: off + (b["k"] + 1) * S])

    def gather():
        for b in ranks:
            for i, (off, _n, S, _) in enumerate(buckets):
                for q in range(K):
                    sh_q = ranks[b["grp"] * K + q]["shards"]
                    b["full"][off + q * S: off + (q + 1) * S].copy_(sh_q[bases[i]:bases[i] + S])

    def xfer_parts():
        for b in ranks:
            for g in range(G):
                b["parts"][g * L:(g + 1) * L].copy_(ranks[g * K + b["k"]]["part"])

    def xfer_sums():
        for b in ranks:
            for q in range(K):
                b["sums"][q:q + 1].copy_(ranks[b["grp"] * K + q]["sumsq"])

    def src(b):
        return b["parts"] if G > 1 else b["recv"]

    # the library's calls, phase by phase
    def lib_partial():
        for b in ranks:
            zg._check(lib.zero_rank_partial(b["ctx"], b["recv"].data_ptr(), b["part"].data_ptr(), sh),
                      "zero_rank_partial")

    def lib_sumsq():
        for b in ranks:
            zg._check(lib.zero_rank_sumsq(b["ctx"], src(b).data_ptr(), ctypes.byref(h), b["sumsq"].data_ptr(), sh),
                      "zero_rank_sumsq")

    def lib_step():
        for b in ranks:
            zg._check(lib.zero_rank_step(b["ctx"], src(b).data_ptr(), b["sums"].data_ptr() if clip else None,
                                         w.stage, ctypes.byref(h), sh), "zero_rank_step")

    phases = [("copy", exchange)]
    if G > 1:
        phases += [("lib", lib_partial), ("copy", xfer_parts)]
    if clip:
        phases += [("lib", lib_sumsq), ("copy", xfer_sums)]
    phases += [("lib", lib_step), ("copy", gather)]

    def kernels():  # the library's calls alone (for per-kernel timing), with the copies between
        for kind, fn in phases[1:-1]:
            fn()

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        exchange()
        kernels()
        gather()
    torch.cuda.synchronize()
    for b in ranks:
        if lib.zero_sync_status(b["ctx"]) != 0:
            raise SystemExit("warm-up step saw a non-finite gradient norm")
    # every step: the exchange copies, the ranks' kernels (events around them), the all-gather
    nlib = sum(1 for kind, _ in phases if kind == "lib")
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nlib)]
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        j = 0
        for kind, fn in phases:
            if kind == "lib":
                ev[i][j][0].record(stream)
                fn()
                ev[i][j][1].record(stream)
                j += 1
            else:
                fn()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    kms = [sum(a.elapsed_time(b) for a, b in step) for step in ev]
    k_ms = sum(kms) / args.steps
    total_ms = t0.elapsed_time(t1) / args.steps
    # per-kernel times in a second pass (each launch bracketed by events)
    for b in ranks:
        lib.zero_set_timing(b["ctx"], 1)
        lib.zero_kernel_times(b["ctx"], None, None)
    for _ in range(args.steps):
        kernels()
    torch.cuda.synchronize()
    tot = {}
    for b in ranks:
        ms = (ctypes.c_double * len(zg.KERNELS))()
        cnt = (ctypes.c_int64 * len(zg.KERNELS))()
        lib.zero_kernel_times(b["ctx"], ctypes.cast(ms, ctypes.c_void_p), ctypes.cast(cnt, ctypes.c_void_p))
        for i, k in enumerate(zg.KERNELS):
            t = tot.setdefault(k, [0.0, 0])
            t[0] += ms[i]
            t[1] += cnt[i]
        lib.zero_set_timing(b["ctx"], 0)
    ghat_mode = args.ghat_mode
    if ghat_mode == "auto":
        ghat_mode = ("materialize" if ghat else "recompute") if clip else "none"
    mat = ghat_mode == "materialize"
    # algorithmic bytes per lane of the rank's shard, per kernel kind and step: flat, the
    # emulated kernels' bytes with M bf16 sources; hybrid, the group partial (K bf16 sources
    # in, one fp32 out) and the passes over the G fp32 partials
    if G > 1:
        per_lane = {"rs_norm": (2 * K + 4) + ((4 * G + (4 if mat else 0)) if clip else 0),
                    "rs_adamw": 4 * G + 26, "adamw": 30, "norm_final": 0}
    else:
        per_lane = {"rs_norm": (2 * M + (4 if mat else 0)) if clip else 0, "rs_adamw": 2 * M + 26, "adamw": 30,
                    "norm_final": 0}
    ran = {k: v for k, v in tot.items() if v[1] > 0}
    step_bytes = sum(per_lane.get(k, 0) for k in ran) * L * M
    dom = max(ran, key=lambda k: ran[k][0])
    dom_ms = ran[dom][0] / ran[dom][1]
    dom_bytes = per_lane.get(dom, 0) * L * M * args.steps / ran[dom][1]  # per launch
    peak, peak_kind = hbm_peak()
    n = w.N
    line = {
        "metric": METRIC, "value": n / (k_ms / 1e3), "unit": "params/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": k_ms, "ms_per_step_median": round(statistics.median(kms), 4),
        "ms_per_step_min": round(min(kms), 4), "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name + f"; process-per-rank kernels of all {M} ranks, one process"
                               + (f", hybrid sharding: {G} groups of {K}" if G > 1 else ""),
                   "params": n, "M": M, "groups": G, "stage": w.stage, "clip": w.clip, "bucket_bytes": w.bucket_bytes,
                   "ghat_mode": ghat_mode, "shard_lanes": L, "padded_lanes": npad,
                   "l2": l2_note(2 * npad * M),
                   "parallelism": f"zero-dp{M} emulated: {M} rank contexts on one GPU, collectives as device copies"},
        "value_counts": "the ranks' kernels only (the step's library calls, all ranks one after another)",
        "ms_per_step_with_copies": round(total_ms, 4),
        "kernel_alg_bytes_per_step": step_bytes,
        "frac_of_peak_kernels": round(step_bytes / (k_ms / 1e3) / 1e9 / peak, 4),
        "frac_of_peak_alg": round(alg_bytes_per_param(M) * n / (k_ms / 1e3) / 1e9 / peak, 4) if G == 1 else None,
        "roofline": {"bound": "hbm", "kernel": dom + (" (exchange-layout sources)" if G == 1 else " (hybrid rank kernels)"),
                     "achieved": round(dom_bytes / (dom_ms / 1e3) / 1e9, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(dom_bytes / (dom_ms / 1e3) / 1e9 / peak, 4),
                     "traffic": ncu_traffic(dom, f"{args.workload or '4b'}-ranks-m{M}")
                     if G == 1 and not args.max_params else None,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "alg_bytes_per_launch": dom_bytes, "avg_launch_ms": round(dom_ms, 4),
                     "kernel_share": {k: round(v[0] / max(sum(x[0] for x in tot.values()), 1e-9), 4)
                                      for k, v in tot.items() if v[1]}},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": int(sum(v[1] for v in tot.values())), "clocks": clk,
    }
    for b in ranks:
        lib.zero_destroy(b["ctx"])
    print_line(line)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.shard and args.emulate_ranks:
        run_shard_emulated(args)
    elif args.shard:
        run_shard(args)
    elif args.mode == "stream":
        run_stream(args)
    elif args.mode == "gather":
        run_gather(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
