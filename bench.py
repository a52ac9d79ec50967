#!/usr/bin/env python
"""Benchmark of the chunked causal-attention layer pass (StreamBP / SeCO chunk
calls): reset the dK/dV running sums, forward every chunk, backward every chunk
last to first, all through the libseqattn C ABI.

Metric: causal fwd+bwd TFLOP/s (14 * B * Hq * d * T(T+1)/2 FLOPs credited per
pass).  One JSON line on stdout (rank 0).  Usage:

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--oracle-threads N]

With N > 1 it is launched by torchrun, one process per GPU; every rank runs
its own independent problems (weak scaling, no data-path collective) and the
timing is the max over ranks.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "chunked causal attn fwd+bwd TFLOP/s (causal FLOPs) and % of GB300 BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_BURST_TFLOPS = 1900.0       # used only when no measured peaks file exists
FALLBACK_SUSTAINED_TFLOPS = 1700.0

# DRAM traffic (bytes read + written) of one backward launch, from a full ncu
# capture of a mid-sequence chunk of the workload (chunk 7 of 16 for the
# 32768-token layer: dram__bytes_read.sum + dram__bytes_write.sum), keyed by
# the workload; other workloads report None, and an entry is removed whenever
# the kernel changes until it is measured again.
BWD_TRAFFIC_BYTES_PER_LAUNCH = {
    # bwd_bf16_kernel<128>: dK/dV added by TMA reduce-adds, prefix swept in
    # alternating direction from chunk to chunk (chunk 7 runs it descending)
    "llama3-8b-layer-t32768-c2048": 468.9e6,
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-wgrad", action="store_true")
    ap.add_argument("--oracle-only", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--no-single-core", action="store_true",
                    help="skip the one-core oracle timing of the cpu_baseline")
    ap.add_argument("--oracle-threads", type=int, default=None,
                    help="BLAS threads of the float64 oracle (cpu_baseline and --impl reference); "
                         "default: every core of the process's affinity mask")
    return ap.parse_args()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    """Dense bf16 peaks from the generated MEASURED_PEAKS.json: the burst
    figure (a cuBLAS GEMM timed alone) is the roofline denominator for the
    kernels of a step of a few tens of milliseconds; the sustained figure (the
    same GEMM looped for seconds under the power cap) is reported beside it,
    with the SM clock it was measured at."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        clk = pk.get("clocks_under_load", {}).get("sm_mhz_median")
        return {"burst": float(pk["bf16_tflops"]), "sustained": float(pk["bf16_tflops_sustained"]),
                "sustained_sm_mhz": clk,
                "source": "measured (cuBLAS bf16 GEMM, MEASURED_PEAKS.json)"}
    except (OSError, KeyError, ValueError):
        return {"burst": FALLBACK_BURST_TFLOPS, "sustained": FALLBACK_SUSTAINED_TFLOPS,
                "sustained_sm_mhz": None, "source": "fallback (one earlier GB300 measurement)"}


# ------------------------------------------------------------------ CPU oracle sample

def oracle_sample(w, seed, heads):
    """Bounded sample of the workload for the float64 oracle: the last chunk
    (the longest prefix), forward + backward, for `heads` query heads of key/value
    head 0.  Returns (credited causal FLOPs, seconds, description)."""
    import oracle
    import torch
    from long_context_attention_seqattn_gb300 import inputs, workloads

    dt = inputs.torch_dtype(w.dtype)
    s = workloads.chunk_starts(w.seq, w.chunk)[-1]
    c = min(w.chunk, w.seq - s)
    d = w.head_dim

    def rows(name, r0, r1, H, hs):
        return inputs.draw_rows(name, seed, 0, r0, r1, H, d, dt)[:, hs].to(torch.float64).numpy()[None]

    q = rows("q", s, s + c, w.hq, slice(0, heads))
    do = rows("do", s, s + c, w.hq, slice(0, heads))
    k = rows("k", 0, s + c, w.hkv, slice(0, 1))
    v = rows("v", 0, s + c, w.hkv, slice(0, 1))
    import numpy as np
    t0 = time.perf_counter()
    o, lse = oracle.chunk_forward(q, k, v, s, s, w.scale)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    oracle.chunk_backward(q, k, v, o, lse, do, s, s, w.scale, dk, dv)
    secs = time.perf_counter() - t0
    flops = 14 * heads * d * workloads.causal_pairs(s, c)
    desc = (f"float64 NumPy oracle, last chunk (rows {s}..{s + c - 1}, prefix {s}) fwd+bwd for "
            f"{heads} query head(s) of key/value head 0; credited causal FLOPs {flops:.3e}")
    return flops, secs, desc


ORACLE_THREADS = None   # set from --oracle-threads before NumPy is imported


def affinity_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_cores():
    """Threads the oracle's BLAS may use: the affinity mask's cores, or fewer
    when --oracle-threads caps them."""
    n = affinity_cores()
    return min(n, ORACLE_THREADS) if ORACLE_THREADS else n


def blas_info():
    """Name and live thread count of the BLAS library NumPy loaded (OpenBLAS
    reports its count through its own exported query function)."""
    import ctypes

    import numpy as np
    a = np.ones((64, 64))
    a @ a                                     # make sure the BLAS library is loaded
    info = {"library": None, "threads": None}
    try:
        with open("/proc/self/maps") as fh:
            libs = sorted({ln.split()[-1] for ln in fh if "blas" in ln.lower() and ln.split()[-1].startswith("/")})
    except OSError:
        libs = []
    for path in libs:
        info["library"] = os.path.basename(path)
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                    "openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                info["threads"] = int(fn())
                return info
    return info


def cpu_baseline_record(value, seconds, desc):
    """cpu_baseline object of the bench line: the oracle's rate on this host
    with the cores it could use and the BLAS threads it actually ran with."""
    return {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle", "sample": desc,
            "seconds": seconds, "affinity_cores": affinity_cores(), "cpu_count": os.cpu_count(),
            "blas": blas_info()}


def oracle_only(args, w):
    """--oracle-only: time the oracle's bounded sample of workload ``w`` (all
    query heads of key/value head 0) with the threads --oracle-threads allows
    and print one JSON object; bench.py runs this in a child process for the
    single-core baseline, since the BLAS thread pool is sized at import."""
    G = w.hq // w.hkv
    f, s, desc = oracle_sample(w, w.seed, G)
    rec = cpu_baseline_record(f / s / 1e12, s, desc)
    rec["workload"] = w.name
    print(json.dumps(rec), flush=True)


def single_core_baseline(workload="qwen3-4b-layer-t8192-c512"):
    """The oracle on one core (one BLAS thread, one-core affinity) on the
    8192-token layer's sample, in a child process; None if it fails."""
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-only", "--oracle-threads", "1",
           "--workload", workload]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        return None


# ------------------------------------------------------------------ reference arm

def run_reference(args, w):
    from long_context_attention_seqattn_gb300 import dist
    rank, world = dist.init("gloo")
    if rank != 0:
        dist.finalize()
        return
    for _ in range(args.warmup):
        oracle_sample(w, w.seed, 1)
    flops = secs = 0.0
    desc = ""
    for _ in range(args.steps):
        f, s, desc = oracle_sample(w, w.seed, 1)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": cpu_baseline_record(value, secs / args.steps, desc),
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    dist.finalize()


def workload_config(w):
    in_bytes = 2 * (2 * w.batch * w.seq * w.hq * w.head_dim + 2 * w.batch * w.seq * w.hkv * w.head_dim)
    return {"workload": w.name, "batch": w.batch, "seq_len": w.seq, "chunk": w.chunk,
            "num_chunks": (w.seq + w.chunk - 1) // w.chunk, "num_q_heads": w.hq,
            "num_kv_heads": w.hkv, "head_dim": w.head_dim,
            "l2": f"inputs larger than L2: Q, K, V, dO = {in_bytes / 2**20:.0f} MiB per step"}


# ------------------------------------------------------------------ our arm

def run_ours(args, w):
    import torch

    from long_context_attention_seqattn_gb300 import binding, build, dist, inputs, workloads

    rank, world = dist.init("nccl")
    _, local_rank, _ = dist.rank_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    build.build()
    binding.load_library()

    # every rank owns its own batch entry of independent problems (weak scaling)
    seed = w.seed + rank
    q, k, v, do = inputs.layer_inputs(w, device=dev, seed=seed)
    bufs = binding.LayerBuffers(q, k, w.chunk)
    starts = bufs.starts
    D = len(starts)
    T, c = w.seq, w.chunk

    main = torch.cuda.current_stream()
    n_fwd = binding.auto_fwd_streams(q, c)
    n_bwd = binding.auto_bwd_streams(q, k, c)

    def step(events=None):
        # one layer pass: reset, chunk forwards 0..D-1 over n_fwd streams,
        # chunk backwards D-1..0 over n_bwd streams; each pass is timed as a
        # phase on the main stream, from its fork to its join
        binding.reset_accum(bufs.dk, bufs.dv, w.hq)
        if events is not None:
            events["start"].record(main)
        binding.forward_chunks(q, k, v, c, bufs, None, main, n_fwd)
        if events is not None:
            events["fwd_end"].record(main)
        binding.backward_chunks(q, k, v, do, c, bufs, None, main, n_bwd)
        if events is not None:
            events["bwd_end"].record(main)

    if (T % c) != 0 or w.batch != 1:
        raise SystemExit("bench expects B=1 and T divisible by the chunk")

    for _ in range(args.warmup):
        step()
    binding.sync_status()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    launch_ev = [{"start": ev(), "fwd_end": ev(), "bwd_end": ev()} for _ in range(args.steps)]
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    t0.record()
    for kstep in range(args.steps):
        step(launch_ev[kstep])
    t1.record()
    torch.cuda.synchronize()
    dist.barrier()
    clock_info = clocks.stop()
    binding.sync_status()
    ms_local = t0.elapsed_time(t1)
    ms = dist.max_over_ranks(ms_local, device=dev)
    flops_rank = w.causal_flops()
    value = world * flops_rank * args.steps / (ms / 1e3) / 1e12

    # roofline of both passes, each timed as a phase of every timed step (live
    # CUDA events on the main stream, from the fork to the join of its streams)
    fwd_ms = sum(e["start"].elapsed_time(e["fwd_end"]) for e in launch_ev)
    bwd_ms = sum(e["fwd_end"].elapsed_time(e["bwd_end"]) for e in launch_ev)
    pairs = sum(workloads.causal_pairs(s, min(c, T - s)) for s in starts)
    fwd_flops = 4 * w.batch * w.hq * w.head_dim * pairs * args.steps
    bwd_flops = 10 * w.batch * w.hq * w.head_dim * pairs * args.steps
    pk = measured_peaks()
    peak = pk["burst"]
    bwd_tf = bwd_flops / (bwd_ms / 1e3) / 1e12
    fwd_tf = fwd_flops / (fwd_ms / 1e3) / 1e12
    # the step lasts tens of milliseconds at the clocks sampled below, so the
    # burst figure is the denominator; the sustained one is shown beside it
    roofline = {"kernel": "seqattn_chunk_bwd (row-statistics pre-pass + bwd_bf16_kernel)", "bound": "tensor",
                "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tf / peak,
                "peak_source": pk["source"] + ", burst",
                "peak_sustained": pk["sustained"], "frac_sustained": bwd_tf / pk["sustained"],
                "peak_sustained_sm_mhz": pk["sustained_sm_mhz"], "sm_mhz_timed": clock_info.get("sm_mhz"),
                "traffic": BWD_TRAFFIC_BYTES_PER_LAUNCH.get(w.name),
                "traffic_source": "ncu full capture of one mid-sequence backward launch (chunk 7 of 16)",
                "per_launch": f"causal bwd FLOPs 10*Hq*d*pairs(chunk) over the {D} chunk backwards of a "
                              f"step, timed as a phase ({n_bwd} stream(s), fork to join); avg_launch_ms is "
                              f"the phase divided by {D}",
                "bwd_streams": n_bwd,
                "avg_launch_ms": bwd_ms / (D * args.steps)}
    roofline_fwd = {"kernel": "seqattn_chunk_fwd (fwd_bf16_kernel)", "bound": "tensor", "achieved": fwd_tf,
                    "peak": peak, "unit": "TFLOP/s", "frac": fwd_tf / peak,
                    "frac_sustained": fwd_tf / pk["sustained"],
                    "per_phase": f"causal fwd FLOPs 4*Hq*d*pairs over the {D} chunk forwards of a step, "
                                 f"timed from the {n_fwd}-stream fork to the join",
                    "phase_ms": fwd_ms / args.steps}

    # end to end through the public API with pinned host buffers: inputs are
    # uploaded chunk by chunk ahead of the forward calls and every output
    # chunk is copied back as soon as it is final (last-to-first backward),
    # the copies running on side streams under the compute
    e2e = None
    if not args.no_e2e:
        h_in = [x.to("cpu").pin_memory() for x in (q, k, v, do)]
        hp = binding.HostLayerPass(*h_in, c, device=dev)
        h2d, d2h = hp.bytes_moved()
        for _ in range(max(1, args.warmup)):
            hp.run()
        torch.cuda.synchronize()
        dist.barrier()
        a, b = ev(), ev()
        a.record()
        for _ in range(args.steps):
            hp.run()
        b.record()
        torch.cuda.synchronize()
        dist.barrier()
        binding.sync_status()
        e2e_ms = dist.max_over_ranks(a.elapsed_time(b), device=dev)
        e2e = {"value": world * flops_rank * args.steps / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "api": "binding.HostLayerPass (pinned host in/out, copies overlapped with compute)"}
        del hp

    # the step after the path: the projections' weight gradients in the relay
    # (dW_q, dW_k, dW_v += H^(i)T dQ^(i), dK^(i), dV^(i) after chunk i's
    # backward), timed alone over one pass worth of chunks, with synthetic
    # hidden states H of d_model = Hq d columns; outside the headline metric
    wgrad = None
    if not args.no_wgrad:
        dm = w.hq * w.head_dim
        h = inputs.draw("h", seed, w.batch, w.seq, 1, dm, torch.bfloat16, dev)[:, :, 0].contiguous()
        dws = [torch.zeros((dm, n), device=dev) for n in (w.hq * w.head_dim, w.hkv * w.head_dim,
                                                         w.hkv * w.head_dim)]

        wstreams = binding.side_streams(dev, n_bwd + 5)[n_bwd - 1:]

        def wgrad_pass():
            # the relay's schedule (binding.layer_forward_backward): chunks
            # last to first, two streams per projection taken by alternate
            # chunks, forked from and joined into the main stream
            for r in wstreams:
                r.wait_stream(main)
            for n, i in enumerate(range(D - 1, -1, -1)):
                s = starts[i]
                e = min(s + c, T)
                for x, (g, dw) in enumerate(zip((bufs.dq, bufs.dk, bufs.dv), dws)):
                    binding.proj_wgrad(h, g, dw, s, e, wstreams[2 * x + n % 2])
            for r in wstreams:
                main.wait_stream(r)

        for _ in range(2):
            wgrad_pass()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record()
        for _ in range(args.steps):
            wgrad_pass()
        b.record()
        torch.cuda.synchronize()
        binding.sync_status()
        wg_ms = a.elapsed_time(b) / args.steps
        wg_flops = 2.0 * w.batch * w.seq * dm * (w.hq + 2 * w.hkv) * w.head_dim
        wgrad = {"metric": "projection weight-gradient TFLOP/s (dW_q, dW_k, dW_v of one pass)",
                 "value": wg_flops / (wg_ms / 1e3) / 1e12, "unit": UNIT, "ms_per_pass": wg_ms,
                 "d_model": dm, "kernels": "wgrad_bf16_kernel (tcgen05, g rounded to bf16 in the kernel, float32 accumulate)",
                 "streams": "the relay's schedule: two streams per projection, alternate chunks",
                 "launches_per_pass": 3 * D}
        del h, dws

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        G = w.hq // w.hkv
        f, s, desc = oracle_sample(w, w.seed, G)
        cpu_baseline = cpu_baseline_record(f / s / 1e12, s, desc)
        if not args.no_single_core:
            cpu_baseline["single_core"] = single_core_baseline()

    launches_per_step = 1 + D + 2 * D   # reset, fwd per chunk, (statistics pre-pass + bwd) per chunk
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w),
        "frac_of_peak": value / world / peak, "frac_of_sustained_peak": value / world / pk["sustained"],
        "roofline": roofline, "roofline_fwd": roofline_fwd,
        "cpu_baseline": cpu_baseline, "e2e": e2e, "wgrad": wgrad,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock_info,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.finalize()


def run_sweep(args, w):
    """Partition-size sweep (one GPU): the same T=16384 layer at every chunk
    size, each pass replayed from a CUDA graph so that small chunks measure
    the kernels rather than host launch overhead.  Prints one JSON line whose
    value is the smallest chunk's throughput, with the whole sweep and each
    size's overhead against the unchunked pass."""
    import torch

    from long_context_attention_seqattn_gb300 import binding, build, inputs

    torch.cuda.set_device(0)
    build.build()
    binding.load_library()
    q, k, v, do = inputs.layer_inputs(w, device="cuda")
    flops = w.causal_flops()
    rows = []
    for c in w.chunks:
        graph = binding.LayerGraph(q, k, v, do, c)
        for _ in range(args.warmup):
            graph.replay()
        binding.sync_status()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(args.steps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        binding.sync_status()
        ms = a.elapsed_time(b) / args.steps
        rows.append({"chunk": c, "num_chunks": (w.seq + c - 1) // c, "ms_per_step": ms,
                     "value": flops / (ms / 1e3) / 1e12, "gpu_launches_per_step": 1 + 3 * ((w.seq + c - 1) // c)})
        del graph
    base = next(r for r in rows if r["num_chunks"] == 1)
    for r in rows:
        r["time_vs_unchunked"] = r["ms_per_step"] / base["ms_per_step"]
    first = rows[0]
    peak = measured_peaks()["burst"]
    line = {"metric": METRIC, "value": first["value"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": first["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(w), chunk=first["chunk"], num_chunks=first["num_chunks"]),
            "frac_of_peak": first["value"] / peak, "sweep": rows,
            "gpu_launches": first["gpu_launches_per_step"] * args.steps}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.oracle_threads:
        # before the first NumPy import: the BLAS thread pool is sized once
        global ORACLE_THREADS
        ORACLE_THREADS = args.oracle_threads
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = str(args.oracle_threads)
    from long_context_attention_seqattn_gb300 import workloads
    w = workloads.WORKLOADS[args.workload or workloads.BENCH_WORKLOAD]
    if args.oracle_only:
        if args.oracle_threads == 1 and hasattr(os, "sched_setaffinity"):
            os.sched_setaffinity(0, {min(os.sched_getaffinity(0))})   # one core, before NumPy loads
        oracle_only(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    elif len(w.chunks) > 1:
        run_sweep(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
