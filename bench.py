#!/usr/bin/env python
"""Benchmark of the TurboQuant hot path on one B300 (or N replicas).

One step = the whole hot path over one batch: quantize the layer's K and V
caches (rotation, Lloyd-Max bucketing, QJL signs, packing) and run one GQA
decode step of attention over the compressed cache (query rotation, scores,
online softmax, rotated-domain V accumulation, split merge and unrotation).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama8b] [--bits 3]
    python bench.py --impl reference ...   # the float64 CPU oracle on host cores

Prints one JSON line.  N > 1 runs as torchrun ranks, each an independent
replica of the workload (weak scaling; the path has no exchange step).
"""

import argparse
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

METRIC = "decode-attn KV-tokens/s & % of 8 TB/s HBM roofline; quantize Mvectors/s"
UNIT = "KV-tokens/s"
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--bits", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the long-context decode sweep")
    ap.add_argument("--decode-only", action="store_true",
                    help="time tq_decode_attention alone (cold L2) on --workload / --batch; for profilers")
    ap.add_argument("--generic-only", action="store_true",
                    help="time tq_quantize and tq_search_topk (top-10) alone on --vectors unit-norm d = 1024 fp32 "
                         "vectors and --queries queries; for profilers")
    ap.add_argument("--vectors", type=int, default=262144)
    ap.add_argument("--queries", type=int, default=256)
    ap.add_argument("--quantize-only", action="store_true",
                    help="time tq_quantize_pair alone (K and V, one launch) on --workload / --batch; for profilers")
    ap.add_argument("--append-only", action="store_true",
                    help="time tq_append_kv (one new key and value per batch row and kv head, into full caches) "
                         "followed by tq_decode_attention on --workload / --batch")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch size (0: keep)")
    ap.add_argument("--oracle-rate", type=float, default=0.0, help=argparse.SUPPRESS)  # child of the CPU baseline
    return ap.parse_args()


def rec_bytes(d, m, w):
    return (w * d + m) // 8 + 8


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


# The files that decide what a profiled kernel does per launch: its own
# translation unit, the file that dispatches and launches it, and the shared
# internal headers.  A DRAM-traffic record stays valid while these hash the same.
KERNEL_SOURCES = {
    "quantize_tc_kernel": ("tq_quantize_tc.cu", "tq_quantize.cu"),
    "decode_tc_kernel": ("tq_decode_tc.cu", "tq_decode.cu"),
}
SHARED_SOURCES = ("tq_internal.h", "tq_sm100.cuh")


def kernel_sources_sha(kernel, csrc=None):
    """First 16 hex digits of the SHA-256 of a kernel's source files (KERNEL_SOURCES)."""
    csrc = csrc or os.path.join(ROOT, "online_kv_cache_04_b300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel] + SHARED_SOURCES:
        h.update(f.encode() + b"\0")
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel, workload, record=None, csrc=None):
    """DRAM bytes per launch from the committed ncu summary, if taken on the kernel's current sources."""
    path = record or os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if kernel not in KERNEL_SOURCES or not os.path.exists(path):
        return None
    sha = kernel_sources_sha(kernel, csrc)
    for line in open(path):
        v = line.split()
        if len(v) == 4 and not line.startswith("#") and v[0] == kernel and v[1] == sha and v[3] == workload:
            return float(v[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms.  Polling every
    50 ms slowed the timed step by about 30 % on a B300 (0.187 ms against 0.143 ms
    unsampled, and 0.143-0.147 ms at 200 and 1000 ms), so the interval stays long."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=200):
        self.index = index
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def wait_first(self, timeout=5.0):
        """Block until nvidia-smi has written its first sample (it starts slowly)."""
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < timeout:
            self.file.flush()
            if os.path.getsize(self.file.name) > 0:
                return
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            v = [x.strip() for x in line.split(",")]
            if len(v) < 9:
                continue
            try:
                sm.append(float(v[1]))
                smax.append(float(v[2]))
            except ValueError:
                continue
            for name, flag in zip(names, v[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- oracle arm

def sampled(index, fn):
    """fn() with the GPU's clocks sampled (every 200 ms) over its run: (result, clocks)."""
    sampler = ClockSampler(index, interval_ms=200)
    sampler.wait_first()
    out = fn()
    return out, sampler.stop()


def oracle_step(wl, w, heads, T):
    """The float64 oracle on `heads` kv heads x T tokens of batch row 0: quantize K, V, then decode."""
    import numpy as np

    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED, make_kv, make_queries
    from oracle import codebook, decode, qjl, quantize, rotation

    d = wl.d
    Pi = rotation.make_rotation(d, ROTATION_SEED)
    S = qjl.make_qjl(wl.m, d, QJL_SEED)
    c, b, _, _ = codebook.lloyd_max(d, w)
    K = make_kv(wl, B=1, T=T, which=0)[:, :heads].float().numpy()
    V = make_kv(wl, B=1, T=T, which=1)[:, :heads].float().numpy()
    G = wl.Hq // wl.Hkv
    q = make_queries(wl, B=1)[:, :heads * G].float().numpy()

    def run():
        recs = []
        for X in (K, V):
            z = quantize.quantize(X.reshape(-1, d), Pi, S, c, b)
            recs.append({"idx": z.idx.reshape(1, heads, T, d), "sgn": z.sgn.reshape(1, heads, T, wl.m),
                         "norm": z.norm.reshape(1, heads, T), "rnorm": z.rnorm.reshape(1, heads, T)})
        decode.decode_attention(q, recs[0], recs[1], np.array([T]), Pi, S, c)

    return run, T * heads / wl.Hkv  # KV tokens of the full layer that one run stands for


def cpu_cores():
    """(BLAS threads of this process, host CPUs).  Without threadpoolctl the pool
    size is the one the environment sets, else OpenBLAS's default: every CPU this
    process may run on."""
    avail = len(os.sched_getaffinity(0))
    try:
        from threadpoolctl import threadpool_info

        blas = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:
        env = [os.environ.get(v) for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")]
        blas = next((int(e) for e in env if e and e.isdigit()), avail)
    return blas, os.cpu_count()


def oracle_rate(wl, w, budget):
    """KV tokens/s of the oracle (oracle_sample runs repeated for about budget s)."""
    run, tokens, Ts = oracle_sample(wl, w, 3.0)
    run()
    n, t0 = 0, time.perf_counter()
    while n < 3 or time.perf_counter() - t0 < budget:
        run()
        n += 1
    return tokens / ((time.perf_counter() - t0) / n), n, Ts


def oracle_rate_in_child(args, threads, budget):
    """oracle_rate in a fresh process whose BLAS pool has `threads` threads (set
    through the environment before numpy loads); returns (value, runs, T, threads)."""
    env = dict(os.environ)
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""  # the oracle runs on the host alone
    out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-rate", str(budget),
                          "--workload", args.workload, "--bits", str(args.bits)],
                         env=env, capture_output=True, text=True, check=True)
    r = json.loads(out.stdout.strip().splitlines()[-1])
    return r["value"], r["runs"], r["T"], r["threads"]


def oracle_sample(wl, w, budget_s):
    """(run, tokens, T) with T tokens of one kv head chosen so one run takes about budget_s."""
    probe_T = 1024
    run, _ = oracle_step(wl, w, 1, probe_T)
    run()
    t0 = time.perf_counter()
    run()
    per_token = (time.perf_counter() - t0) / probe_T
    T = int(max(128, min(wl.ctx, budget_s / max(per_token, 1e-9))) // 128 * 128)
    run, tokens = oracle_step(wl, w, 1, T)
    return run, tokens, T


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from online_kv_cache_04_b300.workloads import WORKLOADS

    wl = WORKLOADS[args.workload]
    w = args.bits - 1
    # the whole --warmup/--steps run stays within about two minutes of host time
    budget = min(10.0, 120.0 / max(1, args.steps + args.warmup))
    run, tokens, T = oracle_sample(wl, w, budget)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = tokens / dt
    threads, cores = cpu_cores()
    sample = (f"1 of {wl.Hkv} kv heads x first {T} of {wl.ctx} tokens (batch row 0) per step, "
              f"scaled to the layer's KV tokens")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, args.bits),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "host_cpus": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(times, world, device):
    """Each time (seconds) maximised over the ranks of the default process group.

    Every rank must call it with a list of the same length; with one rank the
    list comes back unchanged.
    """
    times = [float(t) for t in times]
    if world <= 1:
        return times
    import torch
    import torch.distributed as dist

    tt = torch.tensor(times, dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return [float(t) for t in tt.cpu().tolist()]


def job_throughput(units_per_rank, world, seconds):
    """Whole-job rate: the units all replicas processed over the slowest replica's time."""
    return units_per_rank * world / seconds


def workload_config(wl, bits):
    return {"workload": (f"{wl.name}: B={wl.B}, Hq={wl.Hq}, Hkv={wl.Hkv}, d={wl.d}, m={wl.m}, ctx={wl.ctx}, "
                         f"b={bits}, K/V {str(wl.dtype).replace('torch.', '')}"),
            "step": "quantize K and V caches + one GQA decode step over the compressed cache",
            "l2": "flushed between timed steps (256 MiB write)"}


# --------------------------------------------------------------------- GPU arm

def timed(stream, fn, iters, flush=None):
    """Mean device ms of fn() over iters calls, each preceded (untimed) by an L2 flush.

    Everything is enqueued first and synchronised once, so that the host's
    launch work for a call overlaps the flush before it instead of leaving the
    device idle inside the timed interval."""
    import torch

    # a bounded spin (about 0.1 s) at the head of the queue: the host enqueues
    # every call before the device reaches the first one
    torch.cuda._sleep(200_000_000)
    ev = []
    for _ in range(iters):
        if flush is not None:
            flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in ev) / iters


def decode_sweep(_lib, plan_cache, stream, flush, bits_list, iters=20):
    """Decode-only timing on the long-context batch (B=16, ctx 131072, 8 kv heads, GQA 4:1)."""
    import torch

    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED, WORKLOADS, make_kv, make_queries

    wl = WORKLOADS["longctx"]
    d, m = wl.d, wl.m
    B, Hq, Hkv, T = wl.B, wl.Hq, wl.Hkv, wl.ctx
    res = []
    for bits in bits_list:
        w = bits - 1
        plan = plan_cache.setdefault(w, _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED))
        Kr = _lib.Records(B * Hkv * T, d, m, w)
        Vr = _lib.Records(B * Hkv * T, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
        for which, rec in ((0, Kr), (1, Vr)):
            for b0 in range(0, B, 4):
                X = make_kv(wl, B=4, which=which, device="cuda")
                _lib.tq_quantize(plan, X.reshape(-1, d), rec, out_offset=b0 * Hkv * T)
                del X
        q = make_queries(wl, device="cuda")
        ctx = torch.full((B,), T, dtype=torch.int32, device="cuda")
        out = torch.empty(B, Hq, d, device="cuda")
        ws = torch.empty(_lib.tq_decode_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
        fn = lambda: _lib.tq_decode_attention(plan, q, Kr, Vr, ctx, T, Hkv, out, ws)
        for _ in range(3):
            fn()
        ms = timed(stream, fn, iters, flush)
        rb = rec_bytes(d, m, w)
        nbytes = 2 * B * Hkv * T * rb + q.numel() * q.element_size() + out.numel() * 4
        res.append({"bits": bits, "ms_per_call": ms, "bytes_per_call": nbytes, "gbs": nbytes / ms / 1e6,
                    "frac_of_8tbs": nbytes / ms / 1e6 / NOMINAL_HBM_GBS, "kv_tokens_per_s": B * T / ms * 1e3,
                    "l2": "flushed before every call"})
        del Kr, Vr, ws
        torch.cuda.empty_cache()
    return res


def config_sweep(_lib, stream, flush, peak):
    """The two quantize-heavy configurations: bulk prefill quantization (8 kv heads x 65536
    tokens x {K, V}, bf16, b = 3) and generic d = 1024 vectors (1,048,576 unit-norm fp32, b = 4,
    m = 1024) with a top-10 inner-product search for 1024 queries over the compressed set."""
    import torch

    from online_kv_cache_04_b300.workloads import (QJL_SEED, ROTATION_SEED, WORKLOADS, make_generic,
                                                   make_generic_queries, make_kv)

    out = {}
    # bulk prefill: keys by row, values in 32-row blocks, one paired launch
    wl = WORKLOADS["prefill"]
    d, m, w = wl.d, wl.m, 2
    nvec = wl.B * wl.Hkv * wl.ctx
    plan = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    K = make_kv(wl, which=0, device="cuda").reshape(nvec, d)
    V = make_kv(wl, which=1, device="cuda").reshape(nvec, d)
    Kr = _lib.Records(nvec, d, m, w)
    Vr = _lib.Records(nvec, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    fn = lambda: _lib.tq_quantize_pair(plan, K, V, Kr, Vr)
    for _ in range(3):
        fn()
    ms = timed(stream, fn, 20, flush)
    nbytes = 2 * nvec * (d * K.element_size() + rec_bytes(d, m, w))
    out["prefill_quantize"] = {"workload": "8 kv heads x 65536 tokens x {K, V}, bf16, b=3", "vectors": 2 * nvec,
                               "ms_per_call": ms, "mvec_per_s": 2 * nvec / ms / 1e3, "gbs": nbytes / ms / 1e6,
                               "frac_of_measured_hbm": nbytes / ms / 1e6 / peak, "l2": "flushed before every call"}
    del K, V, Kr, Vr
    torch.cuda.empty_cache()
    # generic d = 1024: quantize, then search
    wl = WORKLOADS["generic"]
    d, m, w, n, nq, k = wl.d, wl.m, 3, wl.ctx, wl.n_queries, 10
    plan = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    X = make_generic(wl, device="cuda")
    rec = _lib.Records(n, d, m, w)
    fn = lambda: _lib.tq_quantize(plan, X, rec)
    fn()
    ms = timed(stream, fn, 3, flush)
    rb = rec_bytes(d, m, w)
    nbytes = n * (d * 4 + rb)
    out["generic_quantize"] = {"workload": "1,048,576 unit-norm fp32 vectors, d=m=1024, b=4", "vectors": n,
                               "ms_per_call": ms, "mvec_per_s": n / ms / 1e3, "gbs": nbytes / ms / 1e6,
                               "frac_of_measured_hbm": nbytes / ms / 1e6 / peak, "l2": "flushed before every call"}
    del X
    torch.cuda.empty_cache()
    Q = make_generic_queries(wl, device="cuda")
    ws = torch.empty(_lib.tq_search_workspace_size(plan, nq, n, k), dtype=torch.uint8, device="cuda")
    idx = torch.empty(nq, k, dtype=torch.int32, device="cuda")
    sc = torch.empty(nq, k, dtype=torch.float32, device="cuda")
    fn = lambda: _lib.tq_search_topk(plan, Q, rec, n, k, idx, sc, ws)
    fn()
    ms = timed(stream, fn, 3, flush)
    out["generic_search"] = {"workload": "top-10 of 1,048,576 compressed d=1024 vectors for 1024 queries",
                             "ms_per_call": ms, "queries_per_s": nq / ms * 1e3,
                             "vector_queries_per_s": nq * n / ms * 1e3, "l2": "flushed before every call"}
    del Q, ws, rec
    torch.cuda.empty_cache()
    # stage 1 alone (m = 0) at b = 3 = w on the Llama-3.1-8B-shaped layer: general kernels
    wl = WORKLOADS["llama8b"]
    d, w = wl.d, 3
    B, Hq, Hkv, T = wl.B, wl.Hq, wl.Hkv, wl.ctx
    nvec = B * Hkv * T
    plan = _lib.Plan(d, 0, w, ROTATION_SEED, QJL_SEED)
    K = make_kv(wl, which=0, device="cuda").reshape(nvec, d)
    V = make_kv(wl, which=1, device="cuda").reshape(nvec, d)
    Kr = _lib.Records(nvec, d, 0, w)
    Vr = _lib.Records(nvec, d, 0, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    fq = lambda: _lib.tq_quantize_pair(plan, K, V, Kr, Vr)
    fq()
    ms_q = timed(stream, fq, 10, flush)
    from online_kv_cache_04_b300.workloads import make_queries

    q = make_queries(wl, device="cuda")
    ctx = torch.full((B,), T, dtype=torch.int32, device="cuda")
    o = torch.empty(B, Hq, d, device="cuda")
    ws = torch.empty(_lib.tq_decode_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    fd = lambda: _lib.tq_decode_attention(plan, q, Kr, Vr, ctx, T, Hkv, o, ws)
    fd()
    ms_d = timed(stream, fd, 20, flush)
    rb = d * w // 8 + 4
    out["stage1_only_llama8b"] = {"workload": "Llama-3.1-8B-shaped layer, stage 1 alone (m=0), b=w=3, tensor-core kernels",
                                  "quantize_ms_per_call": ms_q, "quantize_mvec_per_s": 2 * nvec / ms_q / 1e3,
                                  "decode_ms_per_call": ms_d, "decode_kv_tokens_per_s": B * T / ms_d * 1e3,
                                  "decode_gbs": 2 * nvec * rb / ms_d / 1e6, "l2": "flushed before every call"}
    del K, V, Kr, Vr, ws
    torch.cuda.empty_cache()
    out["llama8b_b4"] = llama_step_at(_lib, stream, flush, peak, 4)
    out["split_2p5bit_llama8b"] = split_config(_lib, stream, flush)
    out["polar_llama8b"] = polar_config(_lib, stream, flush)
    return out


def llama_step_at(_lib, stream, flush, peak, bits):
    """The Llama-3.1-8B-shaped layer at another bit width: paired quantize and decode, each alone."""
    import torch

    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED, WORKLOADS, make_kv, make_queries

    wl = WORKLOADS["llama8b"]
    d, m, w = wl.d, wl.m, bits - 1
    B, Hq, Hkv, T = wl.B, wl.Hq, wl.Hkv, wl.ctx
    nvec = B * Hkv * T
    plan = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    K = make_kv(wl, which=0, device="cuda").reshape(nvec, d)
    V = make_kv(wl, which=1, device="cuda").reshape(nvec, d)
    Kr = _lib.Records(nvec, d, m, w)
    Vr = _lib.Records(nvec, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    fq = lambda: _lib.tq_quantize_pair(plan, K, V, Kr, Vr)
    fq()
    ms_q = timed(stream, fq, 50, flush)
    q = make_queries(wl, device="cuda")
    ctx = torch.full((B,), T, dtype=torch.int32, device="cuda")
    o = torch.empty(B, Hq, d, device="cuda")
    ws = torch.empty(_lib.tq_decode_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    fd = lambda: _lib.tq_decode_attention(plan, q, Kr, Vr, ctx, T, Hkv, o, ws)
    fd()
    ms_d = timed(stream, fd, 50, flush)
    rb = rec_bytes(d, m, w)
    qb = 2 * nvec * (d * K.element_size() + rb)
    db = 2 * nvec * rb + q.numel() * q.element_size() + o.numel() * 4
    res = {"workload": f"Llama-3.1-8B-shaped layer (B=1, 32/8 heads, ctx 32768), b={bits}",
           "quantize_ms_per_call": ms_q, "quantize_gbs": qb / ms_q / 1e6, "quantize_frac_of_measured_hbm":
           qb / ms_q / 1e6 / peak, "decode_ms_per_call": ms_d, "decode_gbs": db / ms_d / 1e6,
           "decode_frac_of_8tbs": db / ms_d / 1e6 / NOMINAL_HBM_GBS, "decode_kv_tokens_per_s": B * T / ms_d * 1e3,
           "l2": "flushed before every call"}
    del K, V, Kr, Vr, ws
    torch.cuda.empty_cache()
    return res


def split_config(_lib, stream, flush):
    """Outlier-channel split at 2.5 bits per coordinate on the Llama-3.1-8B-shaped layer: the 64
    channels of largest mean square over the layer's keys (values) at 3 bits, the rest at 2."""
    import numpy as np
    import torch

    from online_kv_cache_04_b300.workloads import SPLIT_SEEDS, WORKLOADS, make_kv, make_queries

    wl = WORKLOADS["llama8b"]
    d, no, bits = wl.d, 64, 2
    B, Hq, Hkv, T = wl.B, wl.Hq, wl.Hkv, wl.ctx
    nvec = B * Hkv * T
    (ro, qo), (rr, qr) = SPLIT_SEEDS["outlier"], SPLIT_SEEDS["regular"]
    po, pr = _lib.Plan(no, no, bits, ro, qo), _lib.Plan(d - no, d - no, bits - 1, rr, qr)
    K = make_kv(wl, which=0, device="cuda").reshape(nvec, d)
    V = make_kv(wl, which=1, device="cuda").reshape(nvec, d)

    def perm_of(X):  # channels by mean square over a sample, largest first (ties to the lower channel)
        ms2 = (X[::64].float() ** 2).mean(dim=0).cpu().numpy()
        order = sorted(range(d), key=lambda j: (-ms2[j], j))
        p = np.concatenate([np.sort(order[:no]), np.sort(order[no:])]).astype(np.int32)
        return torch.from_numpy(p).cuda()

    pk, pv = perm_of(K), perm_of(V)
    Ko, Kr = _lib.Records(nvec, no, no, bits), _lib.Records(nvec, d - no, d - no, bits - 1)
    Vo, Vr = _lib.Records(nvec, no, no, bits), _lib.Records(nvec, d - no, d - no, bits - 1)
    fq = lambda: (_lib.tq_quantize_split(po, pr, pk, K, Ko, Kr), _lib.tq_quantize_split(po, pr, pv, V, Vo, Vr))
    fq()
    ms_q = timed(stream, fq, 10, flush)
    q = make_queries(wl, device="cuda")
    ctx = torch.full((B,), T, dtype=torch.int32, device="cuda")
    o = torch.empty(B, Hq, d, device="cuda")
    ws = torch.empty(_lib.tq_decode_split_workspace_size(po, pr, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    fd = lambda: _lib.tq_decode_attention_split(po, pr, pk, pv, q, Ko, Kr, Vo, Vr, ctx, T, Hkv, o, ws)
    fd()
    ms_d = timed(stream, fd, 20, flush)
    rec = (no * bits + no) // 8 + 8 + ((d - no) * (bits - 1) + (d - no)) // 8 + 8
    res = {"workload": "Llama-3.1-8B-shaped layer, 64 of 128 channels at 3 bits, the rest at 2 (2.5 bit/coord), "
                       "keys and values with their own outlier channels, general kernels",
           "record_bytes_per_vector": rec, "quantize_ms_per_call": ms_q, "quantize_mvec_per_s": 2 * nvec / ms_q / 1e3,
           "decode_ms_per_call": ms_d, "decode_kv_tokens_per_s": B * T / ms_d * 1e3,
           "decode_gbs": 2 * nvec * rec / ms_d / 1e6, "l2": "flushed before every call"}
    del K, V, Ko, Kr, Vo, Vr, ws
    torch.cuda.empty_cache()
    return res


def polar_config(_lib, stream, flush):
    """PolarQuant stage (+ QJL) on the Llama-3.1-8B-shaped layer: 4-bit first level, 2-bit later levels."""
    import torch

    from online_kv_cache_04_b300.workloads import POLAR_SEEDS, WORKLOADS, make_kv, make_queries

    wl = WORKLOADS["llama8b"]
    d = wl.d
    B, Hq, Hkv, T = wl.B, wl.Hq, wl.Hkv, wl.ctx
    nvec = B * Hkv * T
    plan = _lib.PolarPlan(d, d, 4, 2, *POLAR_SEEDS)
    K = make_kv(wl, which=0, device="cuda").reshape(nvec, d)
    V = make_kv(wl, which=1, device="cuda").reshape(nvec, d)
    Kr, Vr = plan.records(nvec), plan.records(nvec)
    fq = lambda: (_lib.tq_quantize_polar(plan, K, Kr), _lib.tq_quantize_polar(plan, V, Vr))
    fq()
    ms_q = timed(stream, fq, 10, flush)
    q = make_queries(wl, device="cuda")
    ctx = torch.full((B,), T, dtype=torch.int32, device="cuda")
    o = torch.empty(B, Hq, d, device="cuda")
    ws = torch.empty(_lib.tq_decode_polar_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    fd = lambda: _lib.tq_decode_attention_polar(plan, q, Kr, Vr, ctx, T, Hkv, o, ws)
    fd()
    ms_d = timed(stream, fd, 20, flush)
    rec = 4 * plan.nw + d // 8 + 8
    res = {"workload": "Llama-3.1-8B-shaped layer, polar stage (4-bit level 1, 2-bit later levels) + QJL, "
                       "general kernels", "record_bytes_per_vector": rec,
           "quantize_ms_per_call": ms_q, "quantize_mvec_per_s": 2 * nvec / ms_q / 1e3,
           "decode_ms_per_call": ms_d, "decode_kv_tokens_per_s": B * T / ms_d * 1e3,
           "decode_gbs": 2 * nvec * rec / ms_d / 1e6, "l2": "flushed before every call"}
    del K, V, Kr, Vr, ws
    torch.cuda.empty_cache()
    return res


def run_generic(args):
    """Generic d = m = 1024, b = 4 vectors: quantize and top-10 search alone (the command profilers capture)."""
    import torch

    from online_kv_cache_04_b300 import _lib
    from online_kv_cache_04_b300.workloads import (QJL_SEED, ROTATION_SEED, WORKLOADS, make_generic,
                                                   make_generic_queries)

    wl = WORKLOADS["generic"]
    d, m, w, n, nq, k = wl.d, wl.m, 3, args.vectors, args.queries, 10
    plan = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    X = make_generic(wl, n=n, device="cuda")
    rec = _lib.Records(n, d, m, w)
    Q = make_generic_queries(wl, nq=nq, device="cuda")
    ws = torch.empty(_lib.tq_search_workspace_size(plan, nq, n, k), dtype=torch.uint8, device="cuda")
    idx = torch.empty(nq, k, dtype=torch.int32, device="cuda")
    sc = torch.empty(nq, k, dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    fq = lambda: _lib.tq_quantize(plan, X, rec)
    fs = lambda: _lib.tq_search_topk(plan, Q, rec, n, k, idx, sc, ws)
    for _ in range(args.warmup):
        fq()
        fs()
    ms_q = timed(stream, fq, args.steps, flush)
    ms_s = timed(stream, fs, args.steps, flush)
    print(json.dumps({"mode": "generic quantize + search", "vectors": n, "queries": nq,
                      "quantize_ms": ms_q, "quantize_mvec_per_s": n / ms_q / 1e3,
                      "search_ms": ms_s, "vector_queries_per_s": n * nq / ms_s * 1e3,
                      "fault_flags": _lib.tq_fault_flags()}), flush=True)


def run_single(args):
    """One kernel family alone on a (possibly smaller) workload: the command profilers capture."""
    import dataclasses

    import torch

    from online_kv_cache_04_b300 import _lib
    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED, WORKLOADS, make_kv, make_queries

    wl = WORKLOADS[args.workload]
    if args.batch:
        wl = dataclasses.replace(wl, B=args.batch)
    w = args.bits - 1
    d, m = wl.d, wl.m
    B, Hq, Hkv, T = wl.B, wl.Hq, wl.Hkv, wl.ctx
    nvec = B * Hkv * T
    plan = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    Kr = _lib.Records(nvec, d, m, w)
    Vr = _lib.Records(nvec, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rb = rec_bytes(d, m, w)
    if args.quantize_only:
        K = make_kv(wl, which=0, device="cuda").reshape(nvec, d)
        V = make_kv(wl, which=1, device="cuda").reshape(nvec, d)
        fn = lambda: _lib.tq_quantize_pair(plan, K, V, Kr, Vr)
        nbytes = 2 * nvec * (rb + d * K.element_size())
        what = "quantize K and V"
    else:
        for which, rec in ((0, Kr), (1, Vr)):
            X = make_kv(wl, which=which, device="cuda").reshape(nvec, d)
            _lib.tq_quantize(plan, X, rec)
            del X
        q = make_queries(wl, device="cuda")
        if args.append_only:
            run_append_step(args, _lib, plan, wl, Kr, Vr, q, stream, flush)
            return
        ctx = torch.full((B,), T, dtype=torch.int32, device="cuda")
        out = torch.empty(B, Hq, d, device="cuda")
        ws = torch.empty(_lib.tq_decode_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
        fn = lambda: _lib.tq_decode_attention(plan, q, Kr, Vr, ctx, T, Hkv, out, ws)
        nbytes = 2 * nvec * rb
        what = "decode attention"
    for _ in range(args.warmup):
        fn()
    ms = timed(stream, fn, args.steps, flush)
    print(json.dumps({"mode": what, "workload": f"{wl.name} B={B}", "bits": args.bits, "ms": ms,
                      "bytes": nbytes, "gbs": nbytes / ms / 1e6, "fault_flags": _lib.tq_fault_flags()}),
          flush=True)


def run_append_step(args, _lib, plan, wl, Kr, Vr, q, stream, flush):
    """A decode step with its online append: tq_append_kv writes token ctx-1 of every (batch row,
    kv head) and advances the lengths to ctx, then tq_decode_attention reads the whole cache."""
    import torch

    from online_kv_cache_04_b300.workloads import make_kv

    B, Hq, Hkv, T, d = wl.B, wl.Hq, wl.Hkv, wl.ctx, wl.d
    kn = make_kv(wl, B=B, T=1, which=0, device="cuda")[:, :, 0].contiguous()  # [B, Hkv, d]
    vn = make_kv(wl, B=B, T=1, which=1, device="cuda")[:, :, 0].contiguous()
    ctx = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, Hq, d, device="cuda")
    ws = torch.empty(_lib.tq_decode_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    evs = []
    n_iter = max(args.warmup, 3) + args.steps
    # a bounded spin (about 0.1 s) at the head of the queue lets the host enqueue every
    # step before the device reaches the first, so no host time lands inside a timed interval
    torch.cuda._sleep(200_000_000)
    for i in range(n_iter):
        ctx.fill_(T - 1)  # outside the timed interval, like the L2 flush
        flush.fill_(1)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        _lib.tq_append_kv(plan, kn, vn, Kr, Vr, ctx, T)
        e[1].record(stream)
        _lib.tq_decode_attention(plan, q, Kr, Vr, ctx, T, Hkv, out, ws)
        e[2].record(stream)
        if i >= max(args.warmup, 3):
            evs.append(e)
    # the same step with the append fused into the decode's launches
    fused = []
    torch.cuda._sleep(200_000_000)
    for i in range(n_iter):
        ctx.fill_(T - 1)
        flush.fill_(1)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        _lib.tq_decode_attention_append(plan, q, kn, vn, Kr, Vr, ctx, T, Hkv, out, ws)
        e[1].record(stream)
        if i >= max(args.warmup, 3):
            fused.append(e)
    torch.cuda.synchronize()
    t_app = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)
    t_dec = sum(e[1].elapsed_time(e[2]) for e in evs) / len(evs)
    t_fused = sum(e[0].elapsed_time(e[1]) for e in fused) / len(fused)
    print(json.dumps({"mode": "append one key and value per (batch row, kv head), then decode",
                      "workload": f"{wl.name} B={B}", "bits": args.bits, "appended_vectors": 2 * B * Hkv,
                      "append_ms": t_app, "decode_ms": t_dec, "step_ms": t_app + t_dec,
                      "fused_step_ms": t_fused, "ctx_after": int(ctx[0].item()),
                      "fault_flags": _lib.tq_fault_flags(), "l2": "flushed before every step"}), flush=True)


def main():
    args = parse()
    if args.oracle_rate > 0:
        from online_kv_cache_04_b300.workloads import WORKLOADS

        value, runs, T = oracle_rate(WORKLOADS[args.workload], args.bits - 1, args.oracle_rate)
        print(json.dumps({"value": value, "runs": runs, "T": T, "threads": cpu_cores()[0]}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.generic_only:
        run_generic(args)
        return
    if args.decode_only or args.quantize_only or args.append_only:
        run_single(args)
        return
    import torch
    import torch.distributed as dist

    from online_kv_cache_04_b300 import _lib
    from online_kv_cache_04_b300.workloads import QJL_SEED, ROTATION_SEED, WORKLOADS, make_kv, make_queries

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    wl = WORKLOADS[args.workload]
    w = args.bits - 1
    d, m = wl.d, wl.m
    B, Hq, Hkv, T = wl.B, wl.Hq, wl.Hkv, wl.ctx
    nvec = B * Hkv * T
    plan = _lib.Plan(d, m, w, ROTATION_SEED, QJL_SEED)
    K = make_kv(wl, which=0, device="cuda").reshape(nvec, d)
    V = make_kv(wl, which=1, device="cuda").reshape(nvec, d)
    q = make_queries(wl, device="cuda")
    # keys by row, values in 32-row blocks (the layout the tensor-core decode reads)
    Kr = _lib.Records(nvec, d, m, w)
    Vr = _lib.Records(nvec, d, m, w, layout=_lib.TQ_LAYOUT_BLOCK32)
    ws = torch.empty(_lib.tq_decode_workspace_size(plan, B, Hq, Hkv, T), dtype=torch.uint8, device="cuda")
    ctx = torch.full((B,), T, dtype=torch.int32, device="cuda")
    out = torch.empty(B, Hq, d, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(ev):
        ev[0].record(stream)
        _lib.tq_quantize_pair(plan, K, V, Kr, Vr)  # keys by row, values in blocks: one launch
        ev[1].record(stream)
        _lib.tq_decode_attention(plan, q, Kr, Vr, ctx, T, Hkv, out, ws)
        ev[2].record(stream)

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(max(args.warmup, 3)):
        step(mk())
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # decode alone with a cold L2 (inside the step it reads records that quantize just
    # wrote); taken before the clock sampler starts, apart from the timed steps
    t_dec, clk_cold = sampled(local, lambda: timed(
        stream, lambda: _lib.tq_decode_attention(plan, q, Kr, Vr, ctx, T, Hkv, out, ws), 50, flush))
    t_dec /= 1e3

    sampler = ClockSampler(local)
    sampler.wait_first()
    events = []
    for _ in range(args.steps):
        flush.fill_(1)
        ev = mk()
        step(ev)
        events.append(ev)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    t_step = sum(e[0].elapsed_time(e[2]) for e in events) / args.steps / 1e3
    t_quant = sum(e[0].elapsed_time(e[1]) for e in events) / args.steps / 1e3
    t_dec_step = sum(e[1].elapsed_time(e[2]) for e in events) / args.steps / 1e3
    fault = _lib.tq_fault_flags()

    # ---- end to end: pinned host inputs in, attention output out, every step
    Kh = K.cpu().pin_memory()
    Vh = V.cpu().pin_memory()
    qh = q.cpu().pin_memory()
    outh = torch.empty_like(out, device="cpu").pin_memory()
    Kd, Vd, qd = torch.empty_like(K), torch.empty_like(V), torch.empty_like(q)

    def e2e_step():
        Kd.copy_(Kh, non_blocking=True)
        Vd.copy_(Vh, non_blocking=True)
        qd.copy_(qh, non_blocking=True)
        _lib.tq_quantize_pair(plan, Kd, Vd, Kr, Vr)
        _lib.tq_decode_attention(plan, qd, Kr, Vr, ctx, T, Hkv, out, ws)
        outh.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps // 2, 50))
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = e0.elapsed_time(e1) / n_e2e / 1e3
    h2d = (Kh.numel() + Vh.numel()) * Kh.element_size() + qh.numel() * qh.element_size()
    d2h = outh.numel() * outh.element_size()

    # ---- end to end, a decode loop: the step's query and new key and value in,
    # appended to the compressed cache (at token T - 1), attention over it, output out
    # The step's inputs travel as one pinned staging buffer (query, new key, new
    # value and the context lengths, each at a 256-byte offset) in one copy; the
    # lengths are the same every step: a fixed-size benchmark cache.
    kn_src = make_kv(wl, T=1, which=0)[:, :, 0].contiguous()  # [B, Hkv, d]
    vn_src = make_kv(wl, T=1, which=1)[:, :, 0].contiguous()
    ctx_src = torch.full((B,), T - 1, dtype=torch.int32)
    parts = [qh, kn_src, vn_src, ctx_src]
    offs, o = [], 0
    for t in parts:
        offs.append(o)
        o += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(o, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(o, dtype=torch.uint8, device="cuda")

    def view(buf, i):
        t = parts[i]
        n = t.numel() * t.element_size()
        return buf[offs[i]:offs[i] + n].view(t.dtype).view(t.shape)

    for i, t in enumerate(parts):
        view(stage_h, i).copy_(t)
    qs_d, kn_d, vn_d, ctx_d = (view(stage_d, i) for i in range(4))

    def loop_step():
        stage_d.copy_(stage_h, non_blocking=True)
        _lib.tq_decode_attention_append(plan, qs_d, kn_d, vn_d, Kr, Vr, ctx_d, T, Hkv, out, ws)
        outh.copy_(out, non_blocking=True)

    for _ in range(3):
        loop_step()
    torch.cuda.synchronize()
    n_loop = max(10, min(args.steps, 200))
    torch.cuda._sleep(200_000_000)
    e0.record(stream)
    for _ in range(n_loop):
        loop_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_loop = e0.elapsed_time(e1) / n_loop / 1e3
    h2d_loop = stage_h.numel()
    # the job is as slow as its slowest replica (every rank joins the reduction)
    t_step, t_quant, t_dec_step, t_dec, t_e2e, t_loop = max_over_ranks(
        [t_step, t_quant, t_dec_step, t_dec, t_e2e, t_loop], world, "cuda")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    rb = rec_bytes(d, m, w)
    in_bytes = nvec * d * K.element_size()
    q_bytes = 2 * (rb * nvec + in_bytes)  # one quantize launch, keys and values: read x, write records
    dec_bytes = 2 * nvec * rb + q.numel() * q.element_size() + out.numel() * 4
    kernels = {
        "quantize": {"launches_per_step": 1, "ms_per_launch": t_quant * 1e3, "bytes_per_launch": q_bytes,
                     "gbs": q_bytes / t_quant / 1e9, "mvec_per_s": 2 * nvec / t_quant / 1e6},
        "decode_attention": {"launches_per_call": 1, "ms_per_call_in_step": t_dec_step * 1e3,
                             "ms_per_call_cold_l2": t_dec * 1e3, "bytes_per_call": dec_bytes,
                             "gbs_cold_l2": dec_bytes / t_dec / 1e9, "kv_tokens_per_s_cold_l2": B * T / t_dec,
                             "frac_of_8tbs_cold_l2": dec_bytes / t_dec / 1e9 / NOMINAL_HBM_GBS},
    }
    if t_quant >= t_dec_step:
        kname, ach, traffic_key = "quantize_tc_kernel", q_bytes / t_quant / 1e9, "quantize_tc_kernel"
    else:
        kname, ach, traffic_key = "decode_tc_kernel", dec_bytes / t_dec / 1e9, "decode_tc_kernel"
    traffic = dram_traffic(traffic_key, wl.name)
    line = {
        "metric": METRIC, "value": job_throughput(B * T, world, t_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(wl, args.bits),
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": ach, "peak": peak, "unit": "GB/s",
                     "frac": ach / peak, "peak_kind": peak_kind, "traffic": traffic},
        "kernels": kernels,
        "decode_kv_tokens_per_s": B * T / t_dec,
        "decode_frac_of_8tbs": dec_bytes / t_dec / 1e9 / NOMINAL_HBM_GBS,
        "quantize_mvec_per_s": 2 * nvec / t_quant / 1e6,
        "e2e": {"value": job_throughput(B * T, world, t_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "step": "pinned host K and V caches (bf16) and queries in, quantize + decode, output out"},
        "e2e_decode_loop": {"value": job_throughput(B * T, world, t_loop), "unit": UNIT,
                            "ms_per_step": t_loop * 1e3, "h2d_bytes_per_step": h2d_loop,
                            "d2h_bytes_per_step": d2h,
                            "step": ("pinned host query, the step's new key and value (bf16) and the context "
                                     "lengths in (one staging copy), "
                                     "tq_decode_attention_append (the append inside the decode's launches) "
                                     f"over the {T}-token compressed cache, output out")},
        "gpu_launches": 4 * args.steps,  # quantize pair; query tables, decode, merge
        "fault_flags": fault,
        "clocks": clocks,
        "clocks_regions": {"cold_decode": clk_cold},
    }
    if world == 1 and not args.no_sweep:
        line["decode_longctx"], line["clocks_regions"]["decode_longctx"] = sampled(
            local, lambda: decode_sweep(_lib, {}, stream, flush, (2, 3, 4)))
        line["configs"], line["clocks_regions"]["configs"] = sampled(
            local, lambda: config_sweep(_lib, stream, flush, peak))
    if world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count()
        v_all, n_all, Ts, threads = oracle_rate_in_child(args, len(os.sched_getaffinity(0)), 10.0)
        v_one, n_one, Ts1, _ = oracle_rate_in_child(args, 1, 10.0)
        sample = lambda n, t: (f"1 of {Hkv} kv heads x first {t} of {T} tokens (batch row 0), {n} runs, "
                               f"scaled to the layer's KV tokens")
        line["cpu_baseline"] = {"value": v_all, "unit": UNIT, "cores": threads, "host_cpus": cores, "kind": "oracle",
                                "sample": sample(n_all, Ts)}
        line["cpu_baseline_1core"] = {"value": v_one, "unit": UNIT, "cores": 1, "host_cpus": cores,
                                      "kind": "oracle", "sample": sample(n_one, Ts1)}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
