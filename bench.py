#!/usr/bin/env python
"""Throughput of the FA2 hot path (forward + backward) on GB300.

One step = the forward pass (fp16 copy of V, attention kernel) followed by
the three backward stages (D preprocess, main recompute kernel, dQ convert)
on one batch of synthetic inputs already resident in HBM.  Default workload: the long-sequence configuration
B=1, H=32, N=16384, d=128, causal (Q, K, V, dO are 134 MB each, so the
inputs of a step exceed the 129 MB L2 and no flush is needed).

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are weak-scaled:
every rank runs its own batch of the same shape; no data-path collective.
``--impl reference`` times the fp64 CPU oracle instead (the reference arm).
"""
from __future__ import annotations

import argparse
import itertools
import json
import os
import statistics
import subprocess
import sys
import threading
import time

_CORES = len(os.sched_getaffinity(0))
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

# One step: fa2_v_to_f16_kernel, fa2_v_scale_kernel, fa2_fwd_kernel, then the
# backward's preprocess, main kernel and dQ conversion (or ordered reduction);
# heads of at most 64K elements get their fp16 copy of V from one kernel
# (fa2_v_to_f16_head_kernel) instead of the first two.
def launches_per_step(N, d):
    return 5 if N * d <= 65536 else 6
METRIC = "causal bf16 FA2 fwd / bwd TFLOPS and % of GB300 dense bf16 peak (1 GPU)"

# DRAM bytes (read + write) per launch of a kernel on a workload, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum, one pass) of the
# kernel build whose device sources hash to the recorded digest; a figure
# whose digest no longer matches the sources is reported as null.
KERNEL_TRAFFIC = {
    # (kernel, workload, causal): (read + write bytes, digest of the sources).
    # Capture summarised in the DRAM-traffic profile of the long causal
    # workload (dram__bytes_read.sum + dram__bytes_write.sum, one launch each).
    ("fa2_fwd_kernel", "long", True): (407450880 + 117617664, "3d4c11422ef5c5e3"),
    ("fa2_bwd_kernel", "long", True): (836262656 + 505752832, "15c764e6e3932078"),
}

KERNEL_SOURCES = {
    "fa2_fwd_kernel": ("fa2_fwd.cu", "ptx.cuh", "tiles.cuh", "launch.h"),
    "fa2_bwd_kernel": ("fa2_bwd.cu", "ptx.cuh", "tiles.cuh", "launch.h"),
}


def kernel_digest(kernel):
    """sha256 (first 16 hex digits) over the device sources of a kernel."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "tiled_exact_attention_fa2_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel, workload, causal):
    entry = KERNEL_TRAFFIC.get((kernel, workload, causal))
    if entry is None or entry[1] != kernel_digest(kernel):
        return None
    return entry[0]


def algorithmic_bytes(kernel, B, H, N, d):
    """HBM bytes a kernel must move at least, per launch.

    Forward: read Q, K, V (bf16), write O (bf16) and LSE (fp32).  Backward
    main kernel: read Q, K, V, dO (bf16), LSE and D (fp32); write dK, dV
    (bf16) and the fp32 dQ accumulator once.
    """
    rows = B * H * N
    if kernel == "fa2_fwd_kernel":
        return rows * (4 * d * 2 + 4)
    return rows * (6 * d * 2 + d * 4 + 8)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": p["bf16_tflops"], "bf16_tflops_sustained": p["bf16_tflops_sustained"],
                "hbm_gbs": p["hbm_gbs"], "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def roofline_peak(timed_s, clocks):
    """Which measured bf16 peak a kernel timed in this run is held against.

    The burst figure (a GEMM timed alone) applies when the timed region is
    short and the sampled SM clock stayed at its maximum; the sustained one
    (seconds of back-to-back GEMMs under the power cap) when the region runs
    for seconds or the clock dropped below its maximum.
    """
    at_max = bool(clocks) and clocks.get("sm_max_mhz") and clocks["sm_mhz"] >= 0.97 * clocks["sm_max_mhz"]
    if timed_s < 2.0 and at_max:
        return "bf16_tflops", f"burst: timed region {timed_s:.2f} s at {clocks['sm_mhz']:.0f} MHz"
    why = f"timed region {timed_s:.2f} s" + ("" if at_max else ", SM clock below its maximum or not sampled")
    return "bf16_tflops_sustained", f"sustained: {why}"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

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
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        time.sleep(0.25)
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
            parts = [p.strip() for p in ln.split(",")]
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
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist(backend: str = "nccl"):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def _free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def spawn_local_replicas(n: int, argv, script: str = None) -> int:
    """Run ``python <script> <argv>`` as n local ranks, each with the
    environment torchrun gives one rank of one node (RANK = LOCAL_RANK = i,
    WORLD_SIZE = n, rendezvous on 127.0.0.1 at a free port), so rank i uses
    cuda:i.  Waits for all of them; returns 0, else the first non-zero exit
    code (the other ranks are then stopped, as torchrun does)."""
    script = script or os.path.abspath(__file__)
    port = str(_free_port())
    procs = []
    for i in range(n):
        env = dict(os.environ, RANK=str(i), LOCAL_RANK=str(i), WORLD_SIZE=str(n), LOCAL_WORLD_SIZE=str(n),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=port)
        procs.append(subprocess.Popen([sys.executable, script, *argv], env=env))
    rc = 0
    pending = list(procs)
    while pending:
        for p in list(pending):
            r = p.poll()
            if r is None:
                continue
            pending.remove(p)
            if r != 0 and rc == 0:
                rc = r
                for q in pending:
                    q.terminate()
        time.sleep(0.05)
    return rc


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's value (timing is max over ranks)."""
    if world == 1:
        return x
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(w, rank: int) -> int:
    """Weak scaling: every rank runs the same shape on its own inputs."""
    return w.seed + rank


def job_tflops(world: int, flops_per_rank: float, max_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * flops_per_rank / (max_ms * 1e-3) / 1e12


# --------------------------------------------------------------------------- CPU oracle legs
def _oracle_sample(w, causal: bool, n_prefix: int):
    """fp64 oracle forward + backward on the first n_prefix rows of head (0, 0).

    Returns (flops counted as FA2 work, seconds)."""
    import oracle
    x = workloads.make_inputs(1, 1, n_prefix, w.d, seed=w.seed, qk_mult=w.qk_mult)
    t0 = time.perf_counter()
    oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], w.scale, causal)
    dt = time.perf_counter() - t0
    flops = 14.0 * n_prefix * n_prefix * w.d * (0.5 if causal else 1.0)
    return flops, dt


def _choose_prefix(w, causal, budget_s: float) -> int:
    """Largest head prefix (multiple of 1024, <= N) whose oracle run fits budget_s."""
    base = min(2048, w.N)
    _, t = _oracle_sample(w, causal, base)
    n = base
    while n * 2 <= w.N and t * ((n * 2) / base) ** 2 <= budget_s:
        n *= 2
    for cand in range(n, min(w.N, 2 * n) + 1, 1024):
        if t * (cand / base) ** 2 <= budget_s:
            n = cand
    return min(n, w.N)


def cpu_baseline(w, causal):
    n = _choose_prefix(w, causal, budget_s=20.0)
    flops, dt = _oracle_sample(w, causal, n)
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": _CORES, "kind": "oracle",
            "sample": f"fp64 numpy oracle fwd+bwd on one head (b=0,h=0) of the {w.name} workload, "
                      f"first {n} of {w.N} rows{' (causal prefix)' if causal else ''}; {dt:.1f} s; "
                      f"BLAS threads {_CORES}"}


def run_reference(args, w, causal):
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = _choose_prefix(w, causal, budget)
    for _ in range(args.warmup):
        _oracle_sample(w, causal, n)
    tot_flops, tot_t = 0.0, 0.0
    for _ in range(args.steps):
        f, t = _oracle_sample(w, causal, n)
        tot_flops += f
        tot_t += t
    value = tot_flops / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: B={w.B} H={w.H} N={w.N} d={w.d} "
                               f"{'causal' if causal else 'non-causal'} (oracle on a head prefix per step)",
                   "sample_rows": n},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": _CORES, "kind": "oracle",
                         "sample": f"per step: fp64 oracle fwd+bwd on the first {n} rows of head (0,0)"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm
def _stats(xs):
    xs = sorted(xs)
    return {"mean": statistics.mean(xs), "median": statistics.median(xs), "min": xs[0],
            "p90": xs[min(len(xs) - 1, int(round(0.9 * (len(xs) - 1))))]}


def _time_ms(fn, stream, iters=10, warm=3):
    """Mean milliseconds of fn() over `iters` calls, CUDA events on `stream`."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def measure_rows(fa2, dev, stream, peaks, only=None):
    """Throughput of the rows beside the headline workload: the N = 4096
    workloads (large-logit stress and B=4, H=32), launch latency of the tiny
    and small workloads, grouped-query prefill, split-KV decoding and a
    variable-length batch (the last three on device-generated inputs); `only`
    picks one of "stress", "n4096", "latency", "gqa", "decode", "varlen"."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(2024)

    def rnd(*shape):
        return torch.randn(*shape, device=dev, generator=gen, dtype=torch.float32).to(torch.bfloat16)

    out = {}
    tf = lambda fl, ms: fl / (ms * 1e-3) / 1e12
    want = lambda name: only is None or only == name
    if want("stress"):
        out.update(measure_square_rows(fa2, dev, stream, peaks, ("stress",)))
    if want("n4096"):
        out.update(measure_square_rows(fa2, dev, stream, peaks, ("b4h32n4096",)))
    if want("latency"):
        out["latency"] = measure_latency_rows(fa2, dev, peaks)
    # Grouped-query prefill: 32 query heads over 8 K/V heads.
    B, H, Hkv, N, d = 1, 32, 8, 16384, 128
    if want("gqa"):
        q, dO = rnd(B, H, N, d), rnd(B, H, N, d)
        k, v = rnd(B, Hkv, N, d), rnd(B, Hkv, N, d)
        o, lse = fa2.fa2_fwd_gqa(q, k, v, causal=True, stream=stream)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        f_ms = _time_ms(lambda: fa2.fa2_fwd_gqa(q, k, v, o=o, lse=lse, causal=True, stream=stream), stream)
        b_ms = _time_ms(lambda: fa2.fa2_bwd_gqa(q, k, v, o, dO, lse, dq=dq, dk=dk, dv=dv, causal=True, stream=stream),
                        stream)
        ff, bf = 2.0 * B * H * N * N * d, 5.0 * B * H * N * N * d
        out["gqa_prefill"] = {"workload": f"B={B} H={H} H_kv={Hkv} N={N} d={d} causal",
                              "fwd_ms": f_ms, "fwd_tflops": tf(ff, f_ms), "bwd_ms": b_ms, "bwd_tflops": tf(bf, b_ms),
                              "fwd_pct_of_peak_burst": 100 * tf(ff, f_ms) / peaks["bf16_tflops"],
                              "bwd_pct_of_peak_burst": 100 * tf(bf, b_ms) / peaks["bf16_tflops"]}
        del q, dO, k, v, o, lse, dq, dk, dv
    # Split-KV decoding: one query per sequence against a 16K key-value cache,
    # with the library's suggested split count (2 on a 152-SM GB300: 128 CTAs
    # each streaming 8K keys of K and V, 5.7 TB/s against 5.0 with 16 splits).
    B, H, Hkv, Nq, Nk, d = 8, 32, 8, 1, 16384, 128
    if want("decode"):
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        splits = max(1, fa2.load_library().fa2_fwd_splitkv_suggest_splits(sms, B, H, Hkv, Nq, Nk))
        q, k, v = rnd(B, H, Nq, d), rnd(B, Hkv, Nk, d), rnd(B, Hkv, Nk, d)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
        ws = torch.empty(max(1, fa2.load_library().fa2_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, splits)),
                         dtype=torch.uint8, device=dev)
        ms = _time_ms(lambda: fa2.fa2_fwd_splitkv(q, k, v, splits, o=o, lse=lse, workspace=ws, causal=True,
                                                  stream=stream), stream, iters=50)
        nbytes = 2 * B * Hkv * Nk * d * 2 + 2 * B * H * Nq * d * 2 + B * H * Nq * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        out["decode_splitkv"] = {"workload": f"B={B} H={H} H_kv={Hkv} Nq={Nq} Nk={Nk} d={d} causal, {splits} splits",
                                 "ms": ms, "algorithmic_bytes": nbytes,
                                 "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                              "frac": gbs / peaks["hbm_gbs"]},
                                 "note": "K and V read once per K/V head (query heads of a group share the tile); "
                                         "launches: split kernel + combine kernel"}
        del q, k, v, o, lse, ws
    # Variable-length batch: 16 packed sequences of 1..8192 tokens.
    lens = workloads.varlen_lengths(16, 8192, seed=7)
    if not want("varlen"):
        return _checked(fa2, out)
    H, d = 32, 128
    T = sum(lens)
    q, k, v, dO = rnd(T, H, d), rnd(T, H, d), rnd(T, H, d), rnd(T, H, d)
    cu = torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32, device=dev)
    mx = max(lens)
    o, lse = fa2.fa2_fwd_varlen(q, k, v, cu, cu, mx, mx, causal=True, stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa2.load_library().fa2_bwd_varlen_workspace_bytes(H, T, d), dtype=torch.uint8, device=dev)
    f_ms = _time_ms(lambda: fa2.fa2_fwd_varlen(q, k, v, cu, cu, mx, mx, o=o, lse=lse, causal=True, stream=stream),
                    stream)
    b_ms = _time_ms(lambda: fa2.fa2_bwd_varlen(q, k, v, o, dO, lse, cu, cu, mx, mx, dq=dq, dk=dk, dv=dv,
                                               workspace=ws, causal=True, stream=stream), stream)
    sq = sum(L * L for L in lens)
    ff, bf = 2.0 * H * sq * d, 5.0 * H * sq * d
    out["varlen"] = {"workload": f"16 packed sequences, lengths {lens}, H={H} d={d} causal",
                     "fwd_ms": f_ms, "fwd_tflops": tf(ff, f_ms), "bwd_ms": b_ms, "bwd_tflops": tf(bf, b_ms),
                     "fwd_pct_of_peak_burst": 100 * tf(ff, f_ms) / peaks["bf16_tflops"],
                     "bwd_pct_of_peak_burst": 100 * tf(bf, b_ms) / peaks["bf16_tflops"]}
    return _checked(fa2, out)


def measure_square_rows(fa2, dev, stream, peaks, names=("stress", "b4h32n4096")):
    """Causal forward / backward TFLOPS of square d = 128 workloads at N = 4096:
    the large-logit stress workload (B=2, H=16, Q and K x 3, the seeded recipe
    of the parity tests) and B=4, H=32 on N(0, 1) inputs.  Each pass is timed
    over 10 back-to-back launches after 3 warm-up ones, CUDA events on the
    launching stream; the backward is the three kernels fa2_bwd enqueues, with
    the main kernel also timed alone."""
    shapes = {"stress": workloads.WORKLOADS["stress"],
              "b4h32n4096": workloads.Workload("b4h32n4096", 4, 32, 4096, 128, (True,), 1.0, 1010)}
    out = {}
    for name in names:
        w = shapes[name]
        x = workloads.workload_inputs(w)
        g = {k: t.to(dev) for k, t in x.items()}
        B, H, N, d = w.B, w.H, w.N, w.d
        o = torch.empty_like(g["q"])
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        Dvec = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        acc = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        fws = torch.empty(fa2.fa2_fwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        sc = w.scale
        f_ms = _time_ms(lambda: fa2.fa2_fwd_ws(g["q"], g["k"], g["v"], fws, o, lse, sc, True, stream), stream)
        b_ms = _time_ms(lambda: fa2.fa2_bwd_stages(g["q"], g["k"], g["v"], o, g["dO"], lse, Dvec, acc, dq, dk, dv,
                                                   sc, True, stream), stream)
        lib = fa2.load_library()
        st = stream.cuda_stream
        m_ms = _time_ms(lambda: lib.fa2_bwd_main(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(),
                                                 g["dO"].data_ptr(), lse.data_ptr(), Dvec.data_ptr(), acc.data_ptr(),
                                                 dk.data_ptr(), dv.data_ptr(), B, H, N, d, sc, 1, st), stream)
        ff, bf = w.fwd_flops(True), w.bwd_flops(True)
        tf = lambda fl, ms: fl / (ms * 1e-3) / 1e12
        out[name] = {"workload": f"B={B} H={H} N={N} d={d} causal" + (", Q and K x 3" if w.qk_mult != 1 else ""),
                     "fwd_ms": f_ms, "fwd_tflops": tf(ff, f_ms),
                     "fwd_pct_of_peak_burst": 100 * tf(ff, f_ms) / peaks["bf16_tflops"],
                     "bwd_ms": b_ms, "bwd_tflops": tf(bf, b_ms),
                     "bwd_pct_of_peak_burst": 100 * tf(bf, b_ms) / peaks["bf16_tflops"],
                     "bwd_main_ms": m_ms, "bwd_main_tflops": tf(bf, m_ms),
                     "target": "forward >= 60 %, backward >= 45 % of the burst peak"}
        del g, o, lse, dq, dk, dv, Dvec, acc, fws
    return out


def measure_dq_modes(fa2, dev, stream, peaks, names=("stress", "long")):
    """The three ways dQ can leave the backward main kernel (TMA bulk
    reduce-add, fp32 vector atomics, per-tile partial slots plus a
    fixed-order reduction), timed on the same inputs: the main kernel alone
    and the whole backward pass (the three stages), 3 warm-up and 5 timed
    runs each, CUDA events on the launching stream."""
    out = {}
    lib = fa2.load_library()
    for name in names:
        w = workloads.WORKLOADS[name]
        x = workloads.workload_inputs(w)
        g = {k: t.to(dev) for k, t in x.items()}
        B, H, N, d = w.B, w.H, w.N, w.d
        o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=True, stream=stream)
        Dvec = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        row = {"workload": f"{name}: B={B} H={H} N={N} d={d} causal"}
        bf = w.bwd_flops(True)
        for mode, label in ((0, "tma_reduce_add"), (1, "atomics_red_transposed"), (2, "split_accumulate")):
            if mode == 2:
                buf = torch.empty(lib.fa2_bwd_dq_partials_bytes(B, H, N, d, 1) // 4, dtype=torch.float32, device=dev)
            else:
                buf = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            mains, totals = [], []
            for it in range(8):
                fa2.fa2_bwd_stages(g["q"], g["k"], g["v"], o, g["dO"], lse, Dvec, buf, dq, dk, dv, w.scale, True,
                                   stream, hook=lambda j: ev[j].record(stream), dq_mode=mode)
                torch.cuda.synchronize()
                if it >= 3:
                    mains.append(ev[1].elapsed_time(ev[2]))
                    totals.append(ev[0].elapsed_time(ev[3]))
            m, t = statistics.median(mains), statistics.median(totals)
            row[label] = {"main_ms": m, "bwd_ms": t, "main_tflops": bf / (m * 1e-3) / 1e12,
                          "bwd_tflops": bf / (t * 1e-3) / 1e12,
                          "dq_buffer_bytes": buf.numel() * buf.element_size()}
            del buf
        out[name] = row
        del g, o, lse, Dvec, dq, dk, dv
    return out


def measure_latency_rows(fa2, dev, peaks, names=("tiny", "small")):
    """Microseconds per forward + backward step on the small workloads, where
    launch work rather than the GPU sets the time: 200 steps enqueued back to
    back (fa2_fwd_ws + fa2_bwd_ws: 3 kernels each; device time per step from CUDA
    events, host time per step from the clock around the enqueue), the same
    through prepared_step (arguments marshalled once), and the step replayed
    from a CUDA graph."""
    out = {}
    for name in names:
        w = workloads.WORKLOADS[name]
        x = workloads.workload_inputs(w)
        g = {k: t.to(dev) for k, t in x.items()}
        B, H, N, d = w.B, w.H, w.N, w.d
        o = torch.empty_like(g["q"])
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
        ws = torch.empty(fa2.fa2_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        fws = torch.empty(fa2.fa2_fwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream(device=dev)

        def step():
            fa2.fa2_fwd_ws(g["q"], g["k"], g["v"], fws, o, lse, w.scale, True, side)
            fa2.fa2_bwd_ws(g["q"], g["k"], g["v"], o, g["dO"], lse, ws, dq, dk, dv, w.scale, True, side)

        prepared = fa2.prepared_step(g["q"], g["k"], g["v"], o, lse, g["dO"], dq, dk, dv, fws, ws, w.scale, True, side)
        n = 200
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def timed(fn):
            for _ in range(20):
                fn()
            torch.cuda.synchronize()
            a.record(side)
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
            host = (time.perf_counter() - t0) / n * 1e6
            b.record(side)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n * 1e3, host

        dev_us, host_us = timed(step)
        prep_us, prep_host_us = timed(prepared)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                fa2.fa2_fwd_ws(g["q"], g["k"], g["v"], fws, o, lse, w.scale, True, None)
                fa2.fa2_bwd_ws(g["q"], g["k"], g["v"], o, g["dO"], lse, ws, dq, dk, dv, w.scale, True, None)
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize()
        a.record(side)
        with torch.cuda.stream(side):
            for _ in range(n):
                graph.replay()
        b.record(side)
        torch.cuda.synchronize()
        graph_us = a.elapsed_time(b) / n * 1e3
        out[name] = {"workload": f"B={B} H={H} N={N} d={d} causal", "us_per_step": dev_us,
                     "host_enqueue_us_per_step": host_us, "prepared_step_us": prep_us,
                     "prepared_host_enqueue_us_per_step": prep_host_us, "graph_replay_us_per_step": graph_us,
                     "launches_per_step": launches_per_step(N, d)}
        del graph, prepared, g, o, lse, dq, dk, dv, ws, fws
    return out


def _checked(fa2, out):
    torch.cuda.synchronize()
    if fa2.fa2_device_status(reset=True) != 0:
        raise RuntimeError("a kernel reported a device status during the row measurements")
    return out


def run_gpu(args, w, causal):
    world, rank, local = _dist()
    import tiled_exact_attention_fa2_gb300 as fa2
    from tiled_exact_attention_fa2_gb300 import _build
    _build.build()
    fa2.load_library()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    B, H, N, d = w.B, w.H, w.N, w.d
    x = workloads.make_inputs(B, H, N, d, seed=rank_seed(w, rank), qk_mult=w.qk_mult)
    g = {k: t.to(dev) for k, t in x.items()}
    o = torch.empty_like(g["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(g["q"]) for _ in range(3))
    Dvec = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if args.dq_mode == 2:  # per-tile partial slots
        dq_acc = torch.empty(fa2.load_library().fa2_bwd_dq_partials_bytes(B, H, N, d, int(causal)) // 4,
                             dtype=torch.float32, device=dev)
    else:
        dq_acc = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    fws = torch.empty(fa2.fa2_fwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    scale = w.scale
    fwd_flops, bwd_flops = w.fwd_flops(causal), w.bwd_flops(causal)

    n_ev = args.steps + args.warmup
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_ev)]

    def step(i):
        e = ev[i]
        e[0].record(stream)
        fa2.fa2_fwd_ws(g["q"], g["k"], g["v"], fws, o, lse, scale, causal, stream)
        fa2.fa2_bwd_stages(g["q"], g["k"], g["v"], o, g["dO"], lse, Dvec, dq_acc, dq, dk, dv, scale, causal,
                           stream, hook=lambda j: e[j + 1].record(stream), dq_mode=args.dq_mode)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    sampler = ClockSampler(local)
    _barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.warmup, n_ev):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    clocks = sampler.stop()
    status = fa2.fa2_device_status(reset=True)
    total_ms = t_start.elapsed_time(t_end)
    total_ms = _max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    timed = ev[args.warmup:]
    fwd_list = [e[0].elapsed_time(e[1]) for e in timed]
    main_list = [e[2].elapsed_time(e[3]) for e in timed]
    fwd_ms = statistics.mean(fwd_list)
    pre_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in timed)
    main_ms = statistics.mean(main_list)
    conv_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in timed)
    bwd_ms = pre_ms + main_ms + conv_ms

    # ---- end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        host = {k: x[k].pin_memory() for k in ("q", "k", "v", "dO")}
        host.update({k: torch.empty_like(host["q"]).pin_memory() for k in ("o", "dq", "dk", "dv")})
        host["lse"] = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        ws = torch.empty(fa2.fa2_step_from_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
        for _ in range(max(1, args.warmup)):
            fa2.fa2_step_from_host(host, causal, scale, stream, workspace=ws)
        torch.cuda.synchronize()
        _barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fa2.fa2_step_from_host(host, causal, scale, stream, workspace=ws)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = _max_over_ranks(a.elapsed_time(b), world) / args.steps
        h2d = sum(host[k].numel() * host[k].element_size() for k in ("q", "k", "v", "dO"))
        d2h = sum(host[k].numel() * host[k].element_size() for k in ("o", "lse", "dq", "dk", "dv"))
        e2e = {"value": job_tflops(world, fwd_flops + bwd_flops, e2e_ms), "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "api": "fa2_step_from_host (C ABI, pinned host buffers)"}

    peaks = _peaks()
    value = job_tflops(world, fwd_flops + bwd_flops, ms_step)
    fwd_tf = fwd_flops / (fwd_ms * 1e-3) / 1e12
    bwd_tf = bwd_flops / (bwd_ms * 1e-3) / 1e12
    main_tf = bwd_flops / (main_ms * 1e-3) / 1e12
    pre_bytes = 2 * B * H * N * d * 2 + B * H * N * 4 + B * H * N * d * 4  # O, dO read; D written; dQacc zeroed
    peak_key, peak_why = roofline_peak(total_ms * 1e-3, clocks)
    rooflines = {
        name: {"kernel": name, "bound": "tensor", "achieved": tf, "peak": peaks[peak_key], "unit": "TFLOP/s",
               "frac": tf / peaks[peak_key], "traffic": kernel_traffic(name, w.name, causal),
               "algorithmic_bytes": algorithmic_bytes(name, B, H, N, d), "ms": ms,
               "peak_source": f"{peaks['source']} {peak_key} ({peak_why})",
               "frac_of_burst": tf / peaks["bf16_tflops"],
               "frac_of_sustained": tf / peaks["bf16_tflops_sustained"]}
        for name, tf, ms in (("fa2_bwd_kernel", main_tf, main_ms), ("fa2_fwd_kernel", fwd_tf, fwd_ms))}
    rooflines["fa2_fwd_kernel"]["note"] = ("time of the whole forward pass (fa2_v_to_f16_kernel, the fp16 copy of V, "
                                           "then fa2_fwd_kernel); the launch list under profiles/ gives the split")
    dominant = "fa2_bwd_kernel" if main_ms >= fwd_ms else "fa2_fwd_kernel"
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}: B={B} H={H} N={N} d={d} {'causal' if causal else 'non-causal'}",
                   "B": B, "H": H, "N": N, "d": d, "causal": causal, "parallelism": f"weak x{world} (heads)",
                   "dq_reduction": ["tma_reduce_add", "atomics_red_transposed", "split_accumulate"][args.dq_mode],
                   "l2": (f"inputs larger than L2 (Q, K, V, dO {B * H * N * d * 2 / 1e6:.0f} MB each), no flush"
                          if 4 * B * H * N * d * 2 > 129e6 else "inputs fit in L2 together; back-to-back steps")},
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "pct_of_peak_burst": 100 * fwd_tf / peaks["bf16_tflops"],
                "pct_of_peak_sustained": 100 * fwd_tf / peaks["bf16_tflops_sustained"]},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "pct_of_peak_burst": 100 * bwd_tf / peaks["bf16_tflops"],
                "pct_of_peak_sustained": 100 * bwd_tf / peaks["bf16_tflops_sustained"],
                "preprocess_ms": pre_ms, "main_ms": main_ms, "dq_convert_ms": conv_ms,
                "preprocess_gbs": pre_bytes / (pre_ms * 1e-3) / 1e9},
        "roofline": rooflines[dominant],
        "roofline_other": rooflines["fa2_fwd_kernel" if dominant == "fa2_bwd_kernel" else "fa2_bwd_kernel"],
        "timing": {"fwd_ms": _stats(fwd_list), "bwd_main_ms": _stats(main_list),
                   "method": "CUDA events on the launching stream around each kernel of every timed step"},
        "gpu_launches": launches_per_step(N, d) * args.steps,
        "device_status": status,
        "clocks": clocks,
        "e2e": e2e,
    }
    if world == 1 and not args.no_rows:
        line["rows"] = measure_rows(fa2, dev, stream, peaks)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, causal)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--noncausal", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the GQA / decoding / varlen measurements")
    ap.add_argument("--dq-mode", type=int, default=0, choices=[0, 1, 2],
                    help="how dQ leaves the backward main kernel: 0 TMA reduce-add (default), 1 fp32 atomics, "
                         "2 per-tile partials + ordered reduction (d = 128 only)")
    ap.add_argument("--row", choices=["gqa", "decode", "varlen", "stress", "n4096", "latency", "dqmodes"],
                    help="measure only this widened row and print it (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    w = workloads.WORKLOADS[args.workload]
    causal = not args.noncausal
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # Not started by torchrun: start the args.gpus replicas here.
        if args.impl == "ours":
            if torch.cuda.device_count() < args.gpus:
                sys.exit(f"--gpus {args.gpus}: only {torch.cuda.device_count()} GPU(s) visible")
            from tiled_exact_attention_fa2_gb300 import _build
            _build.build()
        return spawn_local_replicas(args.gpus, sys.argv[1:])
    if args.impl == "reference":
        return run_reference(args, w, causal)
    if args.row:
        import tiled_exact_attention_fa2_gb300 as fa2
        from tiled_exact_attention_fa2_gb300 import _build
        _build.build()
        dev = torch.device("cuda:0")
        stream = torch.cuda.Stream(device=dev)
        if args.row == "dqmodes":
            res = measure_dq_modes(fa2, dev, stream, _peaks())
            torch.cuda.synchronize()
            res["device_status"] = fa2.fa2_device_status(reset=True)
        else:
            res = measure_rows(fa2, dev, stream, _peaks(), only=args.row)
        print(json.dumps({"row": args.row, **res}), flush=True)
        return 0
    return run_gpu(args, w, causal)


if __name__ == "__main__":
    sys.exit(main())
