#!/usr/bin/env python3
"""Benchmark of one layer of the sparse-KV decode step on GB300.

A step is one ``dd_step`` over one layer: score -> top-k -> union/resolve ->
gather -> attention.  The default (headline) workload is the 32B-class GQA
layer: 32 requests, 64 query / 8 KV heads, head dim 128, 32K context in
chunks of 16, top-128 chunks per KV head, one real + four draft queries per
request sharing one deduplicated gather, all KV in pinned host memory.  Four
layers of independent data are cycled so that no step finds its inputs in L2.
Prints one JSON line (see the keys below).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--mode auto|zerocopy|kernel|memcpy] [--landmarks mean|minmax]
                    [--residency workload|none|all] [--pipeline [--prefetch-ctas N] [--layer-gap-us T]]

At N=1 the headline line carries ``per_config``: every other workload (with
its own residency) and the fully resident lines of the Llama-3-8B-shaped and
32B-class layers, each measured the same way in a child process run before
the headline (so that one process holds its pinned host KV at a time).  It
also carries ``landmark_build_us``, the landmark build (prefill) timed on its
own from pinned host memory and from HBM.
``--impl reference`` times the CPU oracle instead, on whole steps of the same
workload spread over the host cores.  The default line also reports the oracle
on one core (a bounded sample) and on every host core.
``--pipeline`` runs several layers with drifting queries: predictive prefetch
on a low-priority stream, the same steps serialized, and the same steps with
the capped LRU residency update.  Under torchrun every rank runs its own independent
batch (weak scaling, no collective on the data path); the time is the max over
ranks.
"""
from __future__ import annotations

import os

# the CPU oracle runs single-threaded: its BLAS calls must not spread over cores
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import math
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_kv_offload_gb300 import synth                      # noqa: E402
from sparse_kv_offload_gb300.workloads import (BY_NAME, GQA32B_5Q, LLAMA8B_32K, QWEN8B_128K,  # noqa: E402
                                               STRESS_512K, TINY)

METRIC = "sparse decode steps/s per layer; HBM GB/s and host-gather GB/s vs roofline"
UNIT = "steps/s"
N_LAYERS = 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 50 ms for the whole GPU arm; each sample keeps
    the driver's timestamp, so that the clocks can be summarised over the GPU
    work and over each timed block (``window``)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.windows = []            # (name, t0, t1) in time.time() seconds
        try:
            import torch
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", uuid, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def window(self, name, t0, t1):
        self.windows.append((name, t0, t1))

    @staticmethod
    def _parse(out):
        import datetime
        rows = []
        for r in out.strip().splitlines():
            f = [x.strip() for x in r.split(",")]
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]),
                             {n for n, v in zip(ClockSampler.REASONS, f[4:8]) if v.lower() == "active"}))
            except (ValueError, IndexError):
                continue
        return rows

    @staticmethod
    def _summary(rows):
        if not rows:
            return {"samples": 0}
        return {"sm_mhz": float(np.median([r[1] for r in rows])), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": sorted(set().union(*[r[3] for r in rows])), "samples": len(rows)}

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = self._parse(out)
        if not rows:
            return None
        # samples inside the windows of GPU work (timed and untimed blocks); all samples when none fell inside
        inside = [r for r in rows if any(t0 - 0.025 <= r[0] <= t1 + 0.025 for _, t0, t1 in self.windows)]
        res = self._summary(inside or rows)
        res["scope"] = ("samples taken while the GPU arm's kernels ran (every timed and untimed block)" if inside
                        else "every sample of the GPU arm")
        res["samples_all"] = len(rows)
        res["blocks"] = {name: self._summary([r for r in rows if t0 - 0.025 <= r[0] <= t1 + 0.025])
                         for name, t0, t1 in self.windows}
        return res


# ------------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)
class OracleSample:
    """The oracle's step over single (request, KV head) units of the workload.

    Units are independent through every stage, so one unit is 1/(B*Hkv) of a
    step: steps/s = units / (B * Hkv * seconds).  The sample is request 0's
    Hkv units, built from the host generator (the same definition the GPU
    path's inputs come from)."""

    def __init__(self, w, landmarks="mean", heads=None):
        import oracle
        self.oracle = oracle
        self.w = w
        build_lm = oracle.build_minmax_landmarks if landmarks == "minmax" else oracle.build_landmarks
        q = synth.queries(w.seed, 1, w.n_q, w.Hq, w.d, w.spec_scale)
        bias = u_hat = None
        if w.key_bias == "hot":
            bias = synth.hot_chunk_bias(w.seed, 1, w.Hkv, w.C, w.hot_frac, w.bias_sigma)
            u_hat = synth.query_direction(q, w.Hkv)
        elif w.key_bias == "zipf":
            bias = synth.zipf_chunk_bias(w.seed, 1, w.Hkv, w.C, w.zipf_alpha, w.bias_sigma)
            u_hat = synth.query_direction(q, w.Hkv)
        self.units = []
        for g in (range(w.Hkv) if heads is None else heads):
            u = np.array([g])
            K = synth.kv_rows(w.seed, synth.TID_K, 1, w.Hkv, w.L, w.d, w.cs, u, np.zeros(1, np.int64), w.L,
                              bias, u_hat).reshape(1, 1, w.L, w.d)
            V = synth.kv_rows(w.seed, synth.TID_V, 1, w.Hkv, w.L, w.d, w.cs, u, np.zeros(1, np.int64),
                              w.L).reshape(1, 1, w.L, w.d)
            qg = np.ascontiguousarray(q[:, :, g * w.G:(g + 1) * w.G])
            self.units.append((qg, build_lm(K, w.cs), K, V))
        self.slot = np.full((1, 1, w.C), -1, np.int32)
        self.empty = np.zeros((0, w.cs, w.d), np.uint16)
        self.next = 0

    def run_units(self, n: int) -> float:
        t0 = time.perf_counter()
        for _ in range(n):
            qg, lm, K, V = self.units[self.next % len(self.units)]
            self.next += 1
            self.oracle.step(qg, lm, K, V, self.slot, self.empty, self.empty, self.w.k, self.w.cs)
        return time.perf_counter() - t0

    def describe(self, n_units):
        w = self.w
        return (f"oracle (numpy fp64, one thread) on {n_units} (request, KV head) units of request 0 per "
                f"timing, each 1/{w.B * w.Hkv} of a step; steps/s = units / ({w.B * w.Hkv} x seconds)")


def cpu_baseline(w, budget_s=12.0, landmarks="mean"):
    s = OracleSample(w, landmarks)
    s.run_units(1)
    done, spent = 0, 0.0
    while spent < budget_s:
        spent += s.run_units(1)
        done += 1
    return {"value": done / (w.units * spent), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": s.describe(done) + f"; {done} units in {spent:.1f} s"}


def _oracle_worker(task):
    """One process of the all-cores baseline: the oracle step on one (request 0,
    KV head) unit, repeated for `budget` seconds (inputs built before timing)."""
    wname, head, landmarks, budget = task
    s = OracleSample(BY_NAME[wname], landmarks, heads=[head])
    s.run_units(1)
    done, spent = 0, 0.0
    while spent < budget:
        spent += s.run_units(1)
        done += 1
    return done, spent


def cpu_baseline_all_cores(w, budget_s=8.0, landmarks="mean"):
    """The same oracle code over independent (b, g) units on every host core
    (one process per core, spawned: numerics unchanged, units are independent)."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_worker, [(w.name, i % w.Hkv, landmarks, budget_s) for i in range(n)])
    rate = sum(d / t for d, t in res)              # units per second, all processes together
    return {"value": rate / w.units, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{n} processes, each the oracle step on one (request 0, KV head) unit for "
                      f"{budget_s:.0f} s; steps/s = sum of units/s / {w.units}"}


_REF_SAMPLE = None


def _ref_init(wname, landmarks, heads_q):
    """A reference-arm process: the inputs of one of request 0's KV heads."""
    global _REF_SAMPLE
    _REF_SAMPLE = OracleSample(BY_NAME[wname], landmarks, heads=[heads_q.get()])
    _REF_SAMPLE.run_units(1)


def _ref_run(n):
    return _REF_SAMPLE.run_units(n)


def run_reference(args, world, rank):
    """The oracle on whole steps: each step evaluates all B*Hkv (request, KV
    head) units, spread over one process per host core (units are independent
    through every stage, so the numerics are the oracle's own)."""
    if rank != 0:
        return 0
    import multiprocessing as mp
    w = BY_NAME[args.workload]
    n_proc = max(1, min(os.cpu_count() or 1, w.units))
    ctx = mp.get_context("spawn")
    heads_q = ctx.Queue()
    for i in range(n_proc):
        heads_q.put(i % w.Hkv)
    per_task = max(1, w.units // (4 * n_proc))
    tasks = [per_task] * (w.units // per_task) + ([w.units % per_task] if w.units % per_task else [])
    with ctx.Pool(n_proc, initializer=_ref_init, initargs=(w.name, args.landmarks, heads_q)) as pool:
        for _ in range(args.warmup):
            pool.map(_ref_run, tasks, chunksize=1)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.map(_ref_run, tasks, chunksize=1)
        spent = time.perf_counter() - t0
    value = args.steps / spent
    sample = (f"whole steps: each step runs the oracle (numpy fp64) on all {w.units} (request, KV head) units of "
              f"the workload, {per_task} units per task over {n_proc} processes (one per host core); each process "
              f"holds the host inputs of one of request 0's {w.Hkv} KV heads, and every unit of a step is "
              f"evaluated on those inputs (units have the same shape; generating all {w.B} requests' host KV in "
              f"numpy would take minutes)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, "oracle", landmarks=args.landmarks),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_proc, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": spent,
    }
    print(json.dumps(line), flush=True)
    return 0


# the step scores in one streaming kernel (k_score), then runs top-k and the
# resolver as one kernel (k_select_fused); the attention is k_attn (mma.sync)
# up to 16 query vectors per KV head and k_attn_tc (tcgen05) above
# timed steps per CUDA-event bracket of the dominant kernel (see run_ours);
# prime to the N_LAYERS layers cycled, so the bracketed steps cover every layer
EV_EVERY = 7

KERNEL_SOURCE = {"gather": ("k_gather", ("dd_gather.cu",)),
                 "attention": ("k_attn", ("dd_attn.cu", "dd_attn.cuh", "dd_tc.cuh")),
                 "attention_tc": ("k_attn_tc", ("dd_attn_tc.cu", "dd_attn.cuh", "dd_tc.cuh")),
                 "score": ("k_score_tc", ("dd_score_tc.cu", "dd_tc.cuh")), "topk": ("k_select_fused", ("dd_select.cu",))}


def attention_stage(w) -> str:
    """The attention kernel the workload runs: tcgen05 above 16 query vectors per KV head."""
    return "attention_tc" if w.n_q * w.G > 16 else "attention"


def profiled_traffic(stage: str, workload: str):
    """DRAM bytes per launch of the stage's main kernel from the committed ncu
    summary, or None when there is none or the kernel source has changed since
    the counters were taken."""
    import re
    kernel, srcs = KERNEL_SOURCE[stage]
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    t = re.search(r"^traffic_bytes_per_launch: (\d+)$", text, re.M)
    h = re.search(r"^code_sha256_prefix: ([0-9a-f]+)$", text, re.M)
    if not t or not h:
        return None
    cur = code_hash(*[os.path.join(ROOT, "sparse_kv_offload_gb300", "csrc", f) for f in srcs])
    return int(t.group(1)) if cur.startswith(h.group(1)) else None


def code_hash(*paths: str) -> str:
    """sha256 of the CUDA sources of a kernel with their comments and whitespace
    removed: a profile stays valid across comment edits, not across code
    changes."""
    import hashlib
    import re
    parts = []
    for path in paths:
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        parts.append(" ".join(text.split()))
    return hashlib.sha256("\n".join(parts).encode()).hexdigest()


def config_of(w, gather_mode, world=1, landmarks="mean"):
    base, _, auto = gather_mode.partition(" ")
    gather_desc = {"zerocopy": "zero-copy, fused into the attention kernel",
                   "kernel": "zero-copy gather kernel into staging, then the attention",
                   "memcpy": "miss list to host, cudaMemcpyAsync per run of chunks"}.get(base, base) + (
        " (chosen automatically: " + ("a hot pool exists" if base == "kernel" else "no hot pool") + ")"
        if auto else "")
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "L": w.L, "cs": w.cs, "k": w.k,
            "n_q": w.n_q, "residency": w.residency, "gather": gather_desc, "landmarks": landmarks,
            "l2": (f"inputs larger than L2 ({N_LAYERS} layers of landmarks and host KV cycled)" if N_LAYERS >= 4 else
                   f"{N_LAYERS} layer(s) cycled: inputs may stay in L2 between steps (profiling runs only)"),
            "host_pages": "every pinned host K/V page read once by the GPU before timing",
            "parallelism": f"independent batch per GPU x{world}"}


# ------------------------------------------------------------------ GPU arm
def rank_seed(seed: int, rank: int) -> int:
    """Each rank decodes its own batch: a distinct seed per rank."""
    return seed + 7919 * rank


class LayerData:
    def __init__(self, dd, shape, w, layer, rank, lm_vectors=1):
        import torch
        seed = rank_seed(w.seed, rank)
        self.seed = seed
        self.q = torch.empty(w.B * w.n_q * w.Hq * w.d, dtype=torch.bfloat16, device="cuda")
        dd.synth_queries(shape, seed, layer, w.spec_scale, self.q)
        bias = u_hat = None
        if w.key_bias == "hot":
            qh = synth.queries(seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale, layer)
            bias = torch.from_numpy(synth.hot_chunk_bias(seed, w.B, w.Hkv, w.C, w.hot_frac, w.bias_sigma,
                                                         layer)).cuda()
            u_hat = torch.from_numpy(synth.query_direction(qh, w.Hkv)).cuda()
        elif w.key_bias == "zipf":
            qh = synth.queries(seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale, layer)
            bias = torch.from_numpy(synth.zipf_chunk_bias(seed, w.B, w.Hkv, w.C, w.zipf_alpha, w.bias_sigma,
                                                          layer)).cuda()
            u_hat = torch.from_numpy(synth.query_direction(qh, w.Hkv)).cuda()
        n = w.B * w.Hkv * w.L * w.d
        self.Kh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
        self.Vh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
        dd.synth_kv(shape, seed, synth.tensor_id(synth.TID_K, layer), self.Kh, bias, u_hat)
        dd.synth_kv(shape, seed, synth.tensor_id(synth.TID_V, layer), self.Vh)
        self.lm = torch.empty(w.B * w.Hkv * w.C * lm_vectors * w.d, dtype=torch.bfloat16, device="cuda")
        self.bias, self.u_hat = bias, u_hat
        self.Khot = self.Vhot = None   # HBM pool of the resident chunks (slot order)
        self.slot = None               # residency map [B*Hkv*C]: pool slot, or -1 (host)
        self.q_host = torch.empty(self.q.numel(), dtype=torch.bfloat16, pin_memory=True)
        torch.cuda.synchronize()
        self.q_host.copy_(self.q)


def host_link_peaks(dd, shape):
    """Pinned H2D copy peak (best of 10 x 1 GiB cudaMemcpyAsync) and the
    zero-copy gather kernel reading 1 GiB of consecutive chunks."""
    import torch
    n = 1 << 29                                   # 1 GiB of bf16
    src = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    src.fill_(1.0)
    dst = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    best = 0.0
    for _ in range(10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        best = max(best, (2 * n) / (a.elapsed_time(b) * 1e-3) / 1e9)
    # zero-copy: the gather kernel over every chunk of a 512 MiB K half and a
    # 512 MiB V half, in order (8 heads x 16384 chunks)
    from sparse_kv_offload_gb300.dd import Context, Shape
    units, C = 8, 16384
    sh = Shape(1, units, units, shape.d, C * shape.cs, shape.cs, 1, 1)
    m = units * C
    need = m * shape.cs * shape.d
    zc = None
    if 2 * need <= n:
        with Context(sh, max_misses=m) as ctx:
            miss = torch.arange(m, dtype=torch.int32, device="cuda")
            cnt = torch.tensor([m], dtype=torch.int32, device="cuda")
            Kh, Vh = src[:need], src[need:2 * need]
            Kst, Vst = dst[:need], dst[need:2 * need]
            zc = 0.0
            for _ in range(6):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                ctx.gather_kv(Kh, Vh, miss, cnt, Kst, Vst)
                b.record()
                b.synchronize()
                zc = max(zc, (4 * need) / (a.elapsed_time(b) * 1e-3) / 1e9)
            if ctx.status() != 0:
                zc = None
    del src, dst
    return best, zc


def landmark_build_times(dd, shape, w, L_, lm_kind, sampler, reps=5):
    """The landmark build (prefill, off the decode path) timed on its own, from
    the pinned host K (read over the host link) and from a device copy of the
    same K (read from HBM): median of ``reps`` launches after two warm-ups."""
    import torch
    minmax = lm_kind == dd.LM_MINMAX
    vec = 2 if minmax else 1
    lm = torch.empty(w.B * w.Hkv * w.C * vec * w.d, dtype=torch.bfloat16, device="cuda")
    k_bytes = w.B * w.Hkv * w.L * w.d * 2
    lm_bytes = lm.numel() * 2
    res = {"bytes_read": k_bytes, "bytes_written": lm_bytes,
           "kernel": "k_build_minmax" if minmax else "k_build_landmarks"}
    with dd.Context(shape, max_misses=1) as c:
        build = c.build_landmarks_minmax if minmax else c.build_landmarks
        for src_name, K in (("pinned_host", L_.Kh), ("device", None)):
            if K is None:
                K = L_.Kh.to("cuda")
            for _ in range(2):
                build(K, lm)
            torch.cuda.synchronize()
            t_wall = time.time()
            times = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                build(K, lm)
                b.record()
                b.synchronize()
                times.append(a.elapsed_time(b) * 1e3)
            if sampler:
                sampler.window(f"landmark build ({src_name})", t_wall, time.time())
            us = float(np.median(times))
            res[src_name] = {"us": us, "gbs": (k_bytes + lm_bytes) / (us * 1e-6) / 1e9}
            del K
        if c.status() != 0:
            raise RuntimeError("device status after the landmark builds is not OK")
    return res


def run_ours(args, world, rank, local, per_config=None):
    import torch
    torch.cuda.set_device(local)
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd
    sampler = ClockSampler(local) if rank == 0 else None
    w = BY_NAME[args.workload]
    shape = dd.Shape(w.B, w.Hq, w.Hkv, w.d, w.L, w.cs, w.k, w.n_q)
    mode = {"memcpy": dd.GATHER_MEMCPY, "kernel": dd.GATHER_KERNEL, "auto": dd.GATHER_AUTO}.get(args.mode,
                                                                                              dd.GATHER_ZEROCOPY)
    cap = w.max_misses

    minmax = args.landmarks == "minmax"
    lm_kind = dd.LM_MINMAX if minmax else dd.LM_MEAN
    layers = [LayerData(dd, shape, w, l, rank, 2 if minmax else 1) for l in range(N_LAYERS)]
    resident_all = args.residency == "all"
    own_residency = args.residency == "workload" and w.residency in ("uniform", "carry")
    if resident_all:
        # every chunk resident: the layers' K and V also live in an HBM pool, in the
        # host layout ([B*Hkv*C] chunks of cs rows), and the residency map is the identity
        for L_ in layers:
            L_.Khot = L_.Kh.to("cuda")
            L_.Vhot = L_.Vh.to("cuda")
    touch = torch.empty(w.B * w.Hkv * w.C * w.d, dtype=torch.bfloat16, device="cuda")
    with dd.Context(shape, max_misses=cap) as ctx0:
        for L_ in layers:
            if minmax:
                ctx0.build_landmarks_minmax(L_.Kh, L_.lm)
            else:
                ctx0.build_landmarks(L_.Kh, L_.lm)
            # the GPU's first access to a pinned host page pays for its address
            # translation; read every V page once too (K was just read in full),
            # so that the timed steps see the steady state
            ctx0.build_landmarks(L_.Vh, touch)
        del touch
        maps = []
        for l, L_ in enumerate(layers):
            if resident_all or not own_residency:
                maps.append(None)
                continue
            if w.residency == "uniform":
                res = synth.uniform_residency(L_.seed, w.B, w.Hkv, w.C, w.resident_frac, l)
            else:
                # temporal locality: this layer's union, taken from one untimed step with
                # nothing resident, stands in for the previous step's; a seeded share of
                # it is resident
                uidx = torch.empty(w.B * w.Hkv * shape.umax, dtype=torch.int32, device="cuda")
                ucnt = torch.empty(w.B * w.Hkv, dtype=torch.int32, device="cuda")
                Kst0 = [torch.empty(cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
                Vst0 = [torch.empty(cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
                out0 = torch.empty(w.B * w.n_q * w.Hq * w.d, dtype=torch.float32, device="cuda")
                none = torch.full((w.B * w.Hkv * w.C,), -1, dtype=torch.int32, device="cuda")
                ctx0.step(0, L_.q, L_.lm, L_.Kh, L_.Vh, none, None, None, Kst0, Vst0, out0, lm_kind=lm_kind,
                          intermediates={"union_idx": uidx, "union_cnt": ucnt})
                ui = uidx.cpu().numpy().reshape(w.B * w.Hkv, shape.umax)
                uc = ucnt.cpu().numpy()
                sets = [set(ui[u, :uc[u]].tolist()) for u in range(w.B * w.Hkv)]
                res = synth.carried_residency(L_.seed, sets, w.B, w.Hkv, w.C, w.resident_frac, l)
                del Kst0, Vst0, out0, none
            maps.append(res.reshape(-1))
        # one pool size for every layer (the context checks each step's pools against it)
        n_pool = max([int((m >= 0).sum()) for m in maps if m is not None] + [0])
        for l, L_ in enumerate(layers):
            m = maps[l]
            if resident_all:
                L_.slot = torch.arange(w.B * w.Hkv * w.C, dtype=torch.int32, device="cuda")
            elif m is None:
                L_.slot = torch.full((w.B * w.Hkv * w.C,), -1, dtype=torch.int32, device="cuda")
            else:
                n_hot = int((m >= 0).sum())
                chunk_map = np.empty(n_hot, np.int32)
                chunk_map[m[m >= 0]] = np.nonzero(m >= 0)[0]
                L_.Khot = torch.empty(max(1, n_pool) * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
                L_.Vhot = torch.empty(max(1, n_pool) * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
                if n_hot:
                    cm = torch.from_numpy(chunk_map).cuda()
                    dd.synth_kv(shape, L_.seed, synth.tensor_id(synth.TID_K, l), L_.Khot, L_.bias, L_.u_hat,
                                chunk_map=cm)
                    dd.synth_kv(shape, L_.seed, synth.tensor_id(synth.TID_V, l), L_.Vhot, chunk_map=cm)
                L_.slot = torch.from_numpy(m.astype(np.int32)).cuda()
        torch.cuda.synchronize()
    hot_slots = w.B * w.Hkv * w.C if resident_all else n_pool
    ctx = dd.Context(shape, max_misses=cap, hot_slots=hot_slots)
    ns = cap * w.cs * w.d
    Kst = [torch.empty(ns, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Vst = [torch.empty(ns, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    out = torch.empty(w.B * w.n_q * w.Hq * w.d, dtype=torch.float32, device="cuda")
    K = args.steps
    miss_counts = torch.zeros(K, dtype=torch.int32, device="cuda")
    union_cnts = torch.zeros(K, w.B * w.Hkv, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    assert ctx.status() == 0

    link_memcpy, link_zc = host_link_peaks(dd, shape)

    # Timed steps carry events only at the boundaries of the dominant stage
    # (the fused gather + attention, or the gather in memcpy mode): an event
    # between two kernels stops the next one from launching early.  The
    # per-stage breakdown comes from separate steps with all six events.
    # the gather the step runs (auto: the separate gather kernel when there is a hot pool)
    gather_used = args.mode if args.mode != "auto" else ("kernel" if hot_slots > 0 else "zerocopy")
    fused = gather_used == "zerocopy"   # the attention kernel gathers the missing chunks itself
    dom_marks = (4, 5) if fused else (3, 4)
    n_stage = min(K, 200)

    def events(n):
        ev_ = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]
        for row in ev_:
            for e in row:
                e.record()                  # creates the event handles
        return ev_
    ev = events(K)
    ev_stage = events(n_stage)
    # per traced step, the kernels' own first-start / last-end %globaltimer stamps
    # (scoring, selection, attention): their durations inside the step, with no
    # event between them to stop a kernel from starting early (steps of their
    # own, after the timed ones, so the timed steps carry no extra host work)
    n_trace = min(K, 200)
    trace = torch.zeros((n_trace, 3, 2, dd.TRACE_SLOTS), dtype=torch.int64, device="cuda")
    trace[:, :, 0] = -1                    # UINT64_MAX: the per-SM start words (atomic min)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()

    def step(i, layer, events=None, inter=None, trace=None):
        d_ = layers[layer % N_LAYERS]
        ctx.step(layer, d_.q, d_.lm, d_.Kh, d_.Vh, d_.slot, d_.Khot, d_.Vhot, Kst, Vst, out, mode=mode,
                 intermediates=inter, stage_events=events, lm_kind=lm_kind, mass_gamma=args.mass_gamma,
                 softmax_scale=args.softmax_scale, trace=trace)

    for i in range(args.warmup):
        step(i, i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    launches0 = ctx.launch_count()
    t0 = time.perf_counter()
    t0_wall = time.time()
    t_start.record()
    # the dominant kernel is bracketed by CUDA events on every EV_EVERY-th timed
    # step only: an event between two kernels stops the next one from starting
    # early (programmatic dependent launch), so events on every step would slow
    # the very steps they time
    ev_steps = list(range(0, K, EV_EVERY))
    for i in range(K):
        marks = [ev[i][m] if m in dom_marks and i % EV_EVERY == 0 else None for m in range(6)]
        step(i, args.warmup + i, marks, {"miss_count": miss_counts[i:i + 1], "union_cnt": union_cnts[i]})
    t_end.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if sampler:
        sampler.window("timed steps", t0_wall, time.time())
    barrier(world)
    torch.cuda.synchronize()
    launches = ctx.launch_count() - launches0
    st = ctx.status()
    if st != 0:
        raise RuntimeError(f"device status after the timed steps: {dd.status_str(st)}")

    gpu_s = t_start.elapsed_time(t_end) * 1e-3
    t_max = max_over_ranks(gpu_s, world)
    names = ("score", "topk", "resolve", "gather", "attention")
    dom_timed = names[dom_marks[0]]
    dom_ms_timed = float(np.mean([ev[i][dom_marks[0]].elapsed_time(ev[i][dom_marks[1]]) for i in ev_steps]))
    t1_wall = time.time()
    for i in range(n_stage):
        step(i, args.warmup + K + i, ev_stage[i])
    for i in range(n_trace):
        step(i, args.warmup + K + n_stage + i, trace=trace[i])
    torch.cuda.synchronize()
    if sampler:
        sampler.window("stage-breakdown and traced steps", t1_wall, time.time())
    if ctx.status() != 0:
        raise RuntimeError("device status after the stage-breakdown steps is not OK")
    stage_ms = {n: float(np.mean([ev_stage[i][s].elapsed_time(ev_stage[i][s + 1]) for i in range(n_stage)]))
                for s, n in enumerate(names)}
    M = miss_counts.double().mean().item()
    U = union_cnts.double().sum(1).mean().item()
    chunk_b = w.cs * w.d * 2

    # algorithmic bytes per launch
    q_b = w.B * w.n_q * w.Hq * w.d * 2
    score_b = w.B * w.Hkv * w.C * w.d * 2 * (2 if minmax else 1) + q_b + w.B * w.n_q * w.Hkv * w.C * 4
    attn_b = U * 2 * chunk_b + q_b + w.B * w.n_q * w.Hq * w.d * 4
    gather_b = M * 2 * chunk_b                   # bytes read over the host link (written to HBM once more)
    hbm_peak, hbm_kind = peaks()
    stage_bytes = {"score": score_b, "attention": attn_b, "gather": gather_b}
    dom = max(("score", "attention", "gather"), key=lambda n: stage_ms[n])
    folded = dd.step_folds_scoring(shape, torch.cuda.get_device_properties(0).multi_processor_count,
                                   lm_kind, args.mass_gamma) > 0
    # the dominant kernel's duration is the one measured inside the timed region
    t_dom = (dom_ms_timed if dom == dom_timed else stage_ms[dom]) * 1e-3
    traffic = profiled_traffic(dom, w.name)
    wl_name = w.name + "_all_resident" if resident_all else w.name
    att = attention_stage(w)
    att_kernel = KERNEL_SOURCE[att][0]
    if fused and dom == "attention":
        # the kernel reads the hot pool over HBM and the misses over the host
        # link at once: its bound is whichever would take longer at its peak
        t_link = gather_b / (link_memcpy * 1e9) if (M > 0 and link_memcpy) else 0.0
        t_hbm = attn_b / (hbm_peak * 1e9)
        if t_link >= t_hbm:
            roof = {"bound": "host_link", "achieved": gather_b / t_dom / 1e9, "peak": link_memcpy, "unit": "GB/s",
                    "peak_kind": "pinned H2D cudaMemcpyAsync, best of 10 x 1 GiB, measured in this run",
                    "traffic": profiled_traffic(att, wl_name),
                    "kernel": att_kernel + " (gather fused: missing chunks read over the host link)",
                    "hbm_achieved": attn_b / t_dom / 1e9}
        else:
            roof = {"bound": "hbm", "achieved": attn_b / t_dom / 1e9, "peak": hbm_peak, "unit": "GB/s",
                    "peak_kind": hbm_kind, "traffic": profiled_traffic(att, wl_name),
                    "kernel": att_kernel + (" (every chunk resident: K and V by TMA from the HBM pool)" if M == 0 else
                                            " (resident chunks by TMA from the HBM pool, misses over the host link)"),
                    "host_link_achieved": gather_b / t_dom / 1e9}
    elif dom == "gather":
        roof = {"bound": "host_link", "achieved": gather_b / t_dom / 1e9, "peak": link_memcpy, "unit": "GB/s",
                "peak_kind": "pinned H2D cudaMemcpyAsync, best of 10 x 1 GiB, measured in this run",
                "traffic": traffic, "kernel": "k_gather",
                "traffic_note": "DRAM bytes of one launch (ncu); the host-link reads are not DRAM traffic and most "
                                "staging writes stay in L2"}
    elif dom == "score" and folded:
        # the scoring stage's events bracket the selection kernel with the
        # scoring folded in: the landmark stream (the kernel's HBM bytes: its
        # selection works on chip and writes only the small union and miss
        # outputs) and the selection after it
        roof = {"bound": "hbm", "achieved": score_b / t_dom / 1e9, "peak": hbm_peak, "unit": "GB/s",
                "peak_kind": hbm_kind, "traffic": profiled_traffic("topk", w.name),
                "kernel": "k_select_fused with the scoring folded in (bytes: the landmark and query reads and the "
                          "score rows; the time: its scoring and its selection)"}
    else:
        roof = {"bound": "hbm", "achieved": stage_bytes[dom] / t_dom / 1e9, "peak": hbm_peak, "unit": "GB/s",
                "peak_kind": hbm_kind,
                "traffic": profiled_traffic(att, wl_name) if dom == "attention" else profiled_traffic(dom, w.name),
                "kernel": (att_kernel + " (every chunk from HBM: the hot pool and the staging buffer)"
                           if dom == "attention" else KERNEL_SOURCE[dom][0])}
    roof["frac"] = roof["achieved"] / roof["peak"] if roof["peak"] else None
    # the scoring pass is HBM-bound in every mode; when the attention reads its
    # chunks from HBM too (a separate gather into staging, or every chunk
    # resident), scoring + attention is also reported against the HBM peak
    # with the scoring folded into the selection kernel the stage events bracket
    # scoring and selection together; its rate is then taken from the kernel's
    # own timing words of its scoring phase (below)
    roof_hbm = {"bound": "hbm",
                "kernels": ("k_select_fused with the scoring folded in (its scoring phase: the landmark stream "
                            "on the tensor cores; bytes: the landmark and query reads)" if folded else
                            "k_score (the landmark stream; bytes: the landmark and query reads and the score rows)"),
                "achieved": score_b / (stage_ms["score"] * 1e-3) / 1e9,
                "peak": hbm_peak, "unit": "GB/s", "peak_kind": hbm_kind,
                "traffic": {"score": None if folded else profiled_traffic("score", w.name)}}
    roof_hbm["frac"] = roof_hbm["achieved"] / hbm_peak
    # the same fraction inside steps without events, from the kernels' own stamps
    tr_raw = trace.cpu().numpy().view(np.uint64)
    starts = tr_raw[:, :, 0].min(axis=2).astype(np.float64)         # [K, kernel]: the earliest CTA start
    ends = tr_raw[:, :, 1].max(axis=2).astype(np.float64)           # the latest CTA end
    in_step = {}
    for j, name in enumerate(("score", "select", "attention")):
        ok = (starts[:, j] < 2.0 ** 63) & (ends[:, j] > 0)
        in_step[name] = float(np.median(ends[ok, j] - starts[ok, j])) * 1e-3 if ok.any() else None
    ok = (starts[:, 0] < 2.0 ** 63) & (ends[:, 2] > 0)
    in_step["score_start_to_attention_end"] = float(np.median(ends[ok, 2] - starts[ok, 0])) * 1e-3 if ok.any() else None
    if folded and in_step["score"]:
        roof_hbm["achieved"] = score_b / (in_step["score"] * 1e-6) / 1e9
        roof_hbm["frac"] = roof_hbm["achieved"] / hbm_peak
    if in_step["score"]:
        roof_hbm["in_step"] = {"score_us": in_step["score"], "achieved": score_b / (in_step["score"] * 1e-6) / 1e9,
                               "frac": score_b / (in_step["score"] * 1e-6) / 1e9 / hbm_peak,
                               "note": ("the scoring phase of k_select_fused (scoring folded in) from its dependency "
                                        "wait to the last CTA's keys in place" if folded else
                                        "k_score from the end of the kernel before it (its dependency wait) to its last "
                                        "CTA's end") +
                                       ", stamped by the kernel (%globaltimer) in 200 further steps with no "
                                       "events between the kernels; its first landmark requests come before that "
                                       "wait, so this is the time scoring adds to the step; median over the steps"}
    if not fused or M == 0:
        t_sa = (stage_ms["score"] + stage_ms["attention"]) * 1e-3
        roof_hbm["score_plus_attention"] = {
            "kernels": ("the folded scoring phase + k_attn" if folded else "k_score + k_attn") +
                       " (bytes: landmarks, queries and scores + the union's K and V, each read once)",
            "achieved": (score_b + attn_b) / t_sa / 1e9, "frac": (score_b + attn_b) / t_sa / 1e9 / hbm_peak}
        if in_step["score"] and in_step["attention"]:
            t_in = (in_step["score"] + in_step["attention"]) * 1e-6
            roof_hbm["score_plus_attention"]["in_step_frac"] = (score_b + attn_b) / t_in / 1e9 / hbm_peak

    # the same steps captured in a CUDA graph (one capture of all layers) and replayed
    graph = None
    if mode != dd.GATHER_MEMCPY:
        gs = torch.cuda.Stream()
        with torch.cuda.stream(gs):
            for l in range(N_LAYERS):          # warm-up on the capture stream
                d_ = layers[l]
                ctx.step(l, d_.q, d_.lm, d_.Kh, d_.Vh, d_.slot, d_.Khot, d_.Vhot, Kst, Vst, out, mode=mode,
                         lm_kind=lm_kind, stream=gs, mass_gamma=args.mass_gamma,
                         softmax_scale=args.softmax_scale)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gs, capture_error_mode="relaxed"):
            for l in range(N_LAYERS):
                d_ = layers[l]
                ctx.step(l, d_.q, d_.lm, d_.Kh, d_.Vh, d_.slot, d_.Khot, d_.Vhot, Kst, Vst, out, mode=mode,
                         lm_kind=lm_kind, stream=gs, mass_gamma=args.mass_gamma,
                         softmax_scale=args.softmax_scale)
        reps = max(1, K // N_LAYERS)
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(gs):                  # a replay runs on the current stream
            for _ in range(3):
                cg.replay()
            torch.cuda.synchronize()
            tg_wall = time.time()
            ga.record(gs)
            for _ in range(reps):
                cg.replay()
            gb.record(gs)
        torch.cuda.synchronize()
        if sampler:
            sampler.window("graph replay", tg_wall, time.time())
        if ctx.status() != 0:
            raise RuntimeError("device status after the graph replays is not OK")
        g_s = max_over_ranks(ga.elapsed_time(gb) * 1e-3, world)
        graph = {"value": world * reps * N_LAYERS / g_s, "unit": UNIT,
                 "ms_per_step": 1e3 * g_s / (reps * N_LAYERS), "steps": reps * N_LAYERS,
                 "note": f"all {N_LAYERS} layers' steps captured once in a CUDA graph, replayed {reps} times"}
        del cg

    # end to end through the public call with host buffers: q in, out back
    out_host = torch.empty(out.numel(), dtype=torch.float32, pin_memory=True)
    for i in range(3):
        d_ = layers[i % N_LAYERS]
        d_.q.copy_(d_.q_host, non_blocking=True)
        step(i, i)
        out_host.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    te_wall = time.time()
    a.record()
    for i in range(K):
        layer = args.warmup + i
        d_ = layers[layer % N_LAYERS]
        d_.q.copy_(d_.q_host, non_blocking=True)
        step(i, layer)
        out_host.copy_(out, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.window("e2e steps", te_wall, time.time())
    e2e_s = max_over_ranks(a.elapsed_time(b) * 1e-3, world)
    barrier(world)
    lm_times = landmark_build_times(dd, shape, w, layers[0], lm_kind, sampler) if args.landmark_timing else None
    clocks = sampler.stop() if sampler else None

    cpu = cpu_baseline(w, landmarks=args.landmarks) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    cpu_all = (cpu_baseline_all_cores(w, landmarks=args.landmarks)
               if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None)
    ctx.close()
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": world * K / t_max, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_of(w, gather_used + (" (auto)" if args.mode == "auto" else ""), world,
                                 args.landmarks),
                       **({"selection": f"coverage budgets: gamma {args.mass_gamma}, at most k chunks",
                           "softmax_scale": args.softmax_scale or 1 / math.sqrt(w.d)}
                          if args.mass_gamma > 0 else {}),
                       **({"residency": "all: every chunk in an HBM pool, no host reads",
                           "workload": w.name + "_all_resident"} if resident_all else
                          {"residency": "none: every chunk read from host memory",
                           "workload": w.name + "_all_host"} if (args.residency == "none" and w.residency != "none")
                          else {"residency": (f"carry: {w.resident_frac:.0%} of each unit's union (taken from an "
                                              f"untimed step) resident in an HBM pool" if w.residency == "carry" else
                                              f"uniform: {w.resident_frac:.0%} of all chunks resident in an HBM pool")}
                          if own_residency else {})),
        "roofline": roof, "roofline_hbm": roof_hbm,
        "stages_us": {n: 1e3 * v for n, v in stage_ms.items()},
        "in_step_us": in_step,
        "stages_note": f"stages_us: mean over {n_stage} further steps with an event at every stage boundary "
                       f"('score' is the scoring kernel; with the fused selection 'topk' is the one kernel for "
                       f"top-k, union, residency, ordinals and plan, and 'resolve' and 'gather' are empty); "
                       f"{dom_timed}: {1e3 * dom_ms_timed:.1f} us inside the timed region (CUDA events around it "
                       f"on {len(ev_steps)} of the {K} timed steps, every {EV_EVERY}th, all layers); in_step_us: median "
                       f"over {n_trace} further steps with no events, from the kernels' own %globaltimer stamps "
                       f"(from the end of the kernel before, or for the attention from its first copy, to the last "
                       f"CTA's end)",
        "per_step": {"union_chunks": U, "missing_chunks": M, "gather_bytes": gather_b,
                     "host_link_gbs": gather_b / (dom_ms_timed * 1e-3) / 1e9},
        "host_link_peaks_gbs": {"memcpy_h2d": link_memcpy, "zero_copy_gather_sequential": link_zc},
        "wall_s": wall,
        "e2e": {"value": world * K / e2e_s, "unit": UNIT, "h2d_bytes_per_step": q_b,
                "d2h_bytes_per_step": w.B * w.n_q * w.Hq * w.d * 4},
        "graph_replay": graph,
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
    }
    if lm_times:
        hbm_peak_, _ = peaks()
        lm_times["pinned_host"]["frac_of_host_link"] = lm_times["pinned_host"]["gbs"] / link_memcpy
        lm_times["device"]["frac_of_hbm"] = lm_times["device"]["gbs"] / hbm_peak_
        line["landmark_build_us"] = lm_times
    if per_config is not None:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ the other workloads, one process each
PER_CONFIG = (
    (TINY.name, "workload"), (LLAMA8B_32K.name, "workload"), (QWEN8B_128K.name, "workload"),
    (STRESS_512K.name, "workload"), (LLAMA8B_32K.name, "all"), (GQA32B_5Q.name, "all"),
)


def _compact(line):
    """The figures of one workload's line that go into the headline's per_config."""
    keep = ("value", "ms_per_step", "steps", "warmup", "graph_replay", "e2e", "roofline", "per_step",
            "in_step_us", "stages_us", "gpu_launches", "clocks", "host_link_peaks_gbs")
    out = {"workload": line["config"]["workload"], "residency": line["config"]["residency"],
           "gather": line["config"]["gather"]}
    out.update({k: line.get(k) for k in keep})
    rh = line.get("roofline_hbm") or {}
    out["score"] = {"achieved_gbs": rh.get("achieved"), "frac": rh.get("frac"),
                    "in_step": rh.get("in_step")}
    if "score_plus_attention" in rh:
        out["score_plus_attention"] = rh["score_plus_attention"]
    if isinstance(out.get("clocks"), dict):
        out["clocks"] = {k: out["clocks"].get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")}
    return out


def run_per_config(args):
    """Every other workload (and the fully resident lines) through this same
    script, one child process each (each frees its pinned host KV at exit):
    warm-up, timed steps, stage breakdown, graph replay and e2e as in the
    headline line, no CPU baseline."""
    steps = max(20, min(args.steps, 300))
    out = []
    for name, residency in PER_CONFIG:
        if name == args.workload and residency == args.residency:
            continue
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", name, "--residency", residency,
               "--steps", str(steps), "--warmup", str(args.warmup), "--no-cpu-baseline", "--no-per-config",
               "--mode", args.mode]
        t0 = time.perf_counter()
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
            lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
            if r.returncode != 0 or not lines:
                out.append({"workload": name, "residency": residency, "error":
                            f"rc {r.returncode}: " + (r.stderr.strip().splitlines() or ["no output"])[-1][-300:]})
                continue
            item = _compact(json.loads(lines[-1]))
        except subprocess.TimeoutExpired:
            item = {"workload": name, "residency": residency, "error": "timed out after 900 s"}
        item["child_wall_s"] = time.perf_counter() - t0
        out.append(item)
    return out


# ------------------------------------------------------------------ pipelined decode (predictive prefetch)
DRIFT_T, SIGMA_DRIFT, SIGMA_SPEC = 8, 0.3, 0.1
RES_SLOTS_PER_K, RES_CAP_PER_K = 4, 4     # hot pool of 4k slots per (b,g); admit up to k/2 per step


class LayerGap:
    """Stand-in for the rest of a layer between two layers' sparse steps.
    ``gemm``: the projections and MLP, one bf16 GEMM of the step's tokens
    against a weight matrix streamed from HBM, sized so that it takes about
    ``us`` microseconds (a decode GEMM with few rows is bound by the weight
    reads; it occupies every SM).  ``idle``: work that leaves the SMs free
    (one thread spinning for ``us``), such as a wait on another device."""

    def __init__(self, us, tokens, d_model=4096, kind="gemm"):
        import torch
        self.us = us
        self.kind = kind
        self.x = None
        self.cycles = 0
        if us <= 0:
            self.measured_us = 0.0
            return
        if kind == "idle":
            self.cycles = max(1, int(us * 2000.0))     # a first guess at 2 GHz, then calibrated by timing
            for _ in range(2):
                t = self._time()
                self.cycles = max(1, int(self.cycles * us / t))
            self.measured_us = self._time()
            self.shape = None
            return
        self.x = torch.randn(tokens, d_model, dtype=torch.bfloat16, device="cuda")
        n = max(256, int(us * 1e-6 * 6.0e12 / (2 * d_model)) // 256 * 256)
        for _ in range(3):                      # calibrate the width against the measured time
            self.W = torch.randn(d_model, n, dtype=torch.bfloat16, device="cuda")
            t = self._time()
            n = max(256, int(n * us / t) // 256 * 256)
        self.W = torch.randn(d_model, n, dtype=torch.bfloat16, device="cuda")
        self.measured_us = self._time()
        self.shape = (tokens, d_model, n)

    def _time(self, reps=20):
        import torch
        for _ in range(3):
            self.run()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            self.run()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) * 1e3 / reps

    def run(self, stream=None):
        import torch
        if self.cycles:
            with torch.cuda.stream(stream or torch.cuda.current_stream()):
                torch.cuda._sleep(self.cycles)
            return
        if self.x is None:
            return
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            torch.matmul(self.x, self.W)


def run_pipeline(args, world, rank, local):
    """Decode steps over N_LAYERS layers whose queries drift from step to step,
    with the speculative rows of each layer's selection prefetched for its next
    step: after layer l's attention, a low-priority stream fetches the predicted
    chunks of layer l+2 into the transfer half of the staging buffer that layer
    l has just released (same parity), while the high-priority stream runs the
    next layers; each step resolves its true selection against the prefetch map
    and fetches only the chunks the prediction missed (urgent, inside the
    attention kernel).  The same drifting steps are also timed without prefetch."""
    import torch
    torch.cuda.set_device(local)
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd
    w = BY_NAME[args.workload]
    shape = dd.Shape(w.B, w.Hq, w.Hkv, w.d, w.L, w.cs, w.k, w.n_q)
    N, T, units = N_LAYERS, DRIFT_T, w.B * w.Hkv
    if w.n_q < 2:
        raise SystemExit("the pipelined mode predicts from speculative queries: n_q >= 2")
    layers = [LayerData(dd, shape, w, l, rank) for l in range(N)]
    seed = rank_seed(w.seed, rank)
    qs = []
    for l in range(N):
        qh = synth.drift_queries(seed, w.B, w.n_q, w.Hq, w.d, T, SIGMA_DRIFT, SIGMA_SPEC, layer=l)
        qs.append(torch.from_numpy(qh.reshape(T, -1).view(np.int16)).view(torch.bfloat16).cuda())
    cap = w.max_misses
    ctx_hi = dd.Context(shape, max_misses=cap, hot_slots=cap)
    ctx_lo = dd.Context(shape, max_misses=cap)
    touch = torch.empty(w.B * w.Hkv * w.C * w.d, dtype=torch.bfloat16, device="cuda")
    for L_ in layers:
        ctx_hi.build_landmarks(L_.Kh, L_.lm)
        ctx_hi.build_landmarks(L_.Vh, touch)
    del touch
    ns = cap * w.cs * w.d
    Kpf = [torch.empty(ns, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Vpf = [torch.empty(ns, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Kurg = [torch.empty(ns, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Vurg = [torch.empty(ns, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    pf_map = [torch.full((units * w.C,), -1, dtype=torch.int32, device="cuda") for _ in range(2)]
    none_res = torch.full((units * w.C,), -1, dtype=torch.int32, device="cuda")
    sel_store = [torch.empty(w.B * w.n_q * w.Hkv * w.k, dtype=torch.int32, device="cuda") for _ in range(N)]
    out = torch.empty(w.B * w.n_q * w.Hq * w.d, dtype=torch.float32, device="cuda")
    K = args.steps
    miss = torch.zeros(K * N, dtype=torch.int32, device="cuda")
    ucnt = torch.zeros(K * N, units, dtype=torch.int32, device="cuda")
    pfc = torch.zeros(K * N, dtype=torch.int32, device="cuda")
    hi = torch.cuda.Stream(priority=-1)
    lo = torch.cuda.Stream(priority=0)
    ev_step = [torch.cuda.Event() for _ in range(N)]
    ev_pf = [torch.cuda.Event() for _ in range(N)]
    torch.cuda.synchronize()
    link_memcpy, _ = host_link_peaks(dd, shape)
    gap = LayerGap(args.layer_gap_us, w.B * w.n_q, kind=args.layer_gap_kind)
    pf_ev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(K * N)]

    def q_of(i, l):
        return qs[l][i % T]

    n_rec = [0]

    def prefetch(t, p, record=False):
        count = None
        if record and n_rec[0] < pfc.numel():
            count = pfc[n_rec[0]:n_rec[0] + 1]
            n_rec[0] += 1
        L_ = layers[t]
        timed = count is not None
        if timed:
            pf_ev[n_rec[0] - 1][0].record(lo)
        ctx_lo.prefetch_kv(sel_store[t], w.n_q - 1, L_.Kh, L_.Vh, Kpf[p], Vpf[p], pf_map[p], pf_count=count,
                           ctas_per_sm=args.prefetch_ctas, stream=lo, sel_rows=w.n_q, first_row=1)
        if timed:
            pf_ev[n_rec[0] - 1][1].record(lo)
        ev_pf[t].record(lo)

    def pipelined(i, rec=None):
        for l in range(N):
            p, L_ = l & 1, layers[l]
            hi.wait_event(ev_pf[l])
            inter = {"sel": sel_store[l]}
            if rec is not None:
                inter.update(miss_count=miss[rec * N + l:rec * N + l + 1], union_cnt=ucnt[rec * N + l])
            ctx_hi.step(i * N + l, q_of(i, l), L_.lm, L_.Kh, L_.Vh, pf_map[p], Kpf[p], Vpf[p], Kurg, Vurg, out,
                        intermediates=inter, stream=hi)
            ev_step[l].record(hi)
            t = (l + 2) % N
            lo.wait_event(ev_step[l])
            prefetch(t, p, record=rec is not None)
            gap.run(hi)

    def serialized(i, events=None):
        for l in range(N):
            L_ = layers[l]
            ctx_hi.step(i * N + l, q_of(i, l), L_.lm, L_.Kh, L_.Vh, none_res, Kpf[0], Vpf[0], Kurg, Vurg, out,
                        stream=hi, stage_events=None if events is None else events[l])
            gap.run(hi)

    # prime: one step of every layer without prediction fills the selections, then the
    # prefetches of layers 0 and 1 for the first pipelined step
    with torch.cuda.stream(hi):
        for l in range(N):
            L_ = layers[l]
            ctx_hi.step(l, q_of(T - 1, l), L_.lm, L_.Kh, L_.Vh, none_res, Kpf[0], Vpf[0], Kurg, Vurg, out,
                        intermediates={"sel": sel_store[l]}, stream=hi)
            ev_step[l].record(hi)
        for t in (0, 1):
            lo.wait_event(ev_step[N - 1])
            prefetch(t, t)
    for i in range(args.warmup):
        pipelined(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(hi)
    for i in range(K):
        pipelined(args.warmup + i, rec=i)
    lo_done = torch.cuda.Event()
    lo_done.record(lo)
    hi.wait_event(lo_done)
    b.record(hi)
    torch.cuda.synchronize()
    t_pipe = a.elapsed_time(b) * 1e-3
    st_hi, st_lo = ctx_hi.status(), ctx_lo.status()
    if st_hi or st_lo:
        raise RuntimeError(f"device status after the pipelined steps: {dd.status_str(st_hi or st_lo)}")

    # the same drifting steps, serialized, nothing prefetched
    for i in range(args.warmup):
        serialized(i)
    torch.cuda.synchronize()
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a2.record(hi)
    for i in range(K):
        serialized(args.warmup + i)
    b2.record(hi)
    torch.cuda.synchronize()
    t_ser = a2.elapsed_time(b2) * 1e-3
    assert ctx_hi.status() == 0

    # OasisKV eq. (4) terms, each on its own: T_pred = the step's scoring + selection
    # (the predicted rows are the speculative rows of the step's own selection),
    # T_select = resolving the predicted rows into a transfer plan (union, ordinals),
    # T_transfer = copying the planned chunks from pinned host memory
    n_ev = min(K, 20)
    st_ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(N)] for _ in range(n_ev)]
    for row in st_ev:
        for evs in row:
            for e in evs:
                e.record()                  # creates the event handles the step records into
    with torch.cuda.stream(hi):
        for i in range(n_ev):
            serialized(args.warmup + i, st_ev[i])
    torch.cuda.synchronize()
    t_pred = float(np.mean([st_ev[i][l][0].elapsed_time(st_ev[i][l][2]) for i in range(n_ev) for l in range(N)]))
    shape_p = dd.Shape(w.B, w.Hq, w.Hkv, w.d, w.L, w.cs, w.k, w.n_q - 1)
    t_sel, t_xfer = [], []
    with dd.Context(shape_p, max_misses=cap) as ctx_p:
        ui = torch.empty(units * shape_p.umax, dtype=torch.int32, device="cuda")
        us_ = torch.empty_like(ui)
        uq = torch.empty(units * shape_p.umax, dtype=torch.uint8, device="cuda")
        uc = torch.empty(units, dtype=torch.int32, device="cuda")
        ml = torch.empty(cap, dtype=torch.int32, device="cuda")
        mc = torch.empty(1, dtype=torch.int32, device="cuda")
        for r in range(3 + n_ev):
            for l in range(N):
                pred = sel_store[l].view(w.B, w.n_q, w.Hkv, w.k)[:, 1:].contiguous()
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record()
                ctx_p.resolve_union(pred, none_res, ui, us_, uq, uc, ml, mc)
                e[1].record()
                ctx_p.gather_kv(layers[l].Kh, layers[l].Vh, ml, mc, Kpf[0], Vpf[0], mode=dd.GATHER_KERNEL)
                e[2].record()
                torch.cuda.synchronize()
                if r >= 3:
                    t_sel.append(e[0].elapsed_time(e[1]))
                    t_xfer.append(e[1].elapsed_time(e[2]))
        assert ctx_p.status() == 0
    ctx_hi.close()
    ctx_lo.close()

    # lower bound: the same steps (and gaps) with every chunk of every layer resident in an HBM pool
    ctx_a = dd.Context(shape, max_misses=cap, hot_slots=units * w.C)
    ident = torch.arange(units * w.C, dtype=torch.int32, device="cuda")
    pools_all = [(L_.Kh.to("cuda"), L_.Vh.to("cuda")) for L_ in layers]

    def resident(i):
        for l in range(N):
            L_ = layers[l]
            ctx_a.step(i * N + l, q_of(i, l), L_.lm, L_.Kh, L_.Vh, ident, pools_all[l][0], pools_all[l][1], Kurg,
                       Vurg, out, stream=hi)
            gap.run(hi)

    with torch.cuda.stream(hi):
        for i in range(args.warmup):
            resident(i)
    torch.cuda.synchronize()
    a4, b4 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a4.record(hi)
    for i in range(K):
        resident(args.warmup + i)
    b4.record(hi)
    torch.cuda.synchronize()
    t_all = a4.elapsed_time(b4) * 1e-3
    assert ctx_a.status() == 0
    ctx_a.close()
    del pools_all

    # the same drifting steps with a per-(b,g) hot pool kept by the capped LRU
    # residency update after every step (OasisKV delta selection)
    S, cap_r = RES_SLOTS_PER_K * w.k, RES_CAP_PER_K * w.k // 8
    ctx_r = dd.Context(shape, max_misses=cap, hot_slots=units * S)
    nh = units * S * w.cs * w.d
    pools = []
    for _ in range(N):
        pools.append(dict(rs=torch.full((units * w.C,), -1, dtype=torch.int32, device="cuda"),
                          sc=torch.full((units * S,), -1, dtype=torch.int32, device="cuda"),
                          lu=torch.full((units * S,), -1, dtype=torch.int32, device="cuda"),
                          K=torch.empty(nh, dtype=torch.bfloat16, device="cuda"),
                          V=torch.empty(nh, dtype=torch.bfloat16, device="cuda")))
    inter_r = {"union_idx": torch.empty(units * shape.umax, dtype=torch.int32, device="cuda"),
               "union_slot": torch.empty(units * shape.umax, dtype=torch.int32, device="cuda"),
               "union_cnt": torch.empty(units, dtype=torch.int32, device="cuda")}
    miss_r = torch.zeros(K * N, dtype=torch.int32, device="cuda")

    def with_residency(i, rec=None):
        for l in range(N):
            L_, P_ = layers[l], pools[l]
            g_ = i * N + l
            inter = dict(inter_r)
            inter["miss_count"] = miss_r[rec * N + l:rec * N + l + 1] if rec is not None else miss_r[:1]
            ctx_r.step(g_, q_of(i, l), L_.lm, L_.Kh, L_.Vh, P_["rs"], P_["K"], P_["V"], Kurg, Vurg, out,
                       intermediates=inter, stream=hi)
            ctx_r.update_residency(i + 1, cap_r, S, Kurg[g_ & 1], Vurg[g_ & 1], P_["rs"], P_["sc"], P_["lu"],
                                   P_["K"], P_["V"], union_idx=inter["union_idx"], union_slot=inter["union_slot"],
                                   union_cnt=inter["union_cnt"], miss_count=inter["miss_count"], stream=hi)
            gap.run(hi)

    for i in range(max(args.warmup, 2 * T)):       # fill the pools
        with_residency(i)
    torch.cuda.synchronize()
    a3, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a3.record(hi)
    for i in range(K):
        with_residency(max(args.warmup, 2 * T) + i, rec=i)
    b3.record(hi)
    torch.cuda.synchronize()
    t_res = a3.elapsed_time(b3) * 1e-3
    assert ctx_r.status() == 0
    ctx_r.close()
    M_res = miss_r.double().mean().item()
    t_max = max_over_ranks(t_pipe, world)
    U = ucnt.double().sum(1).mean().item()
    M = miss.double().mean().item()
    P = pfc[:max(1, n_rec[0])].double().mean().item()
    chunk_b = 2 * w.cs * w.d * 2
    if rank != 0:
        return 0
    steps = K * N
    line = {
        "metric": METRIC + " (pipelined, predictive prefetch)", "value": world * steps / t_max, "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": args.warmup * N, "ms_per_step": 1e3 * t_max / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_of(w, "zerocopy", world), workload=w.name + "_drift_pipelined", layers=N,
                       queries=f"real query of step t = base + {SIGMA_DRIFT} N(0,1), cyclic over {T} steps; "
                               f"speculative queries of step t = real query of step t+1 + {SIGMA_SPEC} N(0,1)",
                       prefetch="rows 1..n_q-1 of each layer's selection, for its next step, issued after the "
                                f"attention of layer l-2 on a low-priority stream ({args.prefetch_ctas} CTAs/SM)"),
        "per_layer_step": {"true_union_chunks": U, "urgent_chunks": M, "prefetched_chunks": P,
                           "prediction_hit_rate": 1.0 - M / U if U else None,
                           "urgent_bytes": M * chunk_b, "prefetch_bytes": P * chunk_b,
                           "host_link_gbs": (M + P) * chunk_b * steps / t_pipe / 1e9},
        "layer_gap": {"requested_us": args.layer_gap_us, "measured_us": gap.measured_us, "kind": args.layer_gap_kind,
                      "what": ("none: the sparse path alone, layer after layer" if args.layer_gap_us <= 0 else
                               "between layers, one thread spinning (the SMs stay free), standing in for a wait"
                               if args.layer_gap_kind == "idle" else
                               "between layers, a bf16 GEMM of the step's tokens against a weight matrix read from "
                               f"HBM (shape {getattr(gap, 'shape', None)}), standing in for projections and MLP")},
        "serialized_same_steps": {"value": steps / t_ser, "unit": UNIT, "ms_per_step": 1e3 * t_ser / steps},
        "all_resident_same_steps": {"value": steps / t_all, "unit": UNIT, "ms_per_step": 1e3 * t_all / steps,
                                    "note": "every chunk of every layer in an HBM pool: no host transfer at all"},
        "exposed_gather_us_per_layer_step": {
            "pipelined": 1e6 * (t_pipe - t_all) / steps, "serialized": 1e6 * (t_ser - t_all) / steps,
            "note": "time per layer-step above the same steps with every chunk resident (gaps included in both)"},
        "eq4": {"T_pred_us": 1e3 * t_pred, "T_select_us": 1e3 * float(np.mean(t_sel)),
                "T_transfer_us": 1e3 * float(np.mean(t_xfer)),
                "T_pipe_us": 1e3 * max(t_pred, float(np.mean(t_sel)), float(np.mean(t_xfer))),
                "delta_prefetch_us": 1e6 * t_pipe / steps,
                "holds": max(t_pred, float(np.mean(t_sel)), float(np.mean(t_xfer))) * 1e-3 <= t_pipe / steps,
                "prefetch_in_pipeline_us": float(np.mean([e0.elapsed_time(e1) for e0, e1 in pf_ev[:n_rec[0]]]))
                * 1e3 if n_rec[0] else None,
                "note": "OasisKV eq. (4): T_pipe = max(T_pred, T_select, T_transfer) <= Delta_prefetch = T_step / "
                        "N_layer. T_pred: the step's scoring + selection (its speculative rows are the prediction); "
                        "T_select: union and ordinals of the predicted rows (k_union + k_assign); T_transfer: the "
                        "zero-copy gather of the planned chunks (k_gather); each timed on its own, mean over the "
                        "layers; Delta_prefetch: the pipelined time per layer-step"},
        "residency_same_steps": {"value": steps / t_res, "unit": UNIT, "ms_per_step": 1e3 * t_res / steps,
                                 "slots_per_unit": S, "cap_per_unit_and_step": cap_r,
                                 "missing_chunks_per_layer_step": M_res,
                                 "note": "serialized steps, each followed by the capped LRU residency update"},
        "host_link_peaks_gbs": {"memcpy_h2d": link_memcpy},
        "e2e": None,
        "gpu_launches": None,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=GQA32B_5Q.name, choices=sorted(BY_NAME))
    ap.add_argument("--mode", choices=("auto", "zerocopy", "kernel", "memcpy"), default="auto",
                    help="gather: auto (the library's choice: the separate gather kernel when there is a hot pool, "
                         "else fused into the attention), zerocopy (fused), kernel (separate), memcpy")
    ap.add_argument("--landmarks", choices=("mean", "minmax"), default="mean")
    ap.add_argument("--mass-gamma", type=float, default=0.0,
                    help="> 0: coverage budgets (smallest chunk set reaching this attention mass, at most k)")
    ap.add_argument("--softmax-scale", type=float, default=0.0, help="<= 0: 1/sqrt(d)")
    ap.add_argument("--residency", choices=("workload", "none", "all"), default="workload",
                    help="workload: the workload's own residency (none, a carried share of the union, or a "
                         "uniform share of all chunks in an HBM pool); none: every chunk read from host memory; "
                         "all: the whole KV also in an HBM pool (no misses; attention bound by HBM)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' lines (per_config; run only at N=1 with the default workload)")
    ap.add_argument("--no-landmark-timing", action="store_true", help="skip the separate landmark-build timing")
    ap.add_argument("--prefetch-ctas", type=int, default=2, help="pipelined mode: prefetch copy CTAs per SM")
    ap.add_argument("--layer-gap-kind", choices=("gemm", "idle"), default="gemm",
                    help="pipelined mode: the gap's work (a weight-streaming GEMM on every SM, or one spinning thread)")
    ap.add_argument("--layer-gap-us", type=float, default=0.0,
                    help="pipelined mode: microseconds of other per-layer work (a weight-streaming GEMM) between "
                         "two layers' sparse steps")
    ap.add_argument("--pipeline", action="store_true",
                    help="decode steps over several layers with drifting queries and predictive prefetch")
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="layers whose inputs the steps cycle through (fewer than 4 only to hold less device "
                         "memory under a profiler: one layer's inputs then stay in L2 between steps)")
    ap.add_argument("--batch", type=int, default=0,
                    help="> 0: the workload with this many requests instead of its own (a smaller case of the same "
                         "kernels for profiler captures; named <workload>_b<B>)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.batch > 0:
        w = BY_NAME[args.workload]
        ws = w.scaled(name=f"{w.name}_b{args.batch}", B=args.batch)
        BY_NAME[ws.name] = ws
        args.workload = ws.name
        args.no_per_config = True
        args.no_cpu_baseline = True   # the oracle's worker processes know the named workloads only
    if args.layers < 1:
        ap.error("--layers must be at least 1")
    globals()["N_LAYERS"] = args.layers
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.pipeline:
            return run_pipeline(args, world, rank, local)
        args.landmark_timing = not args.no_landmark_timing and not args.no_per_config
        per_config = None
        if world == 1 and not args.no_per_config:
            # the other workloads first, in child processes, while this process holds no GPU memory
            per_config = run_per_config(args)
        return run_ours(args, world, rank, local, per_config)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
