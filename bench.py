#!/usr/bin/env python
"""Forward throughput of multi-round LSH attention on B300 (tokens/s = B*H*L per second).

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference] [--workload NAME]
                    [--pass forward|backward|knn|revblock]

Default workload: the long-text shape B=1, H=8, L=65536, d=128, bf16, 1024 buckets,
8 rounds, chunk 64, causal (the headline L = 64K, 8-round configuration).  Each rank runs
its own copy of the workload (independent heads: weak scaling, no data-path collective).
Rank 0 prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same workload instead.  ``--pass backward`` times lsh_attn_backward (the
gradients in qk and v) on the same workload instead of the forward pass, with its own
metric line; ``--pass knn`` the LSH k-nearest-neighbour search (k = 16) on it;
``--pass revblock`` one reversible residual block around the attention at the long-text
shape (d_model 1024 = 8 heads of 128, d_ff 4096), forward.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LSH-attention fwd tokens/s (B·H·L per sec) at L=64K, 8 rounds; % of roofline"
METRIC_BWD = "LSH-attention bwd tokens/s (B·H·L per sec) at L=64K, 8 rounds: dqk, dv"
METRIC_KNN = "LSH approximate k-NN tokens/s (B·H·L per sec) at L=64K, 8 rounds, k=16; recall@k"
METRIC_REV = ("Reversible LSH-attention block fwd tokens/s (B·L per sec) at L=64K, d_model 1024, "
              "8 heads, d_ff 4096, 8 rounds")
KNN_K = 16
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_BYTES = 126 * 2 ** 20
# fp32 FFMA peak from unit counts: 148 SMs x 128 lanes x 2 flop x 2.032 GHz
FP32_ALU_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


# Where each kernel's arithmetic runs: the bf16 contractions (hash projection, QK^T and
# P V) on the tensor cores, the fp32 ones on the CUDA cores' FFMA lanes.  A kernel's
# bound is the slower of its FLOPs at that peak and its bytes at HBM bandwidth.
COMPUTE_UNIT = {"bf16": "tensor", "f16": "tensor", "f32": "alu"}
# fp16 and bf16 have the same nominal dense tensor rate, so fp16 contractions use the
# measured bf16 peak.
ESIZE = {"f32": 4, "bf16": 2, "f16": 2}


def dt_code_of(lsh, w):
    return {"f32": lsh.LSH_F32, "bf16": lsh.LSH_BF16, "f16": lsh.LSH_F16}[w.dtype]


def torch_dtype_of(torch, w):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.dtype]
# Kernel sources per stage: a DRAM-traffic figure recorded from ncu counts only while
# these files are unchanged.
KERNEL_SOURCES = {
    "hash": ["hash_tc.cu", "sm100.cuh", "tmap.cu"],
    "sort": ["sort.cu"],
    "attn": ["attn_tc.cu", "sm100.cuh"],
    "combine": ["combine.cu", "combine_tma.cu", "sm100.cuh"],
    "attn_bwd": ["attn_bwd.cu", "attn_bwd_tc.cu"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK, "fallback"


def source_digest(stage):
    import hashlib
    h = hashlib.sha1()
    for f in KERNEL_SOURCES[stage]:
        with open(os.path.join(ROOT, "lsh_attention_04_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(workload, stage):
    """DRAM bytes per launch of `stage` on `workload` from the ncu summary, or None when
    there is none or the kernel's sources changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        k = rec[workload][stage]
    except (OSError, ValueError, KeyError):
        return None
    return k["bytes_per_launch"] if k.get("source_sha1") == source_digest(stage) else None


# ------------------------------------------------------------------ algorithmic work


def work(w):
    """Algorithmic FLOPs and bytes per kernel for one forward pass of workload w."""
    N, R, d, nb, c = w.tokens, w.n_rounds, w.d, w.n_buckets, w.chunk
    e = ESIZE[w.dtype]
    wr = e                                   # o_r element width
    S = w.B * w.H * R
    k = {}
    k["hash"] = dict(flops=N * R * d * nb,   # N*R*(nb/2) dot products of length d
                     bytes=N * d * e + R * d * (nb // 2) * e + N * R * 4 + N * 4)
    k["sort"] = dict(flops=0, bytes=N * R * 4 + N * R * 8 + S * (nb + 1) * 4)
    k["attn"] = dict(flops=8 * N * R * c * d,  # QK^T and PV over the c x 2c window
                     bytes=2 * N * d * e + N * R * (d * wr + 4) + N * R * 8 + N * 4)
    # token-order rows (fused forward): o_r and lse_r read once, no inverse permutation
    k["combine"] = dict(flops=0, bytes=N * R * (d * wr + 4) + N * (4 * d + 4))
    return k


def work_backward(w):
    """Algorithmic FLOPs and bytes per kernel for one backward pass of workload w: the
    hash and sort recomputed, then the attention backward.  Per token and round that
    kernel does five contractions over the c x 2c window (Q K^T again, g_out V^T, and the
    gradients in q, k and v), 4 c d flops each; it reads qk, v, out, g_out, lse, g_lse,
    the inverse norms, buckets and perm once and writes dqk and dv once."""
    N, R, d, c = w.tokens, w.n_rounds, w.d, w.chunk
    e = ESIZE[w.dtype]
    k = work(w)
    return {
        "hash": k["hash"],
        "sort": k["sort"],
        "attn_bwd": dict(flops=20 * N * R * c * d,
                         bytes=2 * N * d * e + 2 * N * d * 4 + 3 * N * 4 + 2 * N * R * 4
                         + 2 * N * d * 4),
    }


def kernel_roof(w, name, ms, wk, unit_c, peak_c, peaks, peak_src):
    """Roofline entry of one kernel: the slower of its FLOPs at the compute peak and its
    bytes at HBM bandwidth decides the bound; achieved = algorithmic work / measured time."""
    t = ms / 1e3
    f, by = wk["flops"], wk["bytes"]
    t_c = f / (peak_c * 1e12)
    t_b = by / (peaks["hbm_gbs"] * 1e9)
    if t_c > t_b:
        b, ach, peak, unit = unit_c, f / t / 1e12, peak_c, "TFLOP/s"
        src = (f"{peak_src} bf16 burst" if unit_c == "tensor" else "fp32 lanes x clock")
    else:
        b, ach, peak, unit = "hbm", by / t / 1e9, peaks["hbm_gbs"], "GB/s"
        src = f"{peak_src} copy bandwidth"
    r = {"bound": b, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
         "traffic": recorded_traffic(w.name, name), "kernel": name, "ms": ms,
         "roof_ms": 1e3 * max(t_c, t_b), "algorithmic_flops": f, "algorithmic_bytes": by,
         "peak_source": src}
    if f and unit_c == "tensor":
        r["tensor_frac"] = f / t / 1e12 / peak_c   # of the measured dense bf16 peak
    return r


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle


def oracle_sample(w, max_tokens=32768):
    """A bounded sample of workload w for the fp64 oracle: head 0, the first
    min(L, max_tokens) tokens (a multiple of two chunks), all rounds, the workload's
    bucket count and chunk.  The oracle's work per token does not depend on L (fixed
    chunk and bucket count), so its tokens/s carries over to the whole workload."""
    from lsh_attention_04_b300 import inputs as gen
    Ls = min(w.L, max(2 * w.chunk, (max_tokens // (2 * w.chunk)) * (2 * w.chunk)))
    sub = w.replace(B=1, H=1, L=Ls)
    qk, v, R = gen.make_inputs(sub, seed=w.seed)
    desc = (f"head 0 of {w.name}: first {Ls} tokens, {w.n_rounds} rounds, "
            f"{w.n_buckets} buckets, chunk {w.chunk} (same per-token hash work)")
    return sub, qk, v, R, desc


def cpu_model():
    """The host CPU's model name from /proc/cpuinfo (None where unavailable)."""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def time_oracle(w, threads, steps=1, max_tokens=32768, keep=None):
    """Time the oracle's forward pass on a bounded sample of w.  With ``keep`` (a dict),
    the last run's inputs and per-round buckets and margins are stored in it."""
    import oracle
    sub, qk, v, R, desc = oracle_sample(w, max_tokens)
    oracle.build()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        res = oracle.forward(qk, v, R, sub.n_buckets, sub.chunk, sub.causal, sub.scale,
                             threads=threads, intermediates=keep is not None)
        times.append(time.perf_counter() - t0)
    if keep is not None:
        keep.update(sub=sub, qk=qk, R=R, bucket=res[2]["bucket"], margin=res[2]["margin"])
    used = min(threads, sub.B * sub.H * sub.n_rounds)
    return sub.tokens, times, used, desc


def near_tie_report(lsh, dev, keep, band=1e-5):
    """Bucket mismatches between the GPU hash and the oracle's buckets of the CPU-baseline
    sample (the same input values on both sides).  A mismatch is allowed only where the
    oracle's top-1/top-2 margin is below band * |x| * |R| (|R| = largest column 2-norm of
    R_r); the line reports both counts."""
    import torch
    sub = keep["sub"]
    tdt = torch_dtype_of(torch, sub)
    d_qk = torch.from_numpy(keep["qk"]).to(dev).to(tdt).contiguous()
    d_R = torch.from_numpy(keep["R"]).to(dev).to(tdt).contiguous()
    b, _ = lsh.lsh_hash(d_qk, d_R, sub.n_buckets)
    gb = b.cpu().numpy().reshape(keep["bucket"].shape)
    bad = gb != keep["bucket"]
    xn = np.linalg.norm(keep["qk"].reshape(-1, sub.d).astype(np.float64), axis=1)
    rn = np.linalg.norm(keep["R"].astype(np.float64), axis=1).max(axis=1)
    lim = band * xn.reshape(sub.B, sub.H, 1, sub.L) * rn.reshape(1, 1, -1, 1)
    return {"buckets_compared": int(gb.size), "mismatches": int(bad.sum()),
            "outside_band": int((bad & ~(keep["margin"] < lim)).sum()),
            "band": f"{band:g}*|x|*|R|", "sample": "the cpu_baseline sample"}


def time_oracle_backward(w, steps=1, max_tokens=4096):
    """The oracle's backward pass (one thread per head: a single head here) on a bounded
    sample of w, with seeded output gradients."""
    import oracle
    sub, qk, v, R, desc = oracle_sample(w, max_tokens)
    rng = np.random.default_rng(w.seed + 5)
    g_out = rng.standard_normal(qk.shape)
    g_lse = rng.standard_normal(qk.shape[:-1])
    oracle.build()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.backward(qk, v, R, sub.n_buckets, sub.chunk, sub.causal, sub.scale, g_out, g_lse)
        times.append(time.perf_counter() - t0)
    return sub.tokens, times, 1, desc + "; backward (forward recomputed inside)"


# ------------------------------------------------------------------ runs


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return world, rank, local, dist
    return world, rank, local, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def allmax(dist, x):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank, world, ms_max):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return tokens_per_rank * world / (ms_max / 1e3)


def run_reference(args, w):
    # the CPU oracle runs on rank 0 only; other ranks have nothing to do
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    threads = os.cpu_count() or 1
    # Bound the whole run to a couple of minutes: one 32K-token sample takes a few
    # seconds, so many requested steps get proportionally smaller samples.
    n = args.warmup + args.steps
    if args.pass_ == "backward":
        max_tokens = 4096 if n <= 10 else max(2 * w.chunk, 4096 * 10 // n)
        tokens, times, used, desc = time_oracle_backward(w, steps=n, max_tokens=max_tokens)
    elif args.pass_ == "knn":
        max_tokens = 8192 if n <= 10 else max(2 * w.chunk, 8192 * 10 // n)
        times, used = [], 1
        for _ in range(n):
            tokens, t, desc = time_oracle_knn(w, KNN_K, max_tokens)
            times.append(t)
    else:
        max_tokens = 32768 if n <= 40 else max(2 * w.chunk, 32768 * 40 // n)
        tokens, times, used, desc = time_oracle(w, threads, steps=n, max_tokens=max_tokens)
    timed = times[args.warmup:]
    t = sum(timed) / len(timed)
    value = tokens / t
    line = {
        "impl": "reference",
        "metric": {"backward": METRIC_BWD, "knn": METRIC_KNN}.get(args.pass_, METRIC),
        "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_revblock(args, bw):
    """The oracle's reversible block as the reference arm: rank 0 only, each step a
    bounded sample sized so the run ends within a few minutes."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    n = args.warmup + args.steps
    max_tokens = 2048 if n <= 10 else max(2 * bw.chunk, 2048 * 10 // n)
    times = []
    for _ in range(n):
        tok, t, desc = time_oracle_revblock(bw, max_tokens)
        times.append(t)
    timed = times[args.warmup:]
    t = sum(timed) / len(timed)
    value = tok / t
    line = {
        "impl": "reference", "metric": METRIC_REV, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "pass": "revblock",
        "config": {"workload": bw.name, "B": bw.B, "L": bw.L, "d_model": bw.d_model,
                   "heads": bw.heads, "d_ff": bw.d_ff, "n_buckets": bw.n_buckets,
                   "n_rounds": bw.n_rounds, "chunk": bw.chunk, "causal": bw.causal,
                   "ff_chunk": bw.ff_chunk},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d,
            "n_buckets": w.n_buckets, "n_rounds": w.n_rounds, "chunk": w.chunk,
            "causal": w.causal, "scale": "1/sqrt(d)", "qk": "clustered" if w.clusters else "gauss",
            "clusters": w.clusters}


def run_ours(args, w):
    import torch
    import lsh_attention_04_b300 as lsh
    from lsh_attention_04_b300 import inputs as gen

    world, rank, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = lsh.load()
    dt_code = dt_code_of(lsh, w)
    tdt = torch_dtype_of(torch, w)

    qk, v, R = gen.make_inputs(w, seed=w.seed + 7919 * rank)
    h_qk = torch.from_numpy(qk).to(tdt).pin_memory()
    h_v = torch.from_numpy(v).to(tdt).pin_memory()
    h_R = torch.from_numpy(R).to(tdt).pin_memory()
    d_qk = h_qk.to(dev)
    d_v = h_v.to(dev)
    d_R = h_R.to(dev)
    out = torch.empty((w.B, w.H, w.L, w.d), dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=dev)
    ws = lsh.workspace(w.B, w.H, w.L, w.d, w.n_buckets, w.n_rounds, w.chunk, dt_code, dev)
    stream = torch.cuda.current_stream(dev)
    K, Wm = args.steps, args.warmup

    def fwd(events=None):
        if events is None:
            lsh.lsh_attn_forward(d_qk, d_v, d_R, w.n_buckets, w.chunk, w.causal, w.scale,
                                 out=out, lse=lse, ws=ws)
        else:
            lsh.lsh_attn_forward_timed(d_qk, d_v, d_R, w.n_buckets, w.chunk, w.causal, w.scale,
                                       out, lse, ws, events)

    for _ in range(Wm):
        fwd()
    torch.cuda.synchronize()
    st, dd = lsh.lsh_workspace_status(ws)
    if st != lsh.LSH_OK:
        raise RuntimeError(f"device check failed after warm-up: {lsh.lsh_status_string(st)} {dd}")

    # ---- device-resident timed region: K forward calls, stage events inside each call
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    for evs in events:          # create the events (torch creates them on first record)
        for e in evs:
            e.record(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for k in range(K):
        fwd(events[k])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / K
    ms_max = allmax(dist, ms)
    stage_names = ("hash", "sort", "attn", "combine")
    stage_ms = {n: statistics.mean(events[k][i].elapsed_time(events[k][i + 1]) for k in range(K))
                for i, n in enumerate(stage_names)}
    st, dd = lsh.lsh_workspace_status(ws)
    if st != lsh.LSH_OK:
        raise RuntimeError(f"device check failed: {lsh.lsh_status_string(st)} {dd}")

    # ---- end to end through host buffers: H2D inputs, forward, D2H outputs
    h_out = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        d_qk.copy_(h_qk, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_R.copy_(h_R, non_blocking=True)
        fwd()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allmax(dist, e0.elapsed_time(e1) / K)
    barrier(dist)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    tokens = w.tokens * world
    value = job_value(w.tokens, world, ms_max)
    peaks, peak_src = load_peaks()
    wk = work(w)
    # dominant kernel and its roofline
    dom = max(stage_ms, key=stage_ms.get)
    unit_c = COMPUTE_UNIT[w.dtype]
    peak_c = peaks["bf16_tflops"] if unit_c == "tensor" else FP32_ALU_TFLOPS

    def roof(name):
        return kernel_roof(w, name, stage_ms[name], wk[name], unit_c, peak_c, peaks, peak_src)

    F = sum(k["flops"] for k in wk.values())
    Bts = sum(k["bytes"] for k in wk.values())
    # the same compute peak as the per-kernel entries: tensor for bf16, fp32 lanes for f32
    t_roof = max(F / (peak_c * 1e12), Bts / (peaks["hbm_gbs"] * 1e9))

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(config_of(w), parallelism=f"replicas{world}",
                       l2=f"inputs larger than L2: qk+v {2 * w.tokens * w.d * ESIZE[w.dtype] / 2**20:.0f} MiB, "
                          f"per-round outputs {w.tokens * w.n_rounds * w.d * ESIZE[w.dtype] / 2**20:.0f} MiB "
                          f"> L2 126 MiB; no flush"),
        "roofline": roof(dom),
        "kernels": {n: roof(n) for n in stage_names},
        "path_roofline": {"flops": F, "bytes": Bts, "t_roof_ms": 1e3 * t_roof,
                          "frac": 1e3 * t_roof / ms_max, "peaks": peak_src},
        "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_qk.nbytes + h_v.nbytes + h_R.nbytes),
                "d2h_bytes_per_step": int(h_out.nbytes + h_lse.nbytes), "ms_per_step": e2e_ms},
        "clocks": clk,
        "gpu_launches": int(lib.lsh_attn_kernel_launches(w.B, w.H, w.L, w.d, w.n_buckets,
                                                         w.n_rounds, w.chunk, dt_code)) * K,
    }
    if not args.no_cpu_baseline and world == 1:
        threads = os.cpu_count() or 1
        keep = {}
        tok, times, used, desc = time_oracle(w, threads, steps=1, keep=keep)
        line["cpu_baseline"] = {"value": tok / times[0], "unit": "tokens/s", "cores": used,
                                "cpu_model": cpu_model(), "kind": "oracle", "sample": desc}
        line["near_ties"] = near_tie_report(lsh, dev, keep)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_backward(args, w):
    """The backward pass of workload w: K timed lsh_attn_backward calls on device-resident
    inputs (qk, v, R, the forward's out and lse, seeded g_out and g_lse), stage events
    inside each call, then the same calls end to end from pinned host buffers."""
    import torch
    import lsh_attention_04_b300 as lsh
    from lsh_attention_04_b300 import inputs as gen

    world, rank, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = lsh.load()
    dt_code = dt_code_of(lsh, w)
    tdt = torch_dtype_of(torch, w)

    qk, v, R = gen.make_inputs(w, seed=w.seed + 7919 * rank)
    rng = np.random.default_rng(w.seed + 5 + 7919 * rank)
    h_qk = torch.from_numpy(qk).to(tdt).pin_memory()
    h_v = torch.from_numpy(v).to(tdt).pin_memory()
    h_R = torch.from_numpy(R).to(tdt).pin_memory()
    h_g = torch.from_numpy(rng.standard_normal(qk.shape).astype(np.float32)).pin_memory()
    h_gl = torch.from_numpy(rng.standard_normal(qk.shape[:-1]).astype(np.float32)).pin_memory()
    d_qk, d_v, d_R, d_g, d_gl = (t.to(dev) for t in (h_qk, h_v, h_R, h_g, h_gl))
    out, lse = lsh.lsh_attn_forward(d_qk, d_v, d_R, w.n_buckets, w.chunk, w.causal, w.scale)
    h_out = out.cpu().pin_memory()
    h_lse = lse.cpu().pin_memory()
    dqk = torch.empty((w.B, w.H, w.L, w.d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dqk)
    n_ws = int(lib.lsh_attn_backward_workspace_bytes(w.B, w.H, w.L, w.d, w.n_buckets,
                                                     w.n_rounds, w.chunk, dt_code))
    ws = torch.empty(n_ws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    K, Wm = args.steps, args.warmup

    def bwd(events=None):
        if events is None:
            lsh.lsh_attn_backward(d_qk, d_v, d_R, w.n_buckets, w.chunk, w.causal, w.scale, out,
                                  lse, d_g, d_gl, dqk=dqk, dv=dv, ws=ws)
        else:
            lsh.lsh_attn_backward_timed(d_qk, d_v, d_R, w.n_buckets, w.chunk, w.causal,
                                        w.scale, out, lse, d_g, d_gl, dqk, dv, ws, events)

    for _ in range(Wm):
        bwd()
    torch.cuda.synchronize()
    st, dd = lsh.lsh_workspace_status(ws)
    if st != lsh.LSH_OK:
        raise RuntimeError(f"device check failed after warm-up: {lsh.lsh_status_string(st)} {dd}")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for evs in events:
        for e in evs:
            e.record(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for k in range(K):
        bwd(events[k])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_max = allmax(dist, t0.elapsed_time(t1) / K)
    stage_names = ("hash", "sort", "attn_bwd")
    stage_ms = {n: statistics.mean(events[k][i].elapsed_time(events[k][i + 1]) for k in range(K))
                for i, n in enumerate(stage_names)}
    st, dd = lsh.lsh_workspace_status(ws)
    if st != lsh.LSH_OK:
        raise RuntimeError(f"device check failed: {lsh.lsh_status_string(st)} {dd}")
    if not (torch.isfinite(dqk).all() and torch.isfinite(dv).all()):
        raise RuntimeError("non-finite gradients")

    # ---- end to end: H2D of every input, backward, D2H of both gradients
    h_dqk = torch.empty(dqk.shape, dtype=torch.float32).pin_memory()
    h_dv = torch.empty(dv.shape, dtype=torch.float32).pin_memory()
    srcs = (h_qk, h_v, h_R, h_out, h_lse, h_g, h_gl)
    dsts = (d_qk, d_v, d_R, out, lse, d_g, d_gl)

    def e2e_step():
        for d_, h_ in zip(dsts, srcs):
            d_.copy_(h_, non_blocking=True)
        bwd()
        h_dqk.copy_(dqk, non_blocking=True)
        h_dv.copy_(dv, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allmax(dist, e0.elapsed_time(e1) / K)
    barrier(dist)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    value = job_value(w.tokens, world, ms_max)
    peaks, peak_src = load_peaks()
    wk = work_backward(w)
    unit_c = COMPUTE_UNIT[w.dtype]
    peak_c = peaks["bf16_tflops"] if unit_c == "tensor" else FP32_ALU_TFLOPS
    kernels = {n: kernel_roof(w, n, stage_ms[n], wk[n], unit_c, peak_c, peaks, peak_src)
               for n in stage_names}
    dom = max(stage_ms, key=stage_ms.get)
    F = sum(k["flops"] for k in wk.values())
    Bts = sum(k["bytes"] for k in wk.values())
    t_roof = max(F / (peak_c * 1e12), Bts / (peaks["hbm_gbs"] * 1e9))
    # kernels per call: the forward's hash and sort launches plus the backward kernel
    # (the forward's count less its attention and combination, plus one), and for bf16
    # the prepass of the tensor-core kernel (g_out in bf16, g_out . out)
    launches = int(lib.lsh_attn_kernel_launches(w.B, w.H, w.L, w.d, w.n_buckets, w.n_rounds,
                                                w.chunk, dt_code)) - 1 + (w.dtype == "bf16")
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "pass": "backward",
        "config": dict(config_of(w), parallelism=f"replicas{world}",
                       l2="inputs larger than L2: qk, v, out, g_out, dqk, dv "
                          f"{w.tokens * w.d * (2 * ESIZE[w.dtype] + 16) / 2**20:.0f} MiB "
                          "> L2 126 MiB; no flush"),
        "roofline": kernels[dom],
        "kernels": kernels,
        "path_roofline": {"flops": F, "bytes": Bts, "t_roof_ms": 1e3 * t_roof,
                          "frac": 1e3 * t_roof / ms_max, "peaks": peak_src},
        "e2e": {"value": w.tokens * world / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(sum(t.nbytes for t in srcs)),
                "d2h_bytes_per_step": int(h_dqk.nbytes + h_dv.nbytes), "ms_per_step": e2e_ms},
        "clocks": clk,
        "gpu_launches": launches * K,
    }
    if not args.no_cpu_baseline and world == 1:
        tok, times, used, desc = time_oracle_backward(w, steps=1)
        line["cpu_baseline"] = {"value": tok / times[0], "unit": "tokens/s", "cores": used,
                                "cpu_model": cpu_model(), "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def work_knn(w, k):
    """Algorithmic FLOPs and bytes of one lsh_knn call: the hash and sort, then per chunk
    the c x 2c similarity tile (4 c d flops per token and round) over window rows
    gathered once per chunk (own and previous chunk: 2 d e bytes per token and round),
    per-round lists written and read back, and the final lists written."""
    N, R, d, c = w.tokens, w.n_rounds, w.d, w.chunk
    e = ESIZE[w.dtype]
    base = work(w)
    return {"hash": base["hash"], "sort": base["sort"],
            "knn": dict(flops=4 * N * R * c * d,
                        bytes=2 * N * R * d * e + N * R * 12 + 2 * N * R * k * 8 + N * k * 8)}


def knn_roofline(F, Bts, ms, peaks, peak_src):
    """Roofline of a whole lsh_knn call: the slower of its FLOPs at the bf16 burst peak and
    its bytes at the copy bandwidth decides the bound; achieved is that quantity's rate."""
    t_f, t_b = F / (peaks["bf16_tflops"] * 1e12), Bts / (peaks["hbm_gbs"] * 1e9)
    if t_f > t_b:
        bound, achieved, peak, unit = "tensor", F / (ms / 1e3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        bound, achieved, peak, unit = "hbm", Bts / (ms / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s"
    return {"bound": bound, "kernel": "whole call (hash, sort, similarity tiles, selection, merge)",
            "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "t_roof_ms": 1e3 * max(t_f, t_b), "algorithmic_flops": F, "algorithmic_bytes": Bts,
            "peaks": peak_src, "traffic": None}


def run_knn(args, w):
    """LSH approximate k-nearest-neighbour search (lsh_knn) at workload w's shape: K timed
    calls on device-resident qk and R, recall@k of 512 sampled queries against an
    exhaustive cosine search of the same head (numpy on the host), end-to-end calls from
    pinned host buffers, and the oracle's search on a bounded sample as CPU baseline."""
    import torch
    import lsh_attention_04_b300 as lsh
    from lsh_attention_04_b300 import inputs as gen

    world, rank, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = lsh.load()
    dt_code = dt_code_of(lsh, w)
    tdt = torch_dtype_of(torch, w)
    k = KNN_K
    qk, _, R = gen.make_inputs(w, seed=w.seed + 7919 * rank)
    h_qk = torch.from_numpy(qk).to(tdt).pin_memory()
    h_R = torch.from_numpy(R).to(tdt).pin_memory()
    d_qk, d_R = h_qk.to(dev), h_R.to(dev)
    nn_idx = torch.empty((w.B, w.H, w.L, k), dtype=torch.int32, device=dev)
    nn_sim = torch.empty((w.B, w.H, w.L, k), dtype=torch.float32, device=dev)
    n_ws = int(lib.lsh_knn_workspace_bytes(w.B, w.H, w.L, w.d, w.n_buckets, w.n_rounds, w.chunk,
                                           k, dt_code))
    ws = torch.empty(n_ws, dtype=torch.uint8, device=dev)
    K, Wm = args.steps, args.warmup

    def call():
        lsh.lsh_knn(d_qk, d_R, w.n_buckets, w.chunk, k, nn_idx, nn_sim, ws)

    for _ in range(Wm):
        call()
    torch.cuda.synchronize()
    st, dd = lsh.lsh_workspace_status(ws)
    if st != lsh.LSH_OK:
        raise RuntimeError(f"device check failed after warm-up: {lsh.lsh_status_string(st)} {dd}")
    stream = torch.cuda.current_stream(dev)
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for _ in range(K):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_max = allmax(dist, t0.elapsed_time(t1) / K)

    # recall@k of sampled queries against an exhaustive search of the same head
    rng = np.random.default_rng(w.seed)
    heads = qk.reshape(-1, w.L, w.d).astype(np.float64)
    got = nn_idx.cpu().numpy().reshape(-1, w.L, k)
    hits = []
    for h in rng.choice(len(heads), size=min(2, len(heads)), replace=False):
        x = heads[h]
        nrm = np.linalg.norm(x, axis=1)
        xn = x / np.where(nrm > 0, nrm, 1.0)[:, None]
        for t in rng.choice(w.L, size=256, replace=False):
            sim = xn @ xn[t]
            sim[t] = -np.inf
            top = np.lexsort((np.arange(w.L), -sim))[:k]
            hits.append(len(set(top.tolist()) & set(got[h, t].tolist())) / k)

    # end to end: H2D of qk and R, the search, D2H of both lists
    h_idx = torch.empty(nn_idx.shape, dtype=torch.int32).pin_memory()
    h_sim = torch.empty(nn_sim.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        d_qk.copy_(h_qk, non_blocking=True)
        d_R.copy_(h_R, non_blocking=True)
        call()
        h_idx.copy_(nn_idx, non_blocking=True)
        h_sim.copy_(nn_sim, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allmax(dist, e0.elapsed_time(e1) / K)
    barrier(dist)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    wk = work_knn(w, k)
    F = sum(x["flops"] for x in wk.values())
    Bts = sum(x["bytes"] for x in wk.values())
    # the similarity tiles run on the tensor cores for 16-bit inputs, the fp32 lanes else
    peak_c = peaks["bf16_tflops"] if COMPUTE_UNIT[w.dtype] == "tensor" else FP32_ALU_TFLOPS
    t_roof = max(F / (peak_c * 1e12), Bts / (peaks["hbm_gbs"] * 1e9))
    line = {
        "metric": METRIC_KNN, "value": job_value(w.tokens, world, ms_max), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic", "pass": "knn",
        "config": dict(config_of(w), k=k, parallelism=f"replicas{world}",
                       l2="inputs and per-round lists larger than L2; no flush"),
        "recall": {"at_k": k, "value": float(np.mean(hits)), "queries": len(hits),
                   "against": "exhaustive cosine search of the same head (numpy, host)"},
        "roofline": knn_roofline(F, Bts, ms_max, peaks, peak_src),
        "e2e": {"value": w.tokens * world / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_qk.nbytes + h_R.nbytes),
                "d2h_bytes_per_step": int(h_idx.nbytes + h_sim.nbytes), "ms_per_step": e2e_ms},
        "clocks": clk,
        # the forward's hash and sort launches, then the round and merge kernels in place
        # of the attention and combination (the same count)
        "gpu_launches": int(lib.lsh_attn_kernel_launches(w.B, w.H, w.L, w.d, w.n_buckets,
                                                         w.n_rounds, w.chunk, dt_code)) * K,
    }
    if not args.no_cpu_baseline and world == 1:
        tok, tsec, desc = time_oracle_knn(w, k)
        line["cpu_baseline"] = {"value": tok / tsec, "unit": "tokens/s", "cores": 1,
                                "cpu_model": cpu_model(), "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def time_oracle_knn(w, k, max_tokens=8192):
    """The oracle's search on a bounded sample: head 0, the first max_tokens tokens, all
    rounds (its hash and sort included), one thread."""
    import oracle
    sub, qk, v, R, desc = oracle_sample(w, max_tokens)
    oracle.build()
    x = qk.reshape(-1, sub.L, sub.d)[0].astype(np.float64)
    t0 = time.perf_counter()
    b = np.empty((sub.n_rounds, sub.L), np.int32)
    p, iv = np.empty_like(b), np.empty_like(b)
    for r in range(sub.n_rounds):
        b[r], _ = oracle.hash(x, R[r], sub.n_buckets)
        p[r], iv[r], _ = oracle.sort(b[r], sub.n_buckets)
    oracle.knn(x, b, p, iv, sub.chunk, k)
    return sub.tokens, time.perf_counter() - t0, desc + f"; k-NN search, k = {k}"


def attn_workload_of(bw):
    """The attention step of block workload bw as an attention workload."""
    from lsh_attention_04_b300 import inputs as gen
    return gen.Workload(bw.name + "_attention", bw.B, bw.heads, bw.L, bw.d, "bf16", bw.n_buckets,
                        bw.n_rounds, bw.chunk, bw.causal, 0, bw.seed)


def block_gemms(bw):
    """The block forward's matrix products: (name, M, N, K, launches, epilogue)."""
    M, dm, dff, c = bw.B * bw.L, bw.d_model, bw.d_ff, bw.ff_chunk
    n_chunks = -(-M // c)
    return [("qk_projection", M, dm, dm, 1, "bf16 heads"),
            ("v_projection", M, dm, dm, 1, "bf16 heads"),
            ("output_projection", M, dm, dm, 1, "fp32 + residual"),
            ("ffn_in", min(c, M), dff, dm, n_chunks, "bias + ReLU, bf16"),
            ("ffn_out", min(c, M), dm, dff, n_chunks, "bias, fp32 + residual")]


def revblock_launches(lib, bw):
    """Kernels one lsh_revblock_forward call launches: the stream's bf16 copy, two
    projections, the attention forward's launches, the status merge, the head merge, the
    output projection, the bf16 copy of y1, and two products per feed-forward chunk."""
    aw = attn_workload_of(bw)
    n_chunks = -(-(bw.B * bw.L) // bw.ff_chunk)
    attn = int(lib.lsh_attn_kernel_launches(aw.B, aw.H, aw.L, aw.d, aw.n_buckets, aw.n_rounds,
                                            aw.chunk, 1))
    return 1 + 2 + attn + 1 + 1 + 1 + 1 + 2 * n_chunks


def run_revblock(args, bw):
    """One reversible block forward (lsh_revblock_forward) at block workload bw: K timed
    calls on device-resident x1, x2 and weights; every matrix product shape and the
    attention forward then timed alone on the same device for the stage breakdown and the
    GEMM roofline; end-to-end calls from pinned host buffers; the oracle's block on a
    bounded sample as CPU baseline."""
    import torch
    import lsh_attention_04_b300 as lsh
    from lsh_attention_04_b300 import inputs as gen

    world, rank, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = lsh.load()
    inp = gen.make_block_inputs(bw, seed=bw.seed + 7919 * rank)
    d = {}
    for k, a in inp.items():
        t = torch.from_numpy(a)
        d[k] = t.to(dev).to(torch.bfloat16) if k in ("Wqk", "Wv", "Wo", "W1", "W2", "R") else t.to(dev)
    h_x1, h_x2 = torch.from_numpy(inp["x1"]).pin_memory(), torch.from_numpy(inp["x2"]).pin_memory()
    y1, y2 = torch.empty_like(d["x1"]), torch.empty_like(d["x2"])
    ws = lsh.revblock_workspace(bw.B, bw.L, bw.d_model, bw.heads, bw.d_ff, bw.n_buckets,
                                bw.n_rounds, bw.chunk, bw.ff_chunk, dev)
    K, Wm = args.steps, args.warmup

    def call():
        lsh.lsh_revblock_forward(d["x1"], d["x2"], d, bw.heads, bw.n_buckets, bw.chunk,
                                 bw.causal, bw.scale, bw.ff_chunk, y1, y2, ws)

    for _ in range(Wm):
        call()
    torch.cuda.synchronize()
    st, dd = lsh.lsh_workspace_status(ws)
    if st != lsh.LSH_OK:
        raise RuntimeError(f"device check failed after warm-up: {lsh.lsh_status_string(st)} {dd}")
    stream = torch.cuda.current_stream(dev)
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for _ in range(K):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_max = allmax(dist, t0.elapsed_time(t1) / K)
    st, dd = lsh.lsh_workspace_status(ws)
    if st != lsh.LSH_OK:
        raise RuntimeError(f"device check failed: {lsh.lsh_status_string(st)} {dd}")

    # stage breakdown: every product shape and the attention forward, each timed alone
    def timed(fn, reps):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    M, dm = bw.B * bw.L, bw.d_model
    a16 = torch.empty((M, max(dm, bw.d_ff)), dtype=torch.bfloat16, device=dev)
    a16.normal_()
    o32 = torch.empty((M, dm), dtype=torch.float32, device=dev)
    o16 = torch.empty((M, max(dm, bw.d_ff)), dtype=torch.bfloat16, device=dev)
    gws = torch.empty(256, dtype=torch.uint8, device=dev)
    reps = max(5, min(50, K))
    stages, g_flops, g_ms = {}, 0.0, 0.0
    for name, m, n, k, launches, epi in block_gemms(bw):
        A = a16[:m, :k].contiguous() if k != a16.shape[1] else a16[:m]
        Wt = {"qk_projection": d["Wqk"], "v_projection": d["Wv"], "output_projection": d["Wo"],
              "ffn_in": d["W1"], "ffn_out": d["W2"]}[name]
        kw = {}
        if epi.startswith("bf16 heads"):
            kw = dict(f32=False, bf16=True, split=(bw.L, bw.d),
                      out_bf16=o16[:m].view(-1)[: m * n].view(m // bw.L, n // bw.d, bw.L, bw.d))
        elif epi.startswith("bias + ReLU"):
            kw = dict(bias=d["b1"], relu=True, f32=False, bf16=True,
                      out_bf16=o16[:m, :n].contiguous() if n != o16.shape[1] else o16[:m])
        elif epi.startswith("bias, fp32"):
            kw = dict(bias=d["b2"], res=o32[:m], out_f32=o32[:m])
        else:
            kw = dict(res=o32[:m], out_f32=o32[:m])
        ms = timed(lambda: lsh.lsh_gemm_bf16(A, Wt, ws=gws, **kw), reps)
        fl = 2.0 * m * n * k
        stages[name] = {"M": m, "N": n, "K": k, "launches": launches, "ms_per_launch": ms,
                        "tflops": fl / (ms / 1e3) / 1e12, "epilogue": epi}
        g_flops += fl * launches
        g_ms += ms * launches
    del a16, o16, o32
    aw = attn_workload_of(bw)
    qk16 = torch.empty((aw.B, aw.H, aw.L, aw.d), dtype=torch.bfloat16, device=dev).normal_()
    v16 = torch.empty_like(qk16).normal_()
    aws = torch.empty(int(lib.lsh_attn_workspace_bytes(aw.B, aw.H, aw.L, aw.d, aw.n_buckets,
                                                        aw.n_rounds, aw.chunk, 1)),
                      dtype=torch.uint8, device=dev)
    aout = torch.empty((aw.B, aw.H, aw.L, aw.d), dtype=torch.float32, device=dev)
    alse = torch.empty((aw.B, aw.H, aw.L), dtype=torch.float32, device=dev)
    attn_ms = timed(lambda: lsh.lsh_attn_forward(qk16, v16, d["R"], aw.n_buckets, aw.chunk,
                                                 aw.causal, aw.scale, aout, alse, aws), reps)
    del qk16, v16, aws, aout, alse

    # end to end: H2D of x1 and x2, the block, D2H of y1 and y2
    h_y1 = torch.empty(y1.shape, dtype=torch.float32).pin_memory()
    h_y2 = torch.empty(y2.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        d["x1"].copy_(h_x1, non_blocking=True)
        d["x2"].copy_(h_x2, non_blocking=True)
        call()
        h_y1.copy_(y1, non_blocking=True)
        h_y2.copy_(y2, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(K, 20))
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allmax(dist, e0.elapsed_time(e1) / n_e2e)
    barrier(dist)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    peak = peaks["bf16_tflops"]
    achieved = g_flops / (g_ms / 1e3) / 1e12
    tokens = bw.B * bw.L
    line = {
        "metric": METRIC_REV, "value": job_value(tokens, world, ms_max), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "pass": "revblock",
        "config": {"workload": bw.name, "B": bw.B, "L": bw.L, "d_model": bw.d_model,
                   "heads": bw.heads, "d": bw.d, "d_ff": bw.d_ff, "n_buckets": bw.n_buckets,
                   "n_rounds": bw.n_rounds, "chunk": bw.chunk, "causal": bw.causal,
                   "ff_chunk": bw.ff_chunk, "stream": "fp32", "products": "bf16 in, fp32 acc",
                   "parallelism": f"replicas{world}",
                   "l2": "inputs (256 MB per stream half) larger than L2; no flush"},
        "roofline": {"bound": "tensor", "kernel": "gemm_tc_kernel (every matrix product of "
                     "the block, each shape timed alone)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peaks": f"{peak_src} bf16 burst",
                     "algorithmic_flops": g_flops, "traffic": None},
        "stages": {"gemm": stages, "gemm_ms_total": g_ms, "attention_ms": attn_ms,
                   "sum_of_stages_ms": g_ms + attn_ms},
        "e2e": {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_x1.nbytes + h_x2.nbytes),
                "d2h_bytes_per_step": int(h_y1.nbytes + h_y2.nbytes), "ms_per_step": e2e_ms},
        "clocks": clk,
        "gpu_launches": revblock_launches(lib, bw) * K,
    }
    if not args.no_cpu_baseline and world == 1:
        tok, tsec, desc = time_oracle_revblock(bw)
        line["cpu_baseline"] = {"value": tok / tsec, "unit": "tokens/s", "cores": 1,
                                "cpu_model": cpu_model(), "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def time_oracle_revblock(bw, max_tokens=4096):
    """The oracle's reversible block on a bounded sample (see _oracle_revblock_sample), in
    a child process whose BLAS runs one thread: returns (positions, seconds, description)."""
    import dataclasses
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"print(json.dumps(bench._oracle_revblock_sample({json.dumps(dataclasses.asdict(bw))!r}, "
            f"{int(max_tokens)})))")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True)
    tok, t, desc = json.loads(out.stdout.strip().splitlines()[-1])
    return tok, t, desc


def _oracle_revblock_sample(bw_json, max_tokens):
    """The first max_tokens positions of batch row 0 of block workload bw with its widths,
    heads, buckets and rounds, through the oracle's block forward on one thread."""
    import dataclasses
    import oracle
    from oracle import reversible as orev
    from lsh_attention_04_b300 import inputs as gen
    bw = gen.BlockWorkload(**json.loads(bw_json))
    Ls = min(bw.L, max(2 * bw.chunk, (max_tokens // (2 * bw.chunk)) * (2 * bw.chunk)))
    sub = dataclasses.replace(bw, B=1, L=Ls, ff_chunk=min(bw.ff_chunk, Ls))
    inp = gen.make_block_inputs(sub, seed=bw.seed)
    p = {k: inp[k].astype(np.float64) for k in ("Wqk", "Wv", "Wo", "W1", "b1", "W2", "b2", "R")}
    p.update(heads=sub.heads, n_buckets=sub.n_buckets, chunk=sub.chunk, causal=sub.causal,
             scale=sub.scale, ff_chunk=sub.ff_chunk, threads=1)
    oracle.build()
    t0 = time.perf_counter()
    orev.forward(inp["x1"].astype(np.float64), inp["x2"].astype(np.float64), p)
    t = time.perf_counter() - t0
    desc = (f"batch row 0 of {bw.name}: first {Ls} positions, d_model {bw.d_model}, "
            f"{bw.heads} heads, d_ff {bw.d_ff}, {bw.n_rounds} rounds, {bw.n_buckets} buckets "
            "(fp64, one thread)")
    return Ls, t, desc


def main():
    from lsh_attention_04_b300 import inputs as gen
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=gen.HEADLINE, choices=sorted(gen.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="pass_", choices=("forward", "backward", "knn", "revblock"),
                    default="forward",
                    help="time the forward pass (default), the backward pass, the LSH "
                         "k-nearest-neighbour search (k = 16), or one reversible block "
                         "around the attention (forward)")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the workload with this many heads instead (small ncu captures); "
                         "the printed line then names the reduced workload")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    w = gen.WORKLOADS[args.workload]
    if args.heads > 0 and args.heads != w.H:
        w = w.replace(H=args.heads, name=w.name.replace(f"_H{w.H}_", f"_H{args.heads}_"))
    if args.pass_ == "revblock":
        return run_reference_revblock(args, gen.BLOCK_LONG) if args.impl == "reference" else \
            run_revblock(args, gen.BLOCK_LONG)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.pass_ == "backward":
        return run_backward(args, w)
    if args.pass_ == "knn":
        return run_knn(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
