"""Benchmark of the fused attention forward on GB300.

One step = one pass of the whole hot path on synthetic inputs already resident in device memory:
  * prefill: B=8, Hq=8, Hkv=2, S=8192, D=128, bf16, causal (long-context throughput workload);
  * decode:  B=32, Hq=8, Hkv=2, D=128, bf16 cache, per-sequence lengths uniform in [256, 4096].
Before each timed kernel region the L2 cache is flushed outside the events: a 512 MiB buffer is
written, then another 512 MiB buffer is read, so the timed kernel starts from a clean L2 (a bare
memset would leave L2 full of dirty lines whose write-back the next kernel would pay for).
Decode is reported twice: one call after a flush (launch latency included), and a CUDA graph of
16 back-to-back calls over 4 rotating KV caches (together over 4x the L2), launch amortised.

Printed (rank 0, one JSON line): ``value`` = prefill TFLOP/s (algorithmic causal flops over the
measured prefill time), the decode GB/s (algorithmic bytes: every valid K/V row once, q and o)
under ``decode``, the roofline fractions against the measured peaks, an end-to-end figure through
the public API with host buffers (copies inside the timed region), SM clocks sampled during the
timed region, and the fp64 CPU oracle timed on a bounded sample of the same workload.

``--impl reference`` times that oracle alone (the only reference that exists for this method) on
the host cores, on the same workload and metric.

Multi-GPU: run under torchrun; every rank runs the same workload independently (replicas, weak
scaling); the slowest rank's time is used and ``value`` is the sum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

PREFILL = workloads.CONFIGS["c5b"]
DECODE = workloads.CONFIGS["c4b"]
E2E_CHUNKS = 4  # batch slices of the end-to-end prefill (upload / compute / download overlap)
METRIC = "prefill attention TFLOP/s and decode KV-read GB/s, % of GB300 roofline"
FLUSH_BYTES = 512 << 20
# Nominal GB300 figures, reported beside the measured peaks: dense bf16 tensor throughput and
# HBM3e bandwidth ("about 8 TB/s").
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0
DECODE_SETS = 4
DECODE_CALLS = 16


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the extra timings (the other configured workloads; cache chunk, "
                        "padded varlen, fused-QKV and head-dim-64 prefill, decode with RoPE)")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle sample")
    p.add_argument("--only", default="all", choices=["all", "prefill", "decode"],
                   help="run one half of the step (profiling); the JSON line is for 'all' only")
    p.add_argument("--prefill-batch", type=int, default=None)
    p.add_argument("--prefill-seq", type=int, default=None)
    p.add_argument("--decode-batch", type=int, default=None)
    p.add_argument("--decode-len", type=int, default=None,
                   help="every sequence this long (cache max_len too) instead of U[256, 4096]")
    args = p.parse_args()
    global PREFILL, DECODE
    if args.prefill_batch or args.prefill_seq:
        PREFILL = workloads.PrefillConfig("custom", args.prefill_batch or PREFILL.B, PREFILL.Hq,
                                          PREFILL.Hkv, args.prefill_seq or PREFILL.S, PREFILL.D,
                                          "bf16")
    if args.decode_batch or args.decode_len:
        DECODE = workloads.DecodeConfig("custom", args.decode_batch or DECODE.B, DECODE.Hq,
                                        DECODE.Hkv, DECODE.D, args.decode_len or DECODE.max_len,
                                        "full" if args.decode_len else "uniform")
    return args


def recorded_traffic():
    """DRAM traffic per launch recorded from ncu in profiles/, valid only while the kernel source
    it was measured on is unchanged (sha256 prefix of the kernel file + ptx.cuh)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic_prefill_b8s8192_decode_b32.md")
    csrc = os.path.join(ROOT, "causal_gqa_attention_gb300", "csrc")
    out = {"prefill_tc_kernel": None, "decode_stream_kernel": None}
    if not os.path.exists(path):
        return out
    text = open(path).read()

    def sha(*names):
        h = hashlib.sha256()
        for n in names:
            h.update(open(os.path.join(csrc, n), "rb").read())
        return h.hexdigest()[:16]

    cur = {"prefill_tc_kernel": sha("prefill_tc.cu", "ptx.cuh"),
           "decode_stream_kernel": sha("decode.cu", "ptx.cuh")}
    tag = {"prefill_tc_kernel": "prefill_tc.cu+ptx.cuh", "decode_stream_kernel": "decode.cu+ptx.cuh"}
    for kname in out:
        rec_sha, rec_bytes = None, None
        for line in text.splitlines():
            if line.startswith(f"source-sha {tag[kname]}:"):
                rec_sha = line.split(":", 1)[1].strip()
            if line.startswith(f"traffic-bytes {kname}:"):
                rec_bytes = int(line.split(":", 1)[1].strip())
        if rec_sha == cur[kname] and rec_bytes:
            out[kname] = rec_bytes
    return out


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "200"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- distributed


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, local_ms: float, world: int, dev):
    """Weak scaling: every rank processes units_per_rank in local_ms. Returns the slowest rank's
    time (ms), the per-GPU rate at that time and the whole-job rate (all ranks' units over the
    slowest time), rates in units per second."""
    ms = max_over_ranks(local_ms, world, dev)
    per_gpu = units_per_rank / (max(ms, 1e-6) * 1e-3)
    return ms, per_gpu, per_gpu * world


# --------------------------------------------------------------------------- oracle sample


def oracle_sample(seconds: float):
    """Time the fp64 oracle on a bounded sample of the bench workload. Returns dict with the
    prefill TFLOP/s and decode GB/s the oracle reaches on its sample, cores and a description."""
    import oracle

    lib = oracle.load()
    cores = oracle.num_threads(lib)
    cfg = PREFILL
    q, k, v = workloads.config_prefill_inputs(cfg)
    # rows spread over the causal range, (b, h) cycling; work per row = (i + 1) keys
    rng = np.random.default_rng(0)
    n_rows = 256
    rows = []
    t_pref = 0.0
    flops = 0
    done = 0
    while True:
        b = rng.integers(0, cfg.B, n_rows)
        h = rng.integers(0, cfg.Hq, n_rows)
        i = rng.integers(0, cfg.S, n_rows)
        rows = ((b * cfg.Hq + h) * cfg.S + i).astype(np.int64)
        t0 = time.perf_counter()
        oracle.prefill(q, k, v, True, cfg.scale, rows=rows, lib=lib)
        t_pref += time.perf_counter() - t0
        flops += int(np.sum(4 * cfg.D * (i + 1)))
        done += n_rows
        if t_pref > 0.7 * seconds:
            break
    dq, dkc, dvc, sl = workloads.config_decode_inputs(DECODE)
    t_dec = 0.0
    reps = 0
    while True:
        t0 = time.perf_counter()
        oracle.decode(dq, dkc, dvc, sl, DECODE.scale, lib=lib)
        t_dec += time.perf_counter() - t0
        reps += 1
        if t_dec > 0.3 * seconds:
            break
    dec_bytes = workloads.decode_bytes(sl.tolist(), DECODE.Hq, DECODE.Hkv, DECODE.D)
    return {
        "prefill_tflops": flops / t_pref / 1e12,
        "decode_gbs": dec_bytes * reps / t_dec / 1e9,
        "cores": cores,
        "sample": (f"prefill: {done} query rows of the B8 S8192 causal workload drawn uniformly "
                   f"over (b, h, i), {t_pref:.1f} s; decode: {reps} full B32 step(s), "
                   f"{t_dec:.1f} s; fp64, OpenMP over rows"),
        "seconds": t_pref + t_dec,
    }


def cpu_model() -> str:
    """The host CPU's model name, as the OS reports it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform

    return platform.processor() or platform.machine()


def oracle_single_core():
    """The fp64 oracle on one core for the three small configured prefill workloads (every
    causal setting each names), full size: seconds and GFLOP/s."""
    import oracle

    lib = oracle.load()
    out = {}
    for name in ("c1", "c2", "c3"):
        cfg = workloads.CONFIGS[name]
        q, k, v = workloads.config_prefill_inputs(cfg)
        for causal in cfg.causal:
            t0 = time.perf_counter()
            oracle.prefill(q, k, v, causal, cfg.scale, nthreads=1, lib=lib)
            dt = time.perf_counter() - t0
            fl = workloads.prefill_flops(cfg.B, cfg.Hq, cfg.S, cfg.D, causal)
            out[f"{name}_{'causal' if causal else 'full'}"] = {"s": dt, "gflops": fl / dt / 1e9}
    return out


def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    steps, warmup = args.steps, args.warmup
    per = max(1.0, 120.0 / max(1, steps + warmup))  # whole run within a few minutes
    per = min(per, 10.0)
    for _ in range(warmup):
        oracle_sample(min(per, 2.0))
    vals, dvals, cores, sample = [], [], None, None
    t0 = time.perf_counter()
    for _ in range(steps):
        r = oracle_sample(per)
        vals.append(r["prefill_tflops"])
        dvals.append(r["decode_gbs"])
        cores, sample = r["cores"], r["sample"]
    wall = time.perf_counter() - t0
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warmup,
        "ms_per_step": wall / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(),
        "decode": {"value": statistics.median(dvals), "unit": "GB/s"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def config_block():
    return {
        "workload": ("prefill B8 S8192 Hq8 Hkv2 D128 bf16 causal + decode B32 Hq8 Hkv2 D128 "
                     "bf16 cache, lengths U[256,4096] (seed 0)"),
        "prefill": {"B": PREFILL.B, "S": PREFILL.S, "Hq": PREFILL.Hq, "Hkv": PREFILL.Hkv,
                    "D": PREFILL.D, "causal": True},
        "decode": {"B": DECODE.B, "Hq": DECODE.Hq, "Hkv": DECODE.Hkv, "D": DECODE.D,
                   "max_len": DECODE.max_len, "lengths": "uniform [256, 4096]"},
        "l2": ("flushed before every timed kernel region (512 MiB written, then another "
               "512 MiB read, so L2 holds no dirty lines)"),
        "parallelism": "replicas",
    }


# --------------------------------------------------------------------------- extra paths


def _time(fn, flush, stream, reps):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def time_extras(cga, dev, stream, flush, steps):
    """Timings of the wider paths on representative shapes (one call each, clean L2)."""
    out = {}
    # chunked prefill: 8 sequences, 512 new tokens each against caches of 4096..8192 tokens
    B, Hq, Hkv, D, Sq, max_len = 8, 8, 2, 128, 512, 8192
    g = torch.Generator().manual_seed(0)
    lens = torch.randint(4096, max_len + 1, (B,), generator=g, dtype=torch.int32)
    q = torch.randn((B, Hq, Sq, D), generator=g).to(torch.bfloat16).to(dev)
    kc = torch.randn((B, Hkv, max_len, D), generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn((B, Hkv, max_len, D), generator=g).to(torch.bfloat16).to(dev)
    dl = lens.to(dev)
    o = torch.empty_like(q)
    ms = _time(lambda: cga.chunk(q, kc, vc, dl, out=o), flush, stream, max(3, steps // 2))
    pairs = sum(int(L) * Sq - Sq * (Sq - 1) // 2 for L in lens.tolist())
    fl = 4 * Hq * D * pairs
    out["chunk_b8_sq512_kv4096to8192"] = {"ms": ms, "value": fl / (ms * 1e-3) / 1e12,
                                          "unit": "TFLOP/s", "flops": fl}
    del q, kc, vc, o
    # padded variable-length prefill: 8 sequences of 1024..8192 tokens padded to 8192
    S = 8192
    lens = torch.randint(1024, S + 1, (B,), generator=g, dtype=torch.int32)
    q, k, v = [t.to(dev) for t in workloads.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=3)]
    dl = lens.to(dev)
    o = torch.empty_like(q)
    ms = _time(lambda: cga.prefill_varlen(q, k, v, dl, out=o), flush, stream, max(3, steps // 2))
    fl = sum(workloads.prefill_flops(1, Hq, int(L), D, True) for L in lens.tolist())
    out["varlen_b8_s1024to8192_padded8192"] = {"ms": ms, "value": fl / (ms * 1e-3) / 1e12,
                                               "unit": "TFLOP/s", "flops": fl}
    del q, k, v, o
    # prefill read in place from a fused QKV projection output [B, S, Hq + 2 Hkv, D], O written
    # as [B, S, Hq, D]; and head dim 64 (both B8 S8192 Hq8 Hkv2 causal)
    S = 8192
    fl = workloads.prefill_flops(B, Hq, S, D, True)
    x = torch.randn((B, S, Hq + 2 * Hkv, D), generator=g).to(torch.bfloat16).to(dev)
    qv, kv, vv = (x[:, :, :Hq].transpose(1, 2), x[:, :, Hq:Hq + Hkv].transpose(1, 2),
                  x[:, :, Hq + Hkv:].transpose(1, 2))
    ov = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device=dev).transpose(1, 2)
    ms = _time(lambda: cga.prefill(qv, kv, vv, causal=True, out=ov), flush, stream,
               max(3, steps // 2))
    out["prefill_fused_qkv_b8_s8192"] = {"ms": ms, "value": fl / (ms * 1e-3) / 1e12,
                                         "unit": "TFLOP/s", "flops": fl}
    del x, qv, kv, vv, ov
    q, k, v = [t.to(dev) for t in workloads.prefill_inputs(B, Hq, Hkv, S, 64, "bf16", seed=4)]
    o = torch.empty_like(q)
    fl = workloads.prefill_flops(B, Hq, S, 64, True)
    ms = _time(lambda: cga.prefill(q, k, v, causal=True, out=o), flush, stream, max(3, steps // 2))
    out["prefill_d64_b8_s8192"] = {"ms": ms, "value": fl / (ms * 1e-3) / 1e12,
                                   "unit": "TFLOP/s", "flops": fl}
    del q, k, v, o
    # decode step with RoPE of the new token and its cache store (32 sequences of 256..4096),
    # beside the plain decode of the same caches
    cfg = workloads.CONFIGS["c4b"]
    q, kc, vc, sl = [t.to(dev) for t in workloads.config_decode_inputs(cfg)]
    Bd, Hkv, D = cfg.B, cfg.Hkv, cfg.D
    k_new = torch.randn((Bd, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
    v_new = torch.randn((Bd, Hkv, D), generator=g).to(torch.bfloat16).to(dev)
    inv = 10000.0 ** (-torch.arange(D // 2, dtype=torch.float64) * 2 / D)
    ang = torch.arange(cfg.max_len, dtype=torch.float64)[:, None] * inv[None, :]
    cos_t, sin_t = ang.cos().float().to(dev), ang.sin().float().to(dev)
    o = torch.empty_like(q)
    reps = max(3, steps // 2)
    ms_rope = _time(lambda: cga.decode_rope(q, k_new, v_new, cos_t, sin_t, kc, vc, sl, out=o),
                    flush, stream, reps)
    ms_plain = _time(lambda: cga.decode(q, kc, vc, sl, out=o), flush, stream, reps)
    lens = sl.cpu().tolist()
    by = (workloads.decode_bytes(lens, cfg.Hq, Hkv, D) + 4 * Bd * Hkv * D * 2
          + 2 * Bd * (D // 2) * 4)  # + k_new/v_new read and stored, + cos/sin rows
    out["decode_rope_b32_l256to4096"] = {"ms": ms_rope, "value": by / (ms_rope * 1e-3) / 1e9,
                                         "unit": "GB/s", "bytes": by,
                                         "plain_decode_ms": ms_plain}
    return out


def time_configs(cga, dev, stream, flush, pk, steps):
    """Every configured workload besides the headline pair, timed with the same L2 flush and CUDA
    events (median of the reps; one call each unless stated). Prefill: TFLOP/s and the fraction
    of the measured bf16 peak (the fp32 parity workloads run on CUDA cores, no roofline claim).
    Decode B1 L4096: one call, and back to back in a CUDA graph over enough caches (40 x 4.2 MB)
    that consecutive calls never find their cache in L2."""
    out = {}
    reps = max(10, steps)
    for name in ("c1", "c2", "c3", "c5a"):
        cfg = workloads.CONFIGS[name]
        q, k, v = [t.to(dev) for t in workloads.config_prefill_inputs(cfg)]
        o = torch.empty(q.shape, dtype=q.dtype, device=dev)
        for causal in cfg.causal:
            ms = _time(lambda: cga.prefill(q, k, v, causal=causal, out=o), flush, stream, reps)
            fl = workloads.prefill_flops(cfg.B, cfg.Hq, cfg.S, cfg.D, causal)
            tf = fl / (ms * 1e-3) / 1e12
            key = f"{name}_{'causal' if causal else 'noncausal'}"
            row = {"workload": cfg.name, "ms": ms, "us": ms * 1e3, "value": tf,
                   "unit": "TFLOP/s", "flops": fl, "dtype": cfg.dtype}
            if cfg.dtype == "bf16":
                row["frac_of_bf16_peak"] = tf / pk["bf16_tflops"]
            else:
                row["note"] = "fp32 I/O parity workload on CUDA cores (fp32 FMA): no roofline claim"
            out[key] = row
        del q, k, v, o
    cfg = workloads.CONFIGS["c4a"]
    q, kc, vc, sl = [t.to(dev) for t in workloads.config_decode_inputs(cfg, nan_fill=False)]
    o = torch.empty_like(q)
    by = workloads.decode_bytes(sl.cpu().tolist(), cfg.Hq, cfg.Hkv, cfg.D)
    ms = _time(lambda: cga.decode(q, kc, vc, sl, out=o), flush, stream, max(20, reps))
    row = {"workload": cfg.name, "us": ms * 1e3, "value": by / (ms * 1e-3) / 1e9, "unit": "GB/s",
           "bytes": by, "frac": by / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
    nsets = 40
    sets = [[t.to(dev) for t in workloads.config_decode_inputs(cfg, seed=200 + i, nan_fill=False)]
            for i in range(nsets)]
    outs = [torch.empty_like(x[0]) for x in sets]
    for (tq, tkc, tvc, tsl), to in zip(sets, outs):
        cga.decode(tq, tkc, tvc, tsl, out=to)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for (tq, tkc, tvc, tsl), to in zip(sets, outs):
            cga.decode(tq, tkc, tvc, tsl, out=to)
    graph.replay()
    torch.cuda.synchronize()
    g_ms = statistics.median(_time_graph(graph, flush, stream, max(5, steps // 2)))
    row["back_to_back"] = {"us_per_call": g_ms * 1e3 / nsets, "calls": nsets,
                           "value": by * nsets / (g_ms * 1e-3) / 1e9, "unit": "GB/s",
                           "frac": by * nsets / (g_ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
    out["c4a"] = row
    del graph, sets, outs
    return out


def _time_graph(graph, flush, stream, reps):
    ts = []
    for _ in range(reps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return ts


# --------------------------------------------------------------------------- our kernels


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    world, rank, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group(backend="nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from causal_gqa_attention_gb300 import build as cbuild

    cbuild.build()
    import causal_gqa_attention_gb300 as cga

    cga.load_library()
    pk = peaks()

    # inputs resident on the device
    q, k, v = [t.to(dev) for t in workloads.config_prefill_inputs(PREFILL)]
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dkc, dvc, dsl = workloads.config_decode_inputs(DECODE, nan_fill=False)
    dec_bytes = workloads.decode_bytes(dsl.tolist(), DECODE.Hq, DECODE.Hkv, DECODE.D)
    dq, dkc, dvc, dsl = dq.to(dev), dkc.to(dev), dvc.to(dev), dsl.to(dev)
    do = torch.empty_like(dq)
    cga.attn_reserve_workspace(DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.D, DECODE.max_len)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush_w.zero_()
        flush_r.sum()
    pflops = workloads.prefill_flops(PREFILL.B, PREFILL.Hq, PREFILL.S, PREFILL.D, True)
    stream = torch.cuda.current_stream(dev)

    def run_prefill():
        if args.only != "decode":
            cga.prefill(q, k, v, causal=True, out=o, lse=lse, return_lse=True)

    def run_decode():
        if args.only != "prefill":
            cga.decode(dq, dkc, dvc, dsl, out=do)

    for _ in range(args.warmup):
        run_prefill()
        run_decode()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush_l2()
        ev[s][0].record(stream)
        run_prefill()
        ev[s][1].record(stream)
        flush_l2()
        ev[s][2].record(stream)
        run_decode()
        ev[s][3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    assert cga.device_status() == 0, "device status word set during the bench"

    pre_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    dec_ms = [ev[s][2].elapsed_time(ev[s][3]) for s in range(args.steps)]
    pre_mean, pre_rate, pre_job = whole_job_rate(pflops, sum(pre_ms) / len(pre_ms), world, dev)
    dec_mean, dec_rate, _ = whole_job_rate(dec_bytes, sum(dec_ms) / len(dec_ms), world, dev)
    step_ms = pre_mean + dec_mean
    tflops = pre_rate / 1e12
    dec_gbs = dec_rate / 1e9

    # ---- decode, back to back: a CUDA graph of DECODE_CALLS calls over DECODE_SETS caches
    b2b = None
    if args.only != "prefill":
        sets = []
        for si in range(DECODE_SETS):
            tq, tkc, tvc, tsl = workloads.config_decode_inputs(DECODE, seed=100 + si, nan_fill=False)
            nb = workloads.decode_bytes(tsl.tolist(), DECODE.Hq, DECODE.Hkv, DECODE.D)
            sets.append((tq.to(dev), tkc.to(dev), tvc.to(dev), tsl.to(dev), nb))
        outs = [torch.empty_like(x[0]) for x in sets]
        for si in range(DECODE_SETS):  # warm (first-use set-up happens outside capture)
            cga.decode(sets[si][0], sets[si][1], sets[si][2], sets[si][3], out=outs[si])
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in range(DECODE_CALLS):
                si = c % DECODE_SETS
                cga.decode(sets[si][0], sets[si][1], sets[si][2], sets[si][3], out=outs[si])
        graph.replay()
        torch.cuda.synchronize()
        g_ms = []
        for _ in range(max(3, args.steps // 2)):
            flush_l2()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            g_ms.append(e0.elapsed_time(e1))
        g_ms = max_over_ranks(statistics.median(g_ms), world, dev)
        g_bytes = sum(sets[c % DECODE_SETS][4] for c in range(DECODE_CALLS))
        b2b = {"value": g_bytes / (g_ms * 1e-3) / 1e9, "unit": "GB/s",
               "us_per_call": g_ms * 1e3 / DECODE_CALLS, "calls": DECODE_CALLS,
               "cache_sets": DECODE_SETS, "frac": g_bytes / (g_ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
        del graph

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = [t.cpu().pin_memory() for t in (q, k, v)]
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hdq, hdk, hdv, hdsl = [t.cpu().pin_memory() for t in (dq, dkc, dvc, dsl)]
        hdo = torch.empty(do.shape, dtype=do.dtype).pin_memory()
        dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ddq, ddk, ddv, ddsl = (torch.empty_like(dq), torch.empty_like(dkc),
                               torch.empty_like(dvc), torch.empty_like(dsl))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdq, hdk, hdv, hdsl))
        d2h = ho.numel() * ho.element_size() + hdo.numel() * hdo.element_size()

        up_stream = torch.cuda.Stream(device=dev)
        down_stream = torch.cuda.Stream(device=dev)
        oo = torch.empty_like(q)
        od = torch.empty_like(do)
        nch = E2E_CHUNKS if PREFILL.B % E2E_CHUNKS == 0 else 1
        cb = PREFILL.B // nch

        def e2e_step():
            # The host link (not the GPU) bounds this step, so the prefill runs as nch calls on
            # batch slices: slice c's upload overlaps slice c-1's prefill and its output goes
            # down while slice c+1 computes; the decode inputs go up behind the last slice.
            ev_in = [torch.cuda.Event() for _ in range(nch)]
            ev_pre = [torch.cuda.Event() for _ in range(nch)]
            ev_dec_in = torch.cuda.Event()
            ev_dec = torch.cuda.Event()
            up_stream.wait_stream(stream)  # the previous step is done with every buffer
            down_stream.wait_stream(stream)
            with torch.cuda.stream(up_stream):
                for c in range(nch):
                    sl = slice(c * cb, (c + 1) * cb)
                    dq2[sl].copy_(hq[sl], non_blocking=True)
                    dk2[sl].copy_(hk[sl], non_blocking=True)
                    dv2[sl].copy_(hv[sl], non_blocking=True)
                    ev_in[c].record(up_stream)
                ddq.copy_(hdq, non_blocking=True)
                ddk.copy_(hdk, non_blocking=True)
                ddv.copy_(hdv, non_blocking=True)
                ddsl.copy_(hdsl, non_blocking=True)
                ev_dec_in.record(up_stream)
            for c in range(nch):
                sl = slice(c * cb, (c + 1) * cb)
                stream.wait_event(ev_in[c])
                cga.prefill(dq2[sl], dk2[sl], dv2[sl], causal=True, out=oo[sl])
                ev_pre[c].record(stream)
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(ev_pre[c])
                    ho[sl].copy_(oo[sl], non_blocking=True)
            stream.wait_event(ev_dec_in)
            cga.decode(ddq, ddk, ddv, ddsl, out=od)
            ev_dec.record(stream)
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(ev_dec)
                hdo.copy_(od, non_blocking=True)
            stream.wait_stream(down_stream)  # the step ends when its results are on the host

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e_steps = max(3, min(args.steps, 10))
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world, dev)
        e2e = {"value": pflops * world / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "note": "prefill flops over the whole step incl. decode and host copies",
               "prefill_calls_per_step": nch}

    extras = None
    configs = None
    if not args.no_extras and args.only == "all":
        extras = time_extras(cga, dev, stream, flush_l2, args.steps)
        configs = time_configs(cga, dev, stream, flush_l2, pk, args.steps)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = oracle_sample(args.cpu_seconds)
        cpu = {"value": r["prefill_tflops"], "unit": "TFLOP/s", "cores": r["cores"],
               "kind": "oracle", "sample": r["sample"], "decode_gbs": r["decode_gbs"],
               "cpu_model": cpu_model(), "single_core": oracle_single_core()}

    if args.only != "all":
        if rank == 0:
            print(json.dumps({"only": args.only, "prefill_ms": pre_mean, "decode_ms": dec_mean,
                              "prefill_tflops": tflops, "decode_gbs": dec_gbs,
                              "decode_back_to_back": b2b}), flush=True)
        return
    if rank == 0:
        peak_t = pk["bf16_tflops"]
        traffic = recorded_traffic()
        line = {
            "metric": METRIC,
            "value": pre_job / 1e12,
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": step_ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": config_block(),
            "prefill": {"value": tflops, "unit": "TFLOP/s", "ms": pre_mean,
                        "flops": pflops, "frac_of_bf16_peak": tflops / peak_t,
                        "frac_of_bf16_sustained": tflops / pk["bf16_tflops_sustained"],
                        "frac_of_nominal": tflops / NOMINAL_BF16_TFLOPS},
            "decode": {"value": dec_gbs, "unit": "GB/s", "ms": dec_mean, "bytes": dec_bytes,
                       "back_to_back": b2b,
                       "roofline": {"bound": "hbm", "achieved": dec_gbs,
                                    "peak": pk["hbm_gbs"], "unit": "GB/s",
                                    "frac": dec_gbs / pk["hbm_gbs"],
                                    "frac_of_nominal": dec_gbs / NOMINAL_HBM_GBS,
                                    "traffic": traffic["decode_stream_kernel"]
                                    if args.decode_batch is None and args.decode_len is None
                                    else None}},
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak_t,
                         "unit": "TFLOP/s", "frac": tflops / peak_t,
                         "traffic": traffic["prefill_tc_kernel"]
                         if args.prefill_batch is None and args.prefill_seq is None else None,
                         "kernel": "prefill_tc_kernel", "peak_source": pk["source"]},
            "e2e": e2e,
            "configs": configs,
            "extras": extras,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": 5 * args.steps,  # V conversion, V scale, prefill; decode stream + merge
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
