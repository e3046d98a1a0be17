#!/usr/bin/env python
"""Throughput of the attention hot path on B300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl attn07|reference]

One step is one pass of the whole hot path on synthetic inputs already resident
in device memory:
  * prefill  -- causal grouped-query attention, B=1, Hq=32, Hkv=8, N=16384,
                d=128, bf16 N(0,1)*0.5 (attn_fwd, tensor-core kernel), and
  * decode   -- B=64 single-token queries against a paged cache, lengths
                U[1024,32768], Hq=32, Hkv=8, d=128, 16-token pages, permuted
                page table (attn_decode_paged: split kernel + merge kernel).
Both inputs are larger than the 126 MB L2 (prefill 335 MB, decode ~4.4 GB), so
no flush is needed between steps.

``value`` is prefill TFLOP/s (causal FLOPs 2*B*Hq*N^2*d over the prefill
launches' device time, CUDA events on the launch stream); ``decode`` reports
KV-cache GB/s (4096 bytes per cached token over the decode launches' time).
Under torchrun every rank runs the same workload (replicas; no data-path
collective): value = all ranks' FLOPs / max-over-ranks time.

``--impl reference`` times the fp64 CPU oracle on the host cores on bounded
samples of the same prefill workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill TFLOP/s (% BF16 tensor peak); paged decode KV GB/s (% HBM peak)"
PREFILL = "gqa_causal_n16384"
DECODE = "decode_paged_b64"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ---------------------------------------------------------------- process layout

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    world, rank, _ = dist_env()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return world, rank


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity for one process)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- peaks, clocks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def library_fingerprint() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attn_fwd_07_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_fingerprint") != library_fingerprint():
            return None
        return d["kernels"][kernel]["dram_bytes_per_launch"]
    except Exception:
        return None


# ---------------------------------------------------------------- workloads

def prefill_flops(w) -> float:
    B, N, Hq, d = w.q.shape
    return 2.0 * B * Hq * N * N * d if w.causal else 4.0 * B * Hq * N * N * d


def decode_bytes(w) -> float:
    Hkv, d = w.k_cache.shape[2], w.k_cache.shape[3]
    return 2.0 * Hkv * d * 2.0 * float(w.seq_lens.sum())  # K and V, bf16


def cpu_oracle_sample(w, seconds: float, seed: int = 0, rows_per_batch: int = 1024):
    """Time the fp64 oracle on random query rows of the prefill workload until
    `seconds` have passed; FLOPs counted like the GPU's (4 * keys * d per row)."""
    from oracle import oracle
    q, k, v = (t.float().numpy() for t in (w.q, w.k, w.v))
    B, N, Hq, d = w.q.shape
    rng = np.random.default_rng(seed)
    flops, rows_done, t0 = 0.0, 0, time.perf_counter()
    while True:
        rows = np.stack([rng.integers(0, B, rows_per_batch), rng.integers(0, Hq, rows_per_batch),
                         rng.integers(0, N, rows_per_batch)], 1).astype(np.int32)
        oracle.attn_rows(q, k, v, rows, w.causal, w.scale)
        keys = (rows[:, 2].astype(np.float64) + 1.0) if w.causal else np.full(len(rows), N, float)
        flops += float(4.0 * keys.sum() * d)
        rows_done += len(rows)
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return flops / el / 1e12, el, rows_done, oracle.max_threads()


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from attn_fwd_07_b300 import inputs
    w = inputs.make(PREFILL)
    per_step = max(0.5, args.ref_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, 0.05)
    vals, els, rows = [], 0.0, 0
    for s in range(args.steps):
        tf, el, r, cores = cpu_oracle_sample(w, per_step, seed=s + 1)
        vals.append(tf)
        els += el
        rows += r
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * els / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL, "B": 1, "Hq": 32, "Hkv": 8, "N": 16384, "d": 128,
                   "causal": True, "parallelism": "replicas", "l2": "not applicable (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "%d random causal query rows of the prefill workload over %d "
                                   "steps (%.1f s)" % (rows, args.steps, els)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def run_gpu(args):
    world, rank = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import attn_fwd_07_b300 as A
    from attn_fwd_07_b300 import inputs
    A.load_library()

    # ---- inputs (host, seeded) -> device
    wp = inputs.make(PREFILL)
    wd = inputs.make(DECODE)
    qp, kp, vp = (t.to(dev) for t in (wp.q, wp.k, wp.v))
    B, N, Hq, d = wp.q.shape
    op = torch.empty_like(qp)
    lsep = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    qd, kc, vc, pt, sl = (t.to(dev) for t in (wd.q, wd.k_cache, wd.v_cache, wd.page_table,
                                               wd.seq_lens))
    od = torch.empty_like(qd)
    lsed = torch.empty(qd.shape[:2], dtype=torch.float32, device=dev)
    Bd, Hqd, dd = wd.q.shape
    ws = torch.empty(A.attn_decode_workspace_size(Bd, Hqd, kc.shape[2], dd, pt.shape[1],
                                                  kc.shape[1]), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    fl_p = prefill_flops(wp)
    by_d = decode_bytes(wd)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        A.attn_fwd(qp, kp, vp, True, wp.scale, o=op, lse=lsep, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        A.attn_decode_paged(qd, kc, vc, pt, sl, wd.scale, o=od, lse=lsed, workspace=ws,
                            stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = A.attn_get_device_status()
    if st != 0:
        raise RuntimeError("device status after warm-up: " + A.attn_status_string(st))

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    t_begin.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    st = A.attn_get_device_status()
    if st != 0:
        raise RuntimeError("device status after timing: " + A.attn_status_string(st))

    total_ms = t_begin.elapsed_time(t_end)
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    pre_sum = max_over_ranks(sum(pre_ms), world, dev)
    dec_sum = max_over_ranks(sum(dec_ms), world, dev)
    total_ms = max_over_ranks(total_ms, world, dev)
    value = sum_over_ranks(fl_p * args.steps, world, dev) / (pre_sum * 1e-3) / 1e12
    dec_gbs = sum_over_ranks(by_d * args.steps, world, dev) / (dec_sum * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers (pinned), copies timed
    n_e2e = max(1, min(args.steps, args.e2e_steps))
    hq, hk, hv = (t.pin_memory() for t in (wp.q, wp.k, wp.v))
    ho, hl = torch.empty_like(hq).pin_memory(), torch.empty(lsep.shape, dtype=torch.float32).pin_memory()
    h2d_p = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h_p = ho.numel() * ho.element_size() + hl.numel() * 4

    def e2e_prefill():
        qp.copy_(hq, non_blocking=True)
        kp.copy_(hk, non_blocking=True)
        vp.copy_(hv, non_blocking=True)
        A.attn_fwd(qp, kp, vp, True, wp.scale, o=op, lse=lsep, stream=stream)
        ho.copy_(op, non_blocking=True)
        hl.copy_(lsep, non_blocking=True)

    e2e_prefill()
    torch.cuda.synchronize(dev)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n_e2e):
        e2e_prefill()
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(a.elapsed_time(b), world, dev)
    e2e_val = sum_over_ranks(fl_p * n_e2e, world, dev) / (e2e_ms * 1e-3) / 1e12
    del hq, hk, hv, ho, hl

    hqd, hkc, hvc, hpt, hsl = (t.pin_memory() for t in (wd.q, wd.k_cache, wd.v_cache,
                                                        wd.page_table, wd.seq_lens))
    hod = torch.empty_like(hqd).pin_memory()
    hld = torch.empty(lsed.shape, dtype=torch.float32).pin_memory()
    h2d_d = sum(t.numel() * t.element_size() for t in (hqd, hkc, hvc, hpt, hsl))
    d2h_d = hod.numel() * hod.element_size() + hld.numel() * 4

    def e2e_decode():
        for dst, src in ((qd, hqd), (kc, hkc), (vc, hvc), (pt, hpt), (sl, hsl)):
            dst.copy_(src, non_blocking=True)
        A.attn_decode_paged(qd, kc, vc, pt, sl, wd.scale, o=od, lse=lsed, workspace=ws,
                            stream=stream)
        hod.copy_(od, non_blocking=True)
        hld.copy_(lsed, non_blocking=True)

    e2e_decode()
    torch.cuda.synchronize(dev)
    barrier(world)
    a.record(stream)
    for _ in range(n_e2e):
        e2e_decode()
    b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_dms = max_over_ranks(a.elapsed_time(b), world, dev)
    e2e_dval = sum_over_ranks(by_d * n_e2e, world, dev) / (e2e_dms * 1e-3) / 1e9
    del hqd, hkc, hvc, hpt, hsl, hod, hld

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, el, rows, cores = cpu_oracle_sample(wp, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": "%d random causal query rows of the prefill workload (%.1f s, fp64)"
                         % (rows, el)}

    peaks, peak_src = load_peaks()
    pre_launch_ms = pre_sum / args.steps
    dec_launch_ms = dec_sum / args.steps
    roof_p = {"bound": "tensor", "achieved": fl_p / (pre_launch_ms * 1e-3) / 1e12,
              "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
              "peak_source": "%s bf16 burst (cuBLAS)" % peak_src,
              "traffic": profiled_traffic("prefill_tc_kernel")}
    roof_p["frac"] = roof_p["achieved"] / roof_p["peak"]
    roof_d = {"bound": "hbm", "achieved": by_d / (dec_launch_ms * 1e-3) / 1e9,
              "peak": peaks["hbm_gbs"], "unit": "GB/s",
              "peak_source": "%s copy bandwidth" % peak_src,
              "traffic": profiled_traffic("decode_split_kernel")}
    roof_d["frac"] = roof_d["achieved"] / roof_d["peak"]

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "%s + %s" % (PREFILL, DECODE), "prefill": {
                "B": B, "Hq": Hq, "Hkv": int(kp.shape[2]), "N": N, "d": d, "causal": True,
                "values": "bf16 N(0,1)*0.5"},
                "decode": {"B": Bd, "Hq": Hqd, "Hkv": int(kc.shape[2]), "d": dd,
                           "page_size": int(kc.shape[1]), "lengths": "U[1024,32768]",
                           "total_tokens": int(wd.seq_lens.sum())},
                "parallelism": "replicas" if world > 1 else "single GPU",
                "l2": "inputs larger than L2 (prefill 335 MB, decode %.1f GB)" % (by_d / 1e9)},
            "roofline": roof_p,
            "decode": {"value": dec_gbs, "unit": "GB/s", "ms_per_step": dec_sum / args.steps,
                       "roofline": roof_d,
                       "e2e": {"value": e2e_dval, "unit": "GB/s", "h2d_bytes_per_step": h2d_d,
                               "d2h_bytes_per_step": d2h_d}},
            "prefill_ms_per_step": pre_sum / args.steps,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d_p,
                    "d2h_bytes_per_step": d2h_p},
            "cpu_baseline": cpu,
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["attn07", "reference"], default="attn07")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
