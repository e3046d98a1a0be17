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

``--workload NAME`` benches one named workload alone (any of the five in
attn_fwd_07_b300.inputs.WORKLOADS; ``--batch`` replaces its batch size) with the
same timing rules; when its inputs fit in twice the L2, a 252 MB buffer is
written between steps to flush it.

``--impl reference`` times the fp64 CPU oracle on the host cores on bounded
samples of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
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


# the source files each profiled kernel is built from (its own header and the PTX
# wrappers); a counter taken on other sources no longer describes the kernel
KERNEL_SOURCES = {
    "prefill_tc_kernel": ("prefill_tc.cuh", "ptx.cuh"),
    "prefill_simt_kernel": ("prefill_simt.cuh", "ptx.cuh"),
    "prefill_simt_rows_kernel<4>": ("prefill_simt.cuh", "ptx.cuh"),
    "prefill_simt_rows_kernel<2>": ("prefill_simt.cuh", "ptx.cuh"),
    "decode_split_kernel<0>": ("decode.cuh", "ptx.cuh"),
    "decode_split_kernel<1>": ("decode.cuh", "ptx.cuh"),
    "decode_split_kernel<2>": ("decode.cuh", "ptx.cuh"),
}


def _code_only(text: bytes) -> bytes:
    """C/C++/CUDA source without comments, blank lines or trailing spaces: what a
    comment-only edit leaves unchanged (string literals in these sources hold no
    comment markers)."""
    t = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    t = re.sub(rb"//[^\n]*", b"", t)
    lines = [ln.rstrip() for ln in t.split(b"\n")]
    return b"\n".join(ln for ln in lines if ln)


def kernel_fingerprint(kernel: str, read=None) -> str:
    """sha256 (16 hex digits) over the code of the kernel's source files, comments left
    out.  `read(name) -> bytes` defaults to the working tree's attn_fwd_07_b300/csrc/<name>."""
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "attn_fwd_07_b300", "csrc", name), "rb") as f:
                return f.read()
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode())
        h.update(_code_only(read(name)))
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload`, from the committed
    ncu summary, or None when there is none or it was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d["kernels"]["%s@%s" % (kernel, workload)]
        if e.get("source_fingerprint") != kernel_fingerprint(kernel):
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


# ---------------------------------------------------------------- workloads

def prefill_flops(w) -> float:
    """Algorithmic FLOPs of one prefill: 4*d per (query, key) pair (QK^T and PV, 2*d
    each) over N^2 pairs per sequence and head, halved when causal (2*B*Hq*N^2*d); a
    sliding window counts its allowed pairs exactly."""
    if hasattr(w, "cu_seqlens_q"):
        # a chunk per sequence: query i of q_len sees positions <= ctx - q_len + i
        _, Hq, d = w.q.shape
        ctx = w.seq_lens.numpy().astype(np.float64)
        ql = w.q_lens.astype(np.float64)
        if w.causal:
            pairs = float((ql * (ctx - ql) + ql * (ql + 1) / 2.0).sum())
        else:
            pairs = float((ql * ctx).sum())
        return 4.0 * Hq * d * pairs
    if getattr(w, "window", None) is not None:
        # a sliding window: the exact number of allowed (query, key) pairs
        B, N, Hq, d = w.q.shape
        wl, wr = w.window
        i = np.arange(N, dtype=np.float64)
        lo = np.zeros(N) if wl < 0 else np.maximum(0.0, i - wl)
        hi = np.full(N, N - 1.0) if wr < 0 else np.minimum(N - 1.0, i + wr)
        return 4.0 * Hq * d * B * float((hi - lo + 1).sum())
    if w.q.dim() == 4:
        B, N, Hq, d = w.q.shape
        pairs = B * float(N) * N
    else:
        _, Hq, d = w.q.shape
        lens = w.lens.astype(np.float64)
        pairs = float((lens * lens).sum())
    return 4.0 * Hq * d * pairs * (0.5 if w.causal else 1.0)


def decode_bytes(w) -> float:
    """Algorithmic bytes of one decode: each cached token's K and V rows read once."""
    Hkv, d = w.k_cache.shape[2], w.k_cache.shape[3]
    return 2.0 * Hkv * d * w.k_cache.element_size() * float(w.seq_lens.sum())


def nbytes(*ts) -> int:
    return int(sum(t.numel() * t.element_size() for t in ts))


def workload_shape(kind, w, spec):
    """The workload's sizes as the JSON line's config reports them (both arms)."""
    if kind in ("decode", "decode_fp8", "decode_int8"):
        B, Hq, d = w.q.shape
        shape = {"B": B, "Hq": Hq, "Hkv": int(w.k_cache.shape[2]), "d": d,
                 "page_size": int(w.k_cache.shape[1]), "total_tokens": int(w.seq_lens.sum())}
    elif kind == "chunk":
        T, Hq, d = w.q.shape
        shape = {"seqs": len(w.q_lens), "total_q": T, "cached_tokens": int(w.seq_lens.sum()),
                 "Hq": Hq, "Hkv": int(w.k_cache.shape[2]), "d": d, "causal": w.causal}
    elif kind == "window":
        B, N, Hq, d = w.q.shape
        shape = {"B": B, "N": N, "Hq": Hq, "Hkv": int(w.k.shape[2]), "d": d,
                 "window": list(w.window)}
    elif kind == "varlen":
        T, Hq, d = w.q.shape
        shape = {"seqs": len(w.lens), "total_tokens": T, "Hq": Hq, "Hkv": int(w.k.shape[1]),
                 "d": d, "causal": w.causal}
    else:
        B, N, Hq, d = w.q.shape
        shape = {"B": B, "N": N, "Hq": Hq, "Hkv": int(w.k.shape[2]), "d": d,
                 "causal": w.causal}
    shape["values"] = spec.description
    shape["name"] = spec.name
    return shape


def config_key(kind):
    return "prefill" if kind == "dense" else kind


class Leg:
    """One workload of the step: device-resident inputs, a launch, its algorithmic work,
    and an end-to-end variant that copies the inputs in from pinned host memory and the
    results out."""

    def __init__(self, name, dev, batch=None):
        import attn_fwd_07_b300 as A
        from attn_fwd_07_b300 import inputs
        self.A = A
        self.name = name
        self.spec = inputs.WORKLOADS[name]
        self.kind = self.spec.kind
        w = inputs.make(name, batch)
        self.w = w
        self.scale = w.scale
        if self.kind in ("decode", "decode_fp8", "decode_int8"):
            self.host = [w.q, w.k_cache, w.v_cache, w.page_table, w.seq_lens]
            if self.kind in ("decode_fp8", "decode_int8"):
                self.host += [w.k_scale, w.v_scale]
            self.dev = [t.to(dev) for t in self.host]
            q, kc = self.dev[0], self.dev[1]
            B, Hq, d = w.q.shape
            self.o = torch.empty_like(q)
            self.lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
            self.ws = torch.empty(A.attn_decode_workspace_size(B, Hq, d, w.page_table.shape[1],
                                                               kc.shape[1]),
                                  dtype=torch.uint8, device=dev)
            self.work, self.unit, self.bound = decode_bytes(w), "GB/s", "hbm"
            # (the split kernel's template argument: 0 bf16, 1 FP8, 2 INT8 cache)
            self.kernel = "decode_split_kernel<%d>" % {"decode": 0, "decode_fp8": 1,
                                                       "decode_int8": 2}[self.kind]
        else:
            if self.kind == "chunk":
                self.host = [w.q, w.k_cache, w.v_cache, w.page_table, w.seq_lens, w.cu_seqlens_q]
            else:
                self.host = [w.q, w.k, w.v] + ([w.cu_seqlens] if self.kind == "varlen" else [])
            self.dev = [t.to(dev) for t in self.host]
            q = self.dev[0]
            self.o = torch.empty_like(q)
            if self.kind == "chunk":
                T, Hq, d = w.q.shape
                self.max_len = int(w.q_lens.max())
                self.lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
            elif self.kind == "varlen":
                T, Hq, d = w.q.shape
                self.max_len = int(w.lens.max())
                self.lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
            else:
                B, N, Hq, d = w.q.shape
                self.lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
            self.f32 = w.q.dtype == torch.float32
            self.work, self.unit = prefill_flops(w), "TFLOP/s"
            self.bound = "alu" if self.f32 else "tensor"
            self.kernel = simt_kernel(w.q.shape, dev) if self.f32 else "prefill_tc_kernel"
        self.shape = workload_shape(self.kind, w, self.spec)
        # end to end: a decode step's query, page table and lengths come from the host and
        # its O and LSE go back, while the cache stays resident on the device (where a
        # serving process keeps it between steps); every other workload copies all of
        # its inputs in
        self.e2e_in = ([0, 3, 4] if self.kind in ("decode", "decode_fp8", "decode_int8")
                       else list(range(len(self.host))))
        self.resident = (nbytes(*[t for i, t in enumerate(self.host) if i not in self.e2e_in])
                         if self.kind in ("decode", "decode_fp8", "decode_int8") else 0)
        self.h2d = nbytes(*[self.host[i] for i in self.e2e_in])
        self.d2h = nbytes(self.o, self.lse)

    def launch(self, stream):
        A, d = self.A, self.dev
        if self.kind == "decode":
            A.attn_decode_paged(d[0], d[1], d[2], d[3], d[4], self.scale, o=self.o, lse=self.lse,
                                workspace=self.ws, stream=stream)
        elif self.kind == "decode_fp8":
            A.attn_decode_paged_fp8(d[0], d[1], d[2], d[5], d[6], d[3], d[4], self.scale,
                                    o=self.o, lse=self.lse, workspace=self.ws, stream=stream)
        elif self.kind == "decode_int8":
            A.attn_decode_paged_int8(d[0], d[1], d[2], d[5], d[6], d[3], d[4], self.scale,
                                     o=self.o, lse=self.lse, workspace=self.ws, stream=stream)
        elif self.kind == "chunk":
            A.attn_fwd_chunked_paged(d[0], d[1], d[2], d[3], d[4], d[5], self.max_len,
                                     self.w.causal, self.scale, o=self.o, lse=self.lse,
                                     stream=stream)
        elif self.kind == "window":
            A.attn_fwd_window(d[0], d[1], d[2], self.w.window[0], self.w.window[1], self.scale,
                              o=self.o, lse=self.lse, stream=stream)
        elif self.kind == "varlen":
            A.attn_fwd_varlen(d[0], d[1], d[2], d[3], self.max_len, self.w.causal, self.scale,
                              o=self.o, lse=self.lse, stream=stream)
        elif self.kind == "two_pass":
            A.attn_fwd_two_pass(d[0], d[1], d[2], self.w.causal, self.scale, o=self.o,
                                lse=self.lse, stream=stream)
        elif self.f32:
            A.attn_fwd_f32(d[0], d[1], d[2], self.w.causal, self.scale, o=self.o, lse=self.lse,
                           stream=stream)
        else:
            A.attn_fwd(d[0], d[1], d[2], self.w.causal, self.scale, o=self.o, lse=self.lse,
                       stream=stream)

    def rate(self, work, ms):
        """work units (FLOPs or bytes) over ms -> TFLOP/s or GB/s."""
        return work / (ms * 1e-3) / (1e12 if self.unit == "TFLOP/s" else 1e9)

    def e2e_setup(self):
        self.h_in = {i: self.host[i].pin_memory() for i in self.e2e_in}
        self.h_out = [torch.empty(self.o.shape, dtype=self.o.dtype).pin_memory(),
                      torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()]

    def e2e_step(self, stream):
        if self.kind == "dense" and not self.f32:
            # the library's host-buffer entry point: it copies the inputs in, runs the
            # prefill and copies O and LSE out (pipelined over key/value head groups),
            # returning when the host buffers hold the result
            self.A.attn_fwd_host(self.h_in[0], self.h_in[1], self.h_in[2], self.w.causal,
                                 self.scale, o=self.h_out[0], lse=self.h_out[1], stream=stream)
            return
        for i, src in self.h_in.items():
            self.dev[i].copy_(src, non_blocking=True)
        self.launch(stream)
        self.h_out[0].copy_(self.o, non_blocking=True)
        self.h_out[1].copy_(self.lse, non_blocking=True)

    def e2e_teardown(self):
        del self.h_in, self.h_out
        if self.kind == "dense" and not self.f32:
            self.A.attn_release_host_staging()


def simt_kernel(q_shape, dev) -> str:
    """The fp32 kernel attn_fwd_f32 launches for q of shape [B, N, Hq, d]: with C CTAs of
    16 rows, 2-row CTAs when 8 C <= #SM, 4-row CTAs when 2 C <= #SM, else 16-row CTAs."""
    B, N, Hq, _ = q_shape
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ctas16 = ((N + 15) // 16) * Hq * B
    if 8 * ctas16 <= sms:
        return "prefill_simt_rows_kernel<2>"
    if 2 * ctas16 <= sms:
        return "prefill_simt_rows_kernel<4>"
    return "prefill_simt_kernel"


def launches_per_call(leg) -> int:
    return 2 if leg.kind in ("decode", "decode_fp8", "decode_int8", "two_pass") else 1


_ORACLE_INPUTS = {}


def _oracle_inputs(w, key, make):
    """A workload's arrays in the form the oracle takes, converted once per workload
    (the decode cache alone is 9.4 GB as float32); the workload is kept with them so
    that its id is not reused."""
    k = (id(w), key)
    if k not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[k] = (w, make())
    return _ORACLE_INPUTS[k][1]


def cpu_oracle_sample(w, kind: str, seconds: float, seed: int = 0):
    """Time the fp64 oracle on random pieces of a workload until `seconds` have passed.

    Prefill (dense or packed): batches of random query rows, each counted like the GPU's
    work (4*d FLOPs per allowed key).  Decode: random whole sequences, counted as their
    K and V bytes.  Returns (rate in TFLOP/s or GB/s, elapsed s, description, threads)."""
    from oracle import oracle
    rng = np.random.default_rng(seed)
    work, done, t0 = 0.0, 0, time.perf_counter()
    if kind == "chunk":
        args = _oracle_inputs(w, "chunk", lambda: (
            w.q.float().numpy(), w.k_cache.float().numpy(), w.v_cache.float().numpy(),
            w.page_table.numpy(), w.seq_lens.numpy(), w.cu_seqlens_q.numpy(), w.causal,
            w.scale))
        cu, ctx = w.cu_seqlens_q.numpy(), w.seq_lens.numpy()
        Tq, Hq, d = w.q.shape
        n_rows = 256 if seconds >= 1.0 else 64
        t0 = time.perf_counter()
        while True:
            t = rng.integers(0, Tq, n_rows)
            rows = np.stack([t, rng.integers(0, Hq, n_rows)], 1)
            oracle.chunk_paged_rows(*args, rows=rows)
            sq = np.searchsorted(cu, t, side="right") - 1
            pos = ctx[sq] - (cu[sq + 1] - cu[sq]) + (t - cu[sq])
            keys = (pos + 1.0) if w.causal else ctx[sq].astype(np.float64)
            work += float(4.0 * d * keys.sum())
            done += n_rows
            el = time.perf_counter() - t0
            if el >= seconds:
                return work / el / 1e12, el, "%d random query rows (%.1f s, fp64)" % (done, el), \
                    oracle.max_threads()
    if kind in ("decode_fp8", "decode_int8"):
        args = _oracle_inputs(w, kind, lambda: (
            w.q.float().numpy(), w.k_cache.numpy(), w.v_cache.numpy(), w.k_scale.numpy(),
            w.v_scale.numpy(), w.page_table.numpy(), w.seq_lens.numpy()))
        fn = oracle.decode_paged_fp8 if kind == "decode_fp8" else oracle.decode_paged_int8
        sl = w.seq_lens.numpy()
        Hkv, d = w.k_cache.shape[2], w.k_cache.shape[3]
        t0 = time.perf_counter()
        while True:
            b = int(rng.integers(0, len(sl)))
            fn(*args, w.scale, seqs=[b])
            work += 2.0 * Hkv * d * 1.0 * float(sl[b])
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return work / el / 1e9, el, "%d random sequences (%.1f s, fp64)" % (done, el), \
                    oracle.max_threads()
    if kind == "decode":
        arrs = _oracle_inputs(w, "decode", lambda: [t.float().numpy()
                                                    for t in (w.q, w.k_cache, w.v_cache)])
        pt, sl = w.page_table.numpy(), w.seq_lens.numpy()
        Hkv, d = w.k_cache.shape[2], w.k_cache.shape[3]
        t0 = time.perf_counter()
        while True:
            b = int(rng.integers(0, len(sl)))
            oracle.decode_paged(*arrs, pt, sl, w.scale, seqs=[b])
            work += 2.0 * Hkv * d * 2.0 * float(sl[b])
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return work / el / 1e9, el, "%d random sequences (%.1f s, fp64)" % (done, el), \
                    oracle.max_threads()
    def make_segs():
        if w.q.dim() == 4:
            return [(w.q.float().numpy(), w.k.float().numpy(), w.v.float().numpy())]
        # packed: each sequence as a batch-1 dense problem
        cu = w.cu_seqlens.numpy()
        q, k, v = (t.float().numpy() for t in (w.q, w.k, w.v))
        return [(q[None, a:b], k[None, a:b], v[None, a:b]) for a, b in zip(cu[:-1], cu[1:])
                if b > a]

    segs = _oracle_inputs(w, "prefill", make_segs)
    n_rows = 1024 if seconds >= 1.0 else 128
    t0 = time.perf_counter()
    while True:
        q, k, v = segs[int(rng.integers(0, len(segs)))]
        B, N, Hq, d = q.shape
        rows = np.stack([rng.integers(0, B, n_rows), rng.integers(0, Hq, n_rows),
                         rng.integers(0, N, n_rows)], 1).astype(np.int32)
        win = getattr(w, "window", None)
        if win is not None:
            oracle.attn_window_rows(q, k, v, rows, win[0], win[1], w.scale)
            i = rows[:, 2].astype(np.float64)
            lo = np.zeros(n_rows) if win[0] < 0 else np.maximum(0.0, i - win[0])
            hi = np.full(n_rows, N - 1.0) if win[1] < 0 else np.minimum(N - 1.0, i + win[1])
            keys = hi - lo + 1
        else:
            oracle.attn_rows(q, k, v, rows, w.causal, w.scale)
            keys = (rows[:, 2].astype(np.float64) + 1.0) if w.causal else np.full(n_rows,
                                                                                 float(N))
        work += float(4.0 * keys.sum() * d)
        done += n_rows
        el = time.perf_counter() - t0
        if el >= seconds:
            return work / el / 1e12, el, "%d random query rows (%.1f s, fp64)" % (done, el), \
                oracle.max_threads()


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The fp64 oracle, as it stands, on the host cores: each step a bounded sample of
    the same workloads, same metric and units as the GPU arm (value = the first
    workload's rate; the default step's decode leg is reported beside it)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from attn_fwd_07_b300 import inputs
    names = [args.workload] if args.workload else [PREFILL, DECODE]
    # the whole run takes about ref_seconds (plus one conversion per workload): each step
    # gets an equal share, and a sample always completes at least one batch of rows
    per_step = args.ref_seconds / max(1, args.steps) / len(names)
    results = []
    shapes = {}
    for name in names:
        kind = inputs.WORKLOADS[name].kind
        w = inputs.make(name, args.batch)
        shapes[config_key(kind)] = workload_shape(kind, w, inputs.WORKLOADS[name])
        for _ in range(args.warmup):
            cpu_oracle_sample(w, kind, 0.05)
        vals, els, descs, cores = [], 0.0, [], 0
        for s in range(args.steps):
            v, el, desc, cores = cpu_oracle_sample(w, kind, per_step, seed=s + 1)
            vals.append(v)
            els += el
            descs.append(desc)
        unit = "GB/s" if kind.startswith("decode") else "TFLOP/s"
        results.append((name, kind, float(np.mean(vals)), unit, els, descs[0], cores))
    name, kind, value, unit, els, desc, cores = results[0]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * sum(r[4] for r in results) / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict({"workload": " + ".join(names), "batch_override": args.batch,
                        "parallelism": "single process", "l2": "not applicable (CPU)"},
                       **shapes),
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": "per step: %s; %d steps" % (desc, args.steps)},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    for name, kind, v, u, els, desc, cores in results[1:]:
        line[kind] = {"value": v, "unit": u, "sample": "per step: " + desc}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

L2_BYTES = 126 * 1024 * 1024


# fp32 CUDA-core peak (no measured figure exists for it): 148 SMs x 128 fp32 lanes x 2 FLOP
# per fused multiply-add x 2032 MHz, the maximum SM clock
ALU_F32_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def roofline(leg, launch_ms, peaks, peak_src):
    if leg.bound == "alu":
        r = {"bound": "alu", "achieved": leg.rate(leg.work, launch_ms), "peak": ALU_F32_TFLOPS,
             "unit": "TFLOP/s",
             "peak_source": "derived: 148 SMs x 128 fp32 lanes x 2 FLOP x 2032 MHz"}
    elif leg.bound == "tensor":
        r = {"bound": "tensor", "achieved": leg.rate(leg.work, launch_ms),
             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
             "peak_source": "%s bf16 burst (cuBLAS)" % peak_src}
    else:
        r = {"bound": "hbm", "achieved": leg.rate(leg.work, launch_ms),
             "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "peak_source": "%s copy bandwidth" % peak_src}
    r["frac"] = r["achieved"] / r["peak"]
    r["traffic"] = profiled_traffic(leg.kernel, leg.name)
    return r


def run_gpu(args):
    world, rank = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import attn_fwd_07_b300 as A
    A.load_library()

    names = [args.workload] if args.workload else [PREFILL, DECODE]
    legs = [Leg(n, dev, args.batch) for n in names]
    stream = torch.cuda.current_stream(dev)
    resident = sum(nbytes(*leg.dev, leg.o, leg.lse) for leg in legs)
    flush = None
    if resident < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    nl = len(legs)

    def step(ev=None):
        if flush is not None:
            flush.zero_()
        for i, leg in enumerate(legs):
            if ev is not None:
                ev[i][0].record(stream)
            leg.launch(stream)
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = A.attn_get_device_status()
    if st != 0:
        raise RuntimeError("device status after warm-up: " + A.attn_status_string(st))

    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nl)]
           for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    # The device first spins (about 0.2 ms per timed step) while the host enqueues every
    # timed step, so that no step's device time includes the host's launch latency: a
    # small workload's kernel runs shorter than the Python call that launches it.  The
    # spin lies before the first step's start event.
    torch.cuda._sleep(int(min(args.steps, 500) * 400_000))
    for s in range(args.steps):
        step(evs[s])
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    st = A.attn_get_device_status()
    if st != 0:
        raise RuntimeError("device status after timing: " + A.attn_status_string(st))

    leg_ms = [max_over_ranks(sum(evs[s][i][0].elapsed_time(evs[s][i][1])
                                 for s in range(args.steps)), world, dev) for i in range(nl)]
    leg_val = [legs[i].rate(sum_over_ranks(legs[i].work * args.steps, world, dev), leg_ms[i])
               for i in range(nl)]
    # the distribution of one leg's per-step device time: median and 90th percentile
    # (each the maximum over ranks)
    step_ms = []
    for i in range(nl):
        t = sorted(evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps))
        p90 = t[min(len(t) - 1, int(math.ceil(0.9 * len(t))) - 1)]
        step_ms.append({"median": max_over_ranks(statistics.median(t), world, dev),
                        "p90": max_over_ranks(p90, world, dev)})

    # ---- end to end through the public API: pinned host inputs in, results out, timed
    n_e2e = max(1, min(args.steps, args.e2e_steps))
    e2e = []
    for leg in legs:
        leg.e2e_setup()
        leg.e2e_step(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_e2e):
            leg.e2e_step(stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(a.elapsed_time(b), world, dev)
        rec = {"value": leg.rate(sum_over_ranks(leg.work * n_e2e, world, dev), ms),
               "unit": leg.unit, "h2d_bytes_per_step": leg.h2d, "d2h_bytes_per_step": leg.d2h}
        if leg.resident:
            rec["resident_bytes"] = leg.resident
            rec["resident"] = "KV cache kept on the device between steps"
        e2e.append(rec)
        leg.e2e_teardown()

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, one GPU only)
    cpu = None
    p0 = legs[0]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, el, desc, cores = cpu_oracle_sample(p0.w, p0.kind, args.cpu_seconds)
        cpu = {"value": v, "unit": p0.unit, "cores": cores, "kind": "oracle", "sample": desc}

    peaks, peak_src = load_peaks()
    roofs = [roofline(legs[i], leg_ms[i] / args.steps, peaks, peak_src) for i in range(nl)]

    if rank == 0:
        l2 = ("inputs larger than L2 (%.2f GB resident)" % (resident / 1e9) if flush is None
              else "L2 flushed between steps (%d MB buffer written)" % (flush.numel() >> 20))
        config = {"workload": " + ".join(names), "batch_override": args.batch,
                  "parallelism": "replicas" if world > 1 else "single GPU", "l2": l2}
        for leg in legs:
            config[config_key(leg.kind)] = dict(leg.shape)
        line = {
            "metric": METRIC, "value": leg_val[0], "unit": p0.unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sum(leg_ms) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("f32" if getattr(p0, "f32", False) else
                      "f16 (E4M3 cache)" if p0.kind == "decode_fp8" else
                      "f16 (INT8 cache)" if p0.kind == "decode_int8" else "bf16"),
            "data": "synthetic",
            "config": config,
            "roofline": roofs[0],
            "e2e": e2e[0],
            "cpu_baseline": cpu,
            "gpu_launches": args.steps * sum(launches_per_call(leg) for leg in legs),
            "clocks": clocks,
        }
        line["%s_ms_per_step" % ("decode" if p0.kind.startswith("decode") else "prefill")] = \
            leg_ms[0] / args.steps
        line["step_ms"] = step_ms[0]
        for i in range(1, nl):
            line[legs[i].kind] = {"value": leg_val[i], "unit": legs[i].unit,
                                  "ms_per_step": leg_ms[i] / args.steps,
                                  "step_ms": step_ms[i],
                                  "roofline": roofs[i], "e2e": e2e[i]}
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
    ap.add_argument("--workload", default=None,
                    help="bench one named workload alone (attn_fwd_07_b300.inputs.WORKLOADS) "
                         "instead of the default prefill + decode step")
    ap.add_argument("--batch", type=int, default=None,
                    help="replace the workload's batch size (sequences) with this one")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload is not None:
        from attn_fwd_07_b300 import inputs
        if args.workload not in inputs.WORKLOADS:
            ap.error("unknown workload %r; one of %s" % (args.workload,
                                                         ", ".join(inputs.WORKLOADS)))
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
