"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and lays them out; it holds none of the
attention arithmetic, and both the CUDA path and the CPU oracle receive exactly
the tensors it returns.

Recipe (fixed so that any run can regenerate the same values):

* A tensor's values are standard normals drawn in float32 in blocks of
  ``BLOCK`` consecutive elements; block ``i`` of the tensor tagged ``tag`` comes
  from ``numpy.random.default_rng([seed, tag, i])`` (PCG64 seeded through
  SeedSequence).  Blocks are independent, so they are drawn on several threads
  and the result does not depend on the thread count.
* Values are multiplied by the workload's factor in float32, then rounded to
  bf16 with round-to-nearest-even (torch's conversion) for bf16 workloads.
* Integer draws (sequence lengths, the page permutation) use
  ``default_rng([seed, tag])``; lengths are ``integers(lo, hi + 1)``.
* Paged caches hold ``sum_b ceil(len_b / page_size)`` pages.  The pages of
  sequence ``b`` are the next ``ceil(len_b / page_size)`` entries of a random
  permutation of the pool, in logical order; unused page-table slots are -1.

The five named workloads are the long-context shapes the attention pages talk
about (a single head; batched causal; long-context grouped-query causal;
packed variable-length causal; decode against a paged cache).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 1 << 22

TAG_Q, TAG_K, TAG_V, TAG_LEN, TAG_PERM, TAG_QCHUNK = 1, 2, 3, 4, 5, 6


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def normal_f32(numel: int, seed: int, tag: int, factor: float = 1.0) -> np.ndarray:
    """``numel`` float32 standard normals (times ``factor``) by the block recipe."""
    out = np.empty(numel, np.float32)
    nblk = (numel + BLOCK - 1) // BLOCK

    def fill(i):
        lo = i * BLOCK
        hi = min(numel, lo + BLOCK)
        g = np.random.default_rng([seed, tag, i])
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if factor != 1.0:
            out[lo:hi] *= np.float32(factor)

    if nblk <= 1:
        for i in range(nblk):
            fill(i)
    else:
        with ThreadPoolExecutor(max_workers=min(_threads(), nblk)) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def normal_tensor(shape, seed: int, tag: int, dtype: torch.dtype, factor: float = 1.0):
    """A CPU tensor of the given shape and dtype (bf16 rounded RNE from float32)."""
    numel = int(np.prod(shape)) if len(shape) else 1
    a = torch.from_numpy(normal_f32(numel, seed, tag, factor)).reshape(shape)
    if dtype == torch.float32:
        return a
    if dtype == torch.bfloat16:
        # convert block by block to bound the transient fp32 + bf16 footprint
        out = torch.empty(shape, dtype=torch.bfloat16)
        flat_in, flat_out = a.view(-1), out.view(-1)
        for lo in range(0, numel, 1 << 26):
            flat_out[lo:lo + (1 << 26)] = flat_in[lo:lo + (1 << 26)].to(torch.bfloat16)
        return out
    raise ValueError("unsupported dtype %r" % (dtype,))


def lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive)."""
    return np.random.default_rng([seed, TAG_LEN]).integers(lo, hi + 1, size=n).astype(np.int32)


@dataclass
class Dense:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    causal: bool
    scale: float
    window: tuple | None = None   # (left, right) extents of a sliding window, -1 = unbounded

    @property
    def shape(self):
        B, N, Hq, d = self.q.shape
        return B, N, Hq, self.k.shape[2], d


def dense(B, N, Hq, Hkv, d, seed, dtype=torch.bfloat16, factor=1.0, causal=True,
          scale=None) -> Dense:
    """q [B,N,Hq,d], k/v [B,N,Hkv,d] in the [batch, token, head, dim] layout."""
    q = normal_tensor((B, N, Hq, d), seed, TAG_Q, dtype, factor)
    k = normal_tensor((B, N, Hkv, d), seed, TAG_K, dtype, factor)
    v = normal_tensor((B, N, Hkv, d), seed, TAG_V, dtype, factor)
    return Dense(q, k, v, causal, (1.0 / math.sqrt(d)) if scale is None else scale)


@dataclass
class Varlen:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens: torch.Tensor  # int32 [S+1]
    causal: bool
    scale: float

    @property
    def lens(self):
        cu = self.cu_seqlens.numpy()
        return (cu[1:] - cu[:-1]).astype(np.int64)


def varlen(lens, Hq, Hkv, d, seed, dtype=torch.bfloat16, factor=1.0, causal=True,
           scale=None) -> Varlen:
    """Sequences of the given lengths packed along the token axis: q [T,Hq,d]."""
    lens = np.asarray(lens, np.int64)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    q = normal_tensor((T, Hq, d), seed, TAG_Q, dtype, factor)
    k = normal_tensor((T, Hkv, d), seed, TAG_K, dtype, factor)
    v = normal_tensor((T, Hkv, d), seed, TAG_V, dtype, factor)
    return Varlen(q, k, v, torch.from_numpy(cu), causal,
                  (1.0 / math.sqrt(d)) if scale is None else scale)


@dataclass
class Paged:
    q: torch.Tensor           # [B, Hq, d]
    k_cache: torch.Tensor     # [P, page_size, Hkv, d]
    v_cache: torch.Tensor
    page_table: torch.Tensor  # int32 [B, maxp], -1 past each sequence's pages
    seq_lens: torch.Tensor    # int32 [B]
    scale: float

    @property
    def page_size(self):
        return self.k_cache.shape[1]


def paged(lens, Hq, Hkv, d, seed, page_size=16, max_pages=None, dtype=torch.bfloat16,
          factor=1.0, scale=None) -> Paged:
    lens = np.asarray(lens, np.int64)
    B = len(lens)
    npages = (lens + page_size - 1) // page_size
    pool = int(npages.sum())
    maxp = int(npages.max()) if max_pages is None else int(max_pages)
    assert maxp >= int(npages.max())
    perm = np.random.default_rng([seed, TAG_PERM]).permutation(pool).astype(np.int32)
    table = np.full((B, maxp), -1, np.int32)
    off = 0
    for b in range(B):
        table[b, :npages[b]] = perm[off:off + npages[b]]
        off += npages[b]
    q = normal_tensor((B, Hq, d), seed, TAG_Q, dtype, factor)
    kc = normal_tensor((pool, page_size, Hkv, d), seed, TAG_K, dtype, factor)
    vc = normal_tensor((pool, page_size, Hkv, d), seed, TAG_V, dtype, factor)
    return Paged(q, kc, vc, torch.from_numpy(table), torch.from_numpy(lens.astype(np.int32)),
                 (1.0 / math.sqrt(d)) if scale is None else scale)


@dataclass
class ChunkPaged:
    q: torch.Tensor           # [Tq, Hq, d] bf16: each sequence's chunk of new queries
    k_cache: torch.Tensor     # [P, page_size, Hkv, d] bf16
    v_cache: torch.Tensor
    page_table: torch.Tensor  # int32 [B, maxp]
    seq_lens: torch.Tensor    # int32 [B]: cached tokens, the chunk's own included
    cu_seqlens_q: torch.Tensor  # int32 [B + 1]
    causal: bool
    scale: float

    @property
    def q_lens(self):
        cu = self.cu_seqlens_q.numpy()
        return (cu[1:] - cu[:-1]).astype(np.int64)


def chunked(ctx_lens, q_lens, Hq, Hkv, d, seed, page_size=16, factor=1.0, causal=True,
            scale=None) -> ChunkPaged:
    """Paged caches of ctx_lens tokens (the paged recipe) and, per sequence, a chunk of
    q_lens new queries packed along the token axis (the chunk's tokens are the last
    q_len of the cache)."""
    ctx = np.asarray(ctx_lens, np.int64)
    ql = np.asarray(q_lens, np.int64)
    assert (ql <= ctx).all() and (ql >= 0).all()
    cache = paged(ctx, Hq, Hkv, d, seed, page_size=page_size, factor=factor)
    cu = np.zeros(len(ql) + 1, np.int32)
    cu[1:] = np.cumsum(ql)
    q = normal_tensor((int(cu[-1]), Hq, d), seed, TAG_QCHUNK, torch.bfloat16, factor)
    return ChunkPaged(q, cache.k_cache, cache.v_cache, cache.page_table, cache.seq_lens,
                      torch.from_numpy(cu), causal,
                      (1.0 / math.sqrt(d)) if scale is None else scale)


@dataclass
class PagedFP8:
    q: torch.Tensor           # [B, Hq, d] bf16
    k_cache: torch.Tensor     # [P, page_size, Hkv, d] uint8 (FP8 E4M3 bytes) or int8
    v_cache: torch.Tensor
    k_scale: torch.Tensor     # [Hkv] float32: element c of head g stands for scale[g] *
                              # e4m3 (or * int8)
    v_scale: torch.Tensor
    page_table: torch.Tensor  # int32 [B, maxp]
    seq_lens: torch.Tensor    # int32 [B]
    scale: float


def _to_e4m3(x: torch.Tensor):
    """float32 [P, ps, Hkv, d] -> (E4M3 bytes, per-head float32 scales) with each head's
    largest magnitude mapped to 448, the largest E4M3 value (torch's float8_e4m3fn cast,
    round to nearest even)."""
    amax = x.abs().amax(dim=(0, 1, 3)).clamp_min(1e-30)
    sc = (amax / 448.0).to(torch.float32)
    q8 = (x / sc.view(1, 1, -1, 1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8).contiguous(), sc


def _to_int8(x: torch.Tensor):
    """float32 [P, ps, Hkv, d] -> (int8 values, per-head float32 scales) with each head's
    largest magnitude mapped to 127 (symmetric: round to nearest even, -127 .. 127)."""
    amax = x.abs().amax(dim=(0, 1, 3)).clamp_min(1e-30)
    sc = (amax / 127.0).to(torch.float32)
    q8 = torch.round(x / sc.view(1, 1, -1, 1)).clamp(-127.0, 127.0).to(torch.int8)
    return q8.contiguous(), sc


def _paged_bytes(lens, Hq, Hkv, d, seed, page_size, max_pages, factor, scale, quantise):
    lens = np.asarray(lens, np.int64)
    B = len(lens)
    npages = (lens + page_size - 1) // page_size
    pool = int(npages.sum())
    maxp = int(npages.max()) if max_pages is None else int(max_pages)
    assert maxp >= int(npages.max())
    perm = np.random.default_rng([seed, TAG_PERM]).permutation(pool).astype(np.int32)
    table = np.full((B, maxp), -1, np.int32)
    off = 0
    for b in range(B):
        table[b, :npages[b]] = perm[off:off + npages[b]]
        off += npages[b]
    q = normal_tensor((B, Hq, d), seed, TAG_Q, torch.bfloat16, factor)
    kc, ks = quantise(normal_tensor((pool, page_size, Hkv, d), seed, TAG_K, torch.float32,
                                    factor))
    vc, vs = quantise(normal_tensor((pool, page_size, Hkv, d), seed, TAG_V, torch.float32,
                                    factor))
    return (q, kc, vc, ks, vs, torch.from_numpy(table), torch.from_numpy(lens.astype(np.int32)),
            (1.0 / math.sqrt(d)) if scale is None else scale)


def paged_fp8(lens, Hq, Hkv, d, seed, page_size=16, max_pages=None, factor=1.0,
              scale=None) -> PagedFP8:
    """The paged recipe above with the cache held as FP8 E4M3 bytes and one scale per
    key/value head for K and for V: the same float32 draws, divided by the head's scale
    and rounded to E4M3 (as a cache writer that quantises on append would)."""
    return PagedFP8(*_paged_bytes(lens, Hq, Hkv, d, seed, page_size, max_pages, factor, scale,
                                  _to_e4m3))


def paged_int8(lens, Hq, Hkv, d, seed, page_size=16, max_pages=None, factor=1.0,
               scale=None) -> PagedFP8:
    """The same recipe with the cache held as INT8 (k_cache / v_cache torch.int8) and one
    scale per key/value head for K and for V: the float32 draws divided by the head's
    scale and rounded to the nearest integer in -127 .. 127."""
    return PagedFP8(*_paged_bytes(lens, Hq, Hkv, d, seed, page_size, max_pages, factor, scale,
                                  _to_int8))


@dataclass
class Workload:
    name: str
    kind: str                 # "dense" | "varlen" | "decode"
    seed: int
    params: dict = field(default_factory=dict)
    description: str = ""


# The workloads: seed = index (the five listed first, then the sliding-window one).
WORKLOADS = {
    "single_head_f32": Workload(
        "single_head_f32", "dense", 1,
        dict(B=1, N=256, Hq=1, Hkv=1, d=64, dtype=torch.float32, factor=1.0, causal=False),
        "B=1 H=1 N=256 d=64, fp32 N(0,1), non-causal, scale 1/8"),
    "batched_causal_b4h16n2048": Workload(
        "batched_causal_b4h16n2048", "dense", 2,
        dict(B=4, N=2048, Hq=16, Hkv=16, d=128, dtype=torch.bfloat16, factor=1.0, causal=True),
        "B=4 H=16 N=2048 d=128, bf16 N(0,1), causal, [B,N,H,d]"),
    "gqa_causal_n16384": Workload(
        "gqa_causal_n16384", "dense", 3,
        dict(B=1, N=16384, Hq=32, Hkv=8, d=128, dtype=torch.bfloat16, factor=0.5, causal=True),
        "B=1 Hq=32 Hkv=8 N=16384 d=128, bf16 N(0,1)*0.5, causal"),
    "varlen_causal_8seq": Workload(
        "varlen_causal_8seq", "varlen", 4,
        dict(S=8, lo=512, hi=8192, Hq=32, Hkv=8, d=128, dtype=torch.bfloat16, factor=1.0,
             causal=True),
        "8 packed sequences, lengths U[512,8192], Hq=32 Hkv=8 d=128, bf16 N(0,1), causal"),
    # the long-context GQA workload computed in the two-pass order (statistics, then
    # output): same inputs as gqa_causal_n16384
    "gqa_causal_n16384_two_pass": Workload(
        "gqa_causal_n16384_two_pass", "two_pass", 3,
        dict(B=1, N=16384, Hq=32, Hkv=8, d=128, dtype=torch.bfloat16, factor=0.5, causal=True),
        "B=1 Hq=32 Hkv=8 N=16384 d=128, bf16 N(0,1)*0.5, causal, two-pass order"),
    # local attention as the sliding-window glossary entry describes it: w/2 keys on
    # either side of each token, here w = 4096 on an 8192-token sequence (the length
    # the entry uses to count full attention's ~67 million pairs)
    "swa_n8192_w4096": Workload(
        "swa_n8192_w4096", "window", 6,
        dict(B=1, N=8192, Hq=32, Hkv=8, d=128, dtype=torch.bfloat16, factor=1.0,
             window=(2048, 2048)),
        "B=1 Hq=32 Hkv=8 N=8192 d=128, bf16 N(0,1), sliding window of 2048 keys left and right"),
    # the decode workload with the cache quantised to FP8 E4M3 (one scale per key/value
    # head), the INT8/FP8 cache the KV-cache glossary entry mentions
    "decode_paged_fp8_b64": Workload(
        "decode_paged_fp8_b64", "decode_fp8", 5,
        dict(B=64, lo=1024, hi=32768, Hq=32, Hkv=8, d=128, page_size=16, factor=1.0),
        "B=64 one query each, lengths U[1024,32768], Hq=32 Hkv=8 d=128, 16-token pages, "
        "permuted page table, N(0,1) cache quantised to FP8 E4M3 with per-head scales"),
    # the decode workload with the cache quantised to INT8 (one scale per key/value
    # head), the other format the KV-cache glossary entry names
    "decode_paged_int8_b64": Workload(
        "decode_paged_int8_b64", "decode_int8", 5,
        dict(B=64, lo=1024, hi=32768, Hq=32, Hkv=8, d=128, page_size=16, factor=1.0),
        "B=64 one query each, lengths U[1024,32768], Hq=32 Hkv=8 d=128, 16-token pages, "
        "permuted page table, N(0,1) cache quantised to INT8 with per-head scales"),
    # chunked prefill with prefix caching: 8 sequences whose cached prefixes are
    # U[1024, 16384] tokens each receive a chunk of 2048 new tokens, which attend
    # causally to the prefix and to themselves through the page table
    "chunked_prefill_b8": Workload(
        "chunked_prefill_b8", "chunk", 7,
        dict(B=8, lo=1024, hi=16384, chunk=2048, Hq=32, Hkv=8, d=128, page_size=16,
             factor=1.0),
        "8 sequences, cached prefixes U[1024,16384] + a 2048-token chunk each, Hq=32 Hkv=8 "
        "d=128, 16-token pages, permuted page table, bf16 N(0,1), causal"),
    "decode_paged_b64": Workload(
        "decode_paged_b64", "decode", 5,
        dict(B=64, lo=1024, hi=32768, Hq=32, Hkv=8, d=128, page_size=16,
             dtype=torch.bfloat16, factor=1.0),
        "B=64 one query each, lengths U[1024,32768], Hq=32 Hkv=8 d=128, 16-token pages, "
        "permuted page table, bf16 N(0,1)"),
}


def make(name: str, batch: int | None = None):
    """Generate the named workload's inputs (CPU tensors).

    ``batch`` replaces the workload's batch size (sequences, for the packed and
    paged workloads) with the same recipe otherwise; None keeps it."""
    w = WORKLOADS[name]
    p = w.params
    if w.kind in ("dense", "two_pass"):
        B = p["B"] if batch is None else int(batch)
        return dense(B, p["N"], p["Hq"], p["Hkv"], p["d"], w.seed, p["dtype"], p["factor"],
                     p["causal"])
    if w.kind == "window":
        B = p["B"] if batch is None else int(batch)
        out = dense(B, p["N"], p["Hq"], p["Hkv"], p["d"], w.seed, p["dtype"], p["factor"],
                    causal=False)
        out.window = tuple(p["window"])
        return out
    if w.kind == "varlen":
        S = p["S"] if batch is None else int(batch)
        lens = lengths(S, p["lo"], p["hi"], w.seed)
        return varlen(lens, p["Hq"], p["Hkv"], p["d"], w.seed, p["dtype"], p["factor"],
                      p["causal"])
    if w.kind == "decode":
        B = p["B"] if batch is None else int(batch)
        lens = lengths(B, p["lo"], p["hi"], w.seed)
        maxp = (p["hi"] + p["page_size"] - 1) // p["page_size"]
        return paged(lens, p["Hq"], p["Hkv"], p["d"], w.seed, p["page_size"], maxp, p["dtype"],
                     p["factor"])
    if w.kind == "chunk":
        B = p["B"] if batch is None else int(batch)
        prefix = lengths(B, p["lo"], p["hi"], w.seed)
        ql = np.full(B, p["chunk"], np.int64)
        return chunked(prefix + ql, ql, p["Hq"], p["Hkv"], p["d"], w.seed, p["page_size"],
                       p["factor"])
    if w.kind in ("decode_fp8", "decode_int8"):
        B = p["B"] if batch is None else int(batch)
        lens = lengths(B, p["lo"], p["hi"], w.seed)
        maxp = (p["hi"] + p["page_size"] - 1) // p["page_size"]
        gen = paged_fp8 if w.kind == "decode_fp8" else paged_int8
        return gen(lens, p["Hq"], p["Hkv"], p["d"], w.seed, p["page_size"], maxp, p["factor"])
    raise ValueError(w.kind)
