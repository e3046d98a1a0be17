"""fp64 CPU oracle for exact scaled-dot-product attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product library never does, and the
two share no code: this module loads ``liboracle.so`` (built from
``attn_oracle.c`` with gcc) through ctypes and hands it numpy arrays.

The arithmetic lives in ``attn_oracle.c``; its header states the definition it
follows ("Donanıma Duyarlı Algoritma Tasarımı: FlashAttention", section
"Transformer Mimarisi ve Self-Attention Mekanizması", the attention formula)
and the pins that check it live in ``tests/test_oracle_pins.py``.

Every function takes fp32 numpy arrays (bf16 values upcast exactly) and returns
fp64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        D = ctypes.c_double
        lib.oracle_attn_rows.argtypes = [P, P, P, I, I, I, I, I, I, I, D, P, I64, P, P, I]
        lib.oracle_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, D, I]
        lib.oracle_attn_window_rows.argtypes = [P, P, P, I, I, I, I, I, I, I, D, P, I64, P, P,
                                                I]
        lib.oracle_attn_varlen.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, D, I]
        lib.oracle_decode_paged_rows.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, D,
                                                 P, I, P, P, I]
        lib.oracle_decode_paged_window_rows.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I,
                                                        D, P, I, P, P, I]
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = D
        lib.oracle_decode_paged_fp8_rows.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, D,
                                                     P, I, P, P, I]
        lib.oracle_int8_value.argtypes = [ctypes.c_uint8]
        lib.oracle_int8_value.restype = D
        lib.oracle_decode_paged_int8_rows.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                                      D, P, I, P, P, I]
        lib.oracle_chunk_paged_rows.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I,
                                                D, P, I64, P, P, I]
        lib.oracle_online_softmax_stats.argtypes = [P, I64, I64, P, P]
        lib.oracle_online_softmax_stats.restype = None
        lib.oracle_merge_parts.argtypes = [P, P, I, I, P, P]
        lib.oracle_merge_parts.restype = None
        lib.oracle_max_threads.argtypes = []
        for name in ("oracle_attn_rows", "oracle_attn_fwd", "oracle_attn_varlen",
                     "oracle_attn_window_rows", "oracle_decode_paged_window_rows",
                     "oracle_decode_paged_fp8_rows", "oracle_decode_paged_int8_rows",
                     "oracle_chunk_paged_rows",
                     "oracle_decode_paged_rows", "oracle_max_threads"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def attn_fwd(q, k, v, causal: bool, scale: float, nthreads: int = 0):
    """Full dense attention.  q [B,N,Hq,d], k/v [B,N,Hkv,d] -> (o [B,N,Hq,d], lse [B,Hq,N])."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, N, Hkv, d) and v.shape == k.shape
    o = np.zeros((B, N, Hq, d), np.float64)
    lse = np.zeros((B, Hq, N), np.float64)
    rc = _load().oracle_attn_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, Hq, Hkv, N, d,
                                 int(bool(causal)), float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def attn_rows(q, k, v, rows, causal: bool, scale: float, nthreads: int = 0):
    """Dense attention for selected rows.  rows: int array [n, 3] of (b, h, i).

    q [B,Nq,Hq,d], k/v [B,Nk,Hkv,d] -> (o [n, d], lse [n]).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    assert k.shape == (B, Nk, Hkv, d) and v.shape == k.shape
    rows = _i32(rows).reshape(-1, 3)
    n = rows.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_attn_rows(_p(q), _p(k), _p(v), B, Hq, Hkv, Nq, Nk, d,
                                  int(bool(causal)), float(scale), _p(rows), n,
                                  _p(o), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    return o, lse


def attn_window_rows(q, k, v, rows, window_left: int, window_right: int, scale: float,
                     nthreads: int = 0):
    """Sliding-window attention for selected rows (b, h, i): query i sees keys
    i - window_left .. i + window_right (a negative extent: no limit on that side).
    q [B,N,Hq,d], k/v [B,N,Hkv,d] -> (o [n, d], lse [n])."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, N, Hkv, d) and v.shape == k.shape
    rows = _i32(rows).reshape(-1, 3)
    n = rows.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_attn_window_rows(_p(q), _p(k), _p(v), B, Hq, Hkv, N, d,
                                         int(window_left), int(window_right), float(scale),
                                         _p(rows), n, _p(o), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_window_rows rejected its arguments")
    return o, lse


def attn_window(q, k, v, window_left: int, window_right: int, scale: float,
                nthreads: int = 0):
    """Sliding-window attention for every row -> (o [B,N,Hq,d], lse [B,Hq,N])."""
    B, N, Hq, d = np.shape(q)
    b, h, i = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(N), indexing="ij")
    rows = np.stack([b.ravel(), h.ravel(), i.ravel()], 1)
    o, lse = attn_window_rows(q, k, v, rows, window_left, window_right, scale, nthreads)
    return (o.reshape(B, Hq, N, d).transpose(0, 2, 1, 3).copy(), lse.reshape(B, Hq, N))


def attn_varlen(q, k, v, cu_seqlens, causal: bool, scale: float, nthreads: int = 0):
    """Packed variable-length attention.  q [T,Hq,d], k/v [T,Hkv,d], cu_seqlens [S+1]

    -> (o [T,Hq,d], lse [Hq,T]).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    cu = _i32(cu_seqlens)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    o = np.zeros((T, Hq, d), np.float64)
    lse = np.zeros((Hq, T), np.float64)
    rc = _load().oracle_attn_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu),
                                    cu.shape[0] - 1, T, Hq, Hkv, d, int(bool(causal)),
                                    float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_varlen rejected its arguments")
    return o, lse


def decode_paged(q, k_cache, v_cache, page_table, seq_lens, scale: float, seqs=None,
                 nthreads: int = 0):
    """Decode of one new query per sequence against a paged cache.

    q [B,Hq,d]; k_cache/v_cache [P,page_size,Hkv,d]; page_table [B,maxp]; seq_lens [B].
    seqs: the sequences to compute (default all) -> (o [len(seqs),Hq,d], lse [len(seqs),Hq]).
    """
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    pt, sl = _i32(page_table), _i32(seq_lens)
    B, Hq, d = q.shape
    P, ps, Hkv, _ = kc.shape
    maxp = pt.shape[1]
    seqs = _i32(np.arange(B) if seqs is None else seqs)
    n = seqs.shape[0]
    o = np.zeros((n, Hq, d), np.float64)
    lse = np.zeros((n, Hq), np.float64)
    rc = _load().oracle_decode_paged_rows(_p(q), _p(kc), _p(vc), _p(pt), _p(sl), B, Hq, Hkv,
                                          d, ps, P, maxp, float(scale), _p(seqs), n,
                                          _p(o), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_paged_rows rejected its arguments")
    return o, lse


def decode_paged_window(q, k_cache, v_cache, page_table, seq_lens, window: int, scale: float,
                        seqs=None, nthreads: int = 0):
    """Decode where the query of sequence b sees only its last window + 1 cached tokens
    (window < 0: all).  Arguments and results as decode_paged."""
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    pt, sl = _i32(page_table), _i32(seq_lens)
    B, Hq, d = q.shape
    P, ps, Hkv, _ = kc.shape
    maxp = pt.shape[1]
    seqs = _i32(np.arange(B) if seqs is None else seqs)
    n = seqs.shape[0]
    o = np.zeros((n, Hq, d), np.float64)
    lse = np.zeros((n, Hq), np.float64)
    rc = _load().oracle_decode_paged_window_rows(_p(q), _p(kc), _p(vc), _p(pt), _p(sl), B, Hq,
                                                 Hkv, d, ps, P, maxp, int(window), float(scale),
                                                 _p(seqs), n, _p(o), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode_paged_window_rows rejected its arguments")
    return o, lse


def chunk_paged_rows(q, k_cache, v_cache, page_table, seq_lens, cu_seqlens_q, causal: bool,
                     scale: float, rows=None, nthreads: int = 0):
    """A chunk of queries per sequence against its paged cache: q [Tq,Hq,d] packed by
    cu_seqlens_q; sequence s has seq_lens[s] cached tokens, the last q_len of them the
    chunk's own, so query i sits at position seq_lens[s] - q_len + i (causal: it sees
    positions <= its own).  rows: [n, 2] (token, head) pairs, default all ->
    (o [n, d], lse [n])."""
    q, kc, vc = _f32(q), _f32(k_cache), _f32(v_cache)
    pt, sl, cu = _i32(page_table), _i32(seq_lens), _i32(cu_seqlens_q)
    Tq, Hq, d = q.shape
    P, ps, Hkv, _ = kc.shape
    maxp = pt.shape[1]
    if rows is None:
        t, h = np.meshgrid(np.arange(Tq), np.arange(Hq), indexing="ij")
        rows = np.stack([t.ravel(), h.ravel()], 1)
    rows = _i32(rows).reshape(-1, 2)
    n = rows.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_chunk_paged_rows(_p(q), _p(kc), _p(vc), _p(pt), _p(sl), _p(cu),
                                         len(cu) - 1, Tq, Hq, Hkv, d, ps, P, maxp,
                                         int(bool(causal)), float(scale), _p(rows), n, _p(o),
                                         _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_chunk_paged_rows rejected its arguments")
    return o, lse


def e4m3_value(byte: int) -> float:
    """The value of one FP8 E4M3 (E4M3FN) byte, from its bit fields."""
    return float(_load().oracle_e4m3_value(int(byte) & 0xFF))


def _bytes(x):
    """A one-byte cache as uint8: int8 arrays keep their bytes, others are cast."""
    a = np.asarray(x)
    if a.dtype == np.int8:
        return np.ascontiguousarray(a).view(np.uint8)
    return np.ascontiguousarray(a, dtype=np.uint8)


def _decode_paged_bytes(fn, name, q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                        scale, seqs, nthreads):
    q = _f32(q)
    kc, vc = _bytes(k_cache), _bytes(v_cache)
    ks, vs = _f32(k_scale), _f32(v_scale)
    pt, sl = _i32(page_table), _i32(seq_lens)
    B, Hq, d = q.shape
    P, ps, Hkv, _ = kc.shape
    assert vc.shape == kc.shape and ks.shape == (Hkv,) and vs.shape == (Hkv,)
    maxp = pt.shape[1]
    seqs = _i32(np.arange(B) if seqs is None else seqs)
    n = seqs.shape[0]
    o = np.zeros((n, Hq, d), np.float64)
    lse = np.zeros((n, Hq), np.float64)
    rc = fn(_p(q), _p(kc), _p(vc), _p(ks), _p(vs), _p(pt), _p(sl), B, Hq, Hkv, d, ps, P, maxp,
            float(scale), _p(seqs), n, _p(o), _p(lse), int(nthreads))
    if rc != 0:
        raise ValueError(name + " rejected its arguments")
    return o, lse


def decode_paged_fp8(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                     scale: float, seqs=None, nthreads: int = 0):
    """Decode against an FP8 E4M3 paged cache: k_cache/v_cache uint8 [P,page_size,Hkv,d]
    (E4M3 bytes), k_scale/v_scale [Hkv] (element c of head g stands for scale[g] *
    e4m3(byte)).  Other arguments and results as decode_paged."""
    return _decode_paged_bytes(_load().oracle_decode_paged_fp8_rows,
                               "oracle_decode_paged_fp8_rows", q, k_cache, v_cache, k_scale,
                               v_scale, page_table, seq_lens, scale, seqs, nthreads)


def int8_value(byte: int) -> float:
    """The value of one INT8 byte (two's complement)."""
    return float(_load().oracle_int8_value(int(byte) & 0xFF))


def decode_paged_int8(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                      scale: float, seqs=None, nthreads: int = 0):
    """Decode against an INT8 paged cache: k_cache/v_cache int8 (or their bytes as uint8)
    [P,page_size,Hkv,d], k_scale/v_scale [Hkv] (element c of head g stands for scale[g] *
    int8).  Other arguments and results as decode_paged."""
    return _decode_paged_bytes(_load().oracle_decode_paged_int8_rows,
                               "oracle_decode_paged_int8_rows", q, k_cache, v_cache, k_scale,
                               v_scale, page_table, seq_lens, scale, seqs, nthreads)


def online_softmax_stats(x, block: int):
    """The online (M, L) recurrence over a row in blocks -> (M, L) with L = sum exp(x - M)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    M = np.zeros(1, np.float64)
    L = np.zeros(1, np.float64)
    _load().oracle_online_softmax_stats(_p(x), x.shape[0], int(block), _p(M), _p(L))
    return float(M[0]), float(L[0])


def merge_parts(o_parts, lse_parts):
    """Combine per-key-subset (o_s, lse_s) into attention over all the keys."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.zeros(d, np.float64)
    lse = np.zeros(1, np.float64)
    _load().oracle_merge_parts(_p(o_parts), _p(lse_parts), n, d, _p(o), _p(lse))
    return o, float(lse[0])
