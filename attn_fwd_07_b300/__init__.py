"""attn_fwd_07_b300 -- exact FlashAttention-style attention for B300 (sm_103a).

Python binding of ``libattn07.so`` (C ABI in ``include/attn07.h``).  The
functions here have the C entry points' names and only marshal arguments:
they read shapes from torch tensors, allocate outputs when none are given, and
pass device pointers and the current CUDA stream to the library.  Every step of
the computation runs in the library's CUDA kernels; there is no other path.
If the library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "AttnError", "load_library", "attn_fwd", "attn_fwd_window", "attn_fwd_chunked_paged",
    "attn_fwd_two_pass",
    "attn_fwd_f32",
    "attn_fwd_varlen", "attn_decode_paged", "attn_decode_paged_window", "attn_decode_paged_fp8",
    "attn_decode_paged_int8",
    "attn_decode_paged_noalloc", "attn_decode_workspace_size", "attn_status_string",
    "attn_get_device_status", "attn_version", "attn_last_cuda_error",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn07.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_DEVICE_BOUNDS = 5

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        msg = "%s: %s (status %d)" % (where, attn_status_string(code), code)
        if self.code == ATTN_ERR_CUDA:
            msg += " [%s]" % attn_last_cuda_error()
        super().__init__(msg)


def load_library(path: str = LIB_PATH):
    """Load libattn07.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise OSError("libattn07.so not found at %s; build it with "
                          "`python -m attn_fwd_07_b300.build`" % path)
        lib = ctypes.CDLL(path)
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.attn_fwd_host.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.attn_release_host_staging.argtypes = []
        lib.attn_selftest_wait_timeout.argtypes = [P, P]
        lib.attn_fwd_f32.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.attn_fwd_window.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.attn_fwd_varlen.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, P]
        lib.attn_decode_paged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, SZ, P]
        lib.attn_fwd_two_pass.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
        lib.attn_fwd_chunked_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I,
                                               I, I, F, P]
        lib.attn_decode_paged_fp8.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F,
                                              P, SZ, P]
        lib.attn_decode_paged_int8.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F,
                                               P, SZ, P]
        lib.attn_decode_paged_window.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F,
                                                 P, SZ, P]
        lib.attn_decode_paged_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F,
                                                  P]
        lib.attn_decode_workspace_size.argtypes = [I, I, I, I, I]
        lib.attn_decode_workspace_size.restype = SZ
        lib.attn_status_string.argtypes = [I]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_get_device_status.argtypes = [P]
        lib.attn_version.argtypes = []
        lib.attn_version.restype = ctypes.c_char_p
        lib.attn_last_cuda_error.argtypes = []
        lib.attn_last_cuda_error.restype = ctypes.c_char_p
        for name in ("attn_fwd", "attn_fwd_f32", "attn_fwd_varlen", "attn_decode_paged",
                     "attn_fwd_window", "attn_decode_paged_window", "attn_decode_paged_fp8",
                     "attn_decode_paged_int8",
                     "attn_fwd_chunked_paged", "attn_fwd_two_pass",
                     "attn_decode_paged_noalloc", "attn_get_device_status", "attn_fwd_host",
                     "attn_release_host_staging", "attn_selftest_wait_timeout"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def attn_status_string(code: int) -> str:
    return load_library().attn_status_string(int(code)).decode()


def attn_version() -> str:
    return load_library().attn_version().decode()


def attn_last_cuda_error() -> str:
    """Text of the last CUDA failure behind an ATTN_ERR_CUDA on this thread."""
    return load_library().attn_last_cuda_error().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, where):
    if code != ATTN_OK:
        raise AttnError(code, where)


def _need(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))


def attn_fwd(q, k, v, causal: bool = True, scale: float | None = None, o=None, lse=None,
             want_lse: bool = True, stream=None):
    """bf16 prefill.  q [B,N,Hq,d], k/v [B,N,Hkv,d] -> (o [B,N,Hq,d] bf16, lse [B,Hq,N] fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [B, N, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    rc = load_library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N,
                                 d, int(bool(causal)), float(scale), _stream(stream))
    _check(rc, "attn_fwd")
    return o, lse


def attn_fwd_host(q, k, v, causal: bool = True, scale: float | None = None, o=None, lse=None,
                  want_lse: bool = True, stream=None):
    """attn_fwd on HOST tensors: q [B,N,Hq,d], k/v [B,N,Hkv,d] bf16 CPU tensors (page-locked
    for overlapped copies) -> (o, lse) CPU tensors, complete on return.  The library copies
    them through a device staging area, overlapping the copies with the compute."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not (t.device.type == "cpu" and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError("%s must be a contiguous CPU bfloat16 tensor" % n)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [B, N, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q.is_pinned()
    if o is None:
        o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=pin)
    for t, n, dt in ((o, "o", torch.bfloat16), (lse, "lse", torch.float32)):
        if t is not None and not (t.device.type == "cpu" and t.dtype == dt and t.is_contiguous()):
            raise ValueError("%s must be a contiguous CPU %s tensor" % (n, dt))
    rc = load_library().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                      N, d, int(bool(causal)), float(scale), _stream(stream))
    _check(rc, "attn_fwd_host")
    return o, lse


def attn_selftest_wait_timeout(stream=None):
    """Run the device check of the pipeline-wait bound (about 2 s); returns the two
    waits' elapsed nanoseconds.  Afterwards attn_get_device_status() reports the
    timeout once."""
    out = (ctypes.c_ulonglong * 2)()
    _check(load_library().attn_selftest_wait_timeout(ctypes.cast(out, ctypes.c_void_p),
                                                     _stream(stream)),
           "attn_selftest_wait_timeout")
    return int(out[0]), int(out[1])


def attn_release_host_staging():
    """Free the device staging area that attn_fwd_host keeps between calls."""
    _check(load_library().attn_release_host_staging(), "attn_release_host_staging")


def attn_fwd_window(q, k, v, window_left: int, window_right: int, scale: float | None = None,
                    o=None, lse=None, want_lse: bool = True, stream=None):
    """bf16 sliding-window prefill: query i sees keys i - window_left .. i + window_right
    (-1: unbounded side).  Layouts as attn_fwd."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [B, N, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    rc = load_library().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq,
                                        Hkv, N, d, int(window_left), int(window_right),
                                        float(scale), _stream(stream))
    _check(rc, "attn_fwd_window")
    return o, lse


def attn_fwd_f32(q, k, v, causal: bool = True, scale: float | None = None, o=None, lse=None,
                 want_lse: bool = True, stream=None):
    """fp32 prefill, same layouts as attn_fwd."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.float32, n)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [B, N, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    rc = load_library().attn_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                     N, d, int(bool(causal)), float(scale), _stream(stream))
    _check(rc, "attn_fwd_f32")
    return o, lse


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = True,
                    scale: float | None = None, o=None, lse=None, want_lse: bool = True,
                    stream=None):
    """Packed prefill.  q [T,Hq,d], k/v [T,Hkv,d], cu_seqlens int32 [S+1] on the device

    -> (o [T,Hq,d] bf16, lse [Hq,T] fp32).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [T, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    rc = load_library().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                        _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                        int(max_seqlen), Hq, Hkv, d, int(bool(causal)),
                                        float(scale), _stream(stream))
    _check(rc, "attn_fwd_varlen")
    return o, lse


def attn_fwd_two_pass(q, k, v, causal: bool = True, scale: float | None = None, o=None,
                      lse=None, stream=None):
    """attn_fwd in the two-pass order (row statistics first, then the output); lse is
    always produced (it carries the statistics between the passes)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k/v must be [B, N, Hkv, d] matching q")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    rc = load_library().attn_fwd_two_pass(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq,
                                          Hkv, N, d, int(bool(causal)), float(scale),
                                          _stream(stream))
    _check(rc, "attn_fwd_two_pass")
    return o, lse


def attn_fwd_chunked_paged(q, k_cache, v_cache, page_table, seq_lens, cu_seqlens_q,
                           max_qlen: int, causal: bool = True, scale: float | None = None,
                           o=None, lse=None, want_lse: bool = True, stream=None):
    """A chunk of queries per sequence against its paged cache.  q [Tq,Hq,d] packed by
    cu_seqlens_q (int32 [S+1], device); caches [P,16,Hkv,d]; page_table int32 [S,maxp];
    seq_lens int32 [S] (device, the chunk's own tokens included)
    -> (o [Tq,Hq,d] bf16, lse [Hq,Tq] fp32)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    for t, n in ((page_table, "page_table"), (seq_lens, "seq_lens"),
                 (cu_seqlens_q, "cu_seqlens_q")):
        _need(t, torch.int32, n)
    Tq, Hq, d = q.shape
    P, ps, Hkv, _ = k_cache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((Hq, Tq), dtype=torch.float32, device=q.device)
    rc = load_library().attn_fwd_chunked_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seq_lens),
        _ptr(cu_seqlens_q), _ptr(o), _ptr(lse), cu_seqlens_q.numel() - 1, Tq, int(max_qlen), Hq,
        Hkv, d, ps, P, page_table.shape[1], int(bool(causal)), float(scale), _stream(stream))
    _check(rc, "attn_fwd_chunked_paged")
    return o, lse


def attn_decode_workspace_size(B: int, Hq: int, d: int, max_pages_per_seq: int,
                               page_size: int) -> int:
    """Bytes of workspace attn_decode_paged (and its window / FP8 forms) needs."""
    return int(load_library().attn_decode_workspace_size(B, Hq, d, max_pages_per_seq,
                                                         page_size))


def attn_decode_paged(q, k_cache, v_cache, page_table, seq_lens, scale: float | None = None,
                      o=None, lse=None, workspace=None, want_lse: bool = True, stream=None):
    """Decode against a paged cache.  q [B,Hq,d]; caches [P,page,Hkv,d]; page_table int32
    [B,maxp]; seq_lens int32 [B] (device) -> (o [B,Hq,d] bf16, lse [B,Hq] fp32)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(page_table, torch.int32, "page_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, d = q.shape
    P, ps, Hkv, _ = k_cache.shape
    maxp = page_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_size(B, Hq, d, maxp, ps)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = load_library().attn_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                          _ptr(seq_lens), _ptr(o), _ptr(lse), B, Hq, Hkv, d, ps, P,
                                          maxp, float(scale), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _stream(stream))
    _check(rc, "attn_decode_paged")
    return o, lse


def _decode_paged_bytes(entry, name, cache_dtype, q, k_cache, v_cache, k_scale, v_scale,
                        page_table, seq_lens, scale, o, lse, workspace, want_lse, stream):
    _need(q, torch.bfloat16, "q")
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, cache_dtype, n)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, torch.float32, n)
    _need(page_table, torch.int32, "page_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, d = q.shape
    P, ps, Hkv, _ = k_cache.shape
    maxp = page_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_size(B, Hq, d, maxp, ps)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = entry(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(page_table),
        _ptr(seq_lens), _ptr(o), _ptr(lse), B, Hq, Hkv, d, ps, P, maxp, float(scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, name)
    return o, lse


def attn_decode_paged_fp8(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                          scale: float | None = None, o=None, lse=None, workspace=None,
                          want_lse: bool = True, stream=None):
    """Decode against an FP8 E4M3 paged cache: k_cache/v_cache uint8 [P,page,Hkv,d] holding
    E4M3 bytes, k_scale/v_scale float32 [Hkv] per-head scales.  q, page_table, seq_lens and
    the results as attn_decode_paged."""
    return _decode_paged_bytes(load_library().attn_decode_paged_fp8, "attn_decode_paged_fp8",
                               torch.uint8, q, k_cache, v_cache, k_scale, v_scale, page_table,
                               seq_lens, scale, o, lse, workspace, want_lse, stream)


def attn_decode_paged_int8(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                           scale: float | None = None, o=None, lse=None, workspace=None,
                           want_lse: bool = True, stream=None):
    """Decode against an INT8 paged cache: k_cache/v_cache int8 [P,page,Hkv,d],
    k_scale/v_scale float32 [Hkv] per-head scales (element c of head g stands for
    scale[g] * int8).  q, page_table, seq_lens and the results as attn_decode_paged."""
    return _decode_paged_bytes(load_library().attn_decode_paged_int8, "attn_decode_paged_int8",
                               torch.int8, q, k_cache, v_cache, k_scale, v_scale, page_table,
                               seq_lens, scale, o, lse, workspace, want_lse, stream)


def attn_decode_paged_window(q, k_cache, v_cache, page_table, seq_lens, window: int,
                             scale: float | None = None, o=None, lse=None, workspace=None,
                             want_lse: bool = True, stream=None):
    """Decode where each query sees only the last window + 1 cached tokens of its
    sequence (-1: all of them).  Arguments and results as attn_decode_paged."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(page_table, torch.int32, "page_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, d = q.shape
    P, ps, Hkv, _ = k_cache.shape
    maxp = page_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_size(B, Hq, d, maxp, ps)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = load_library().attn_decode_paged_window(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), _ptr(seq_lens), _ptr(o),
        _ptr(lse), B, Hq, Hkv, d, ps, P, maxp, int(window), float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_decode_paged_window")
    return o, lse


def attn_decode_paged_noalloc(q, k_cache, v_cache, page_table, seq_lens,
                              scale: float | None = None, o=None, lse=None,
                              want_lse: bool = True, stream=None):
    """attn_decode_paged without a workspace, for callers that cannot allocate device
    memory (the library's built-in scratch array is used instead; calls that overlap
    on the GPU race on it).  Same arguments and results as attn_decode_paged."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(page_table, torch.int32, "page_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, d = q.shape
    P, ps, Hkv, _ = k_cache.shape
    maxp = page_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    rc = load_library().attn_decode_paged_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                  _ptr(page_table), _ptr(seq_lens), _ptr(o),
                                                  _ptr(lse), B, Hq, Hkv, d, ps, P, maxp,
                                                  float(scale), _stream(stream))
    _check(rc, "attn_decode_paged_noalloc")
    return o, lse


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load_library().attn_get_device_status(_stream(stream)))
