"""The C ABI without a GPU: the library loads, exports every function the header
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn07.h")
TEST_HEADER = os.path.join(ROOT, "include", "attn07_testing.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return A.load_library()


def declared_functions(path=HEADER):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("attn_fwd", "attn_fwd_f32", "attn_fwd_varlen", "attn_decode_paged",
                 "attn_decode_workspace_size", "attn_status_string", "attn_get_device_status"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions() + declared_functions(TEST_HEADER):
        assert hasattr(lib, name), name


def test_test_hooks_stay_out_of_the_interface():
    hooks = declared_functions(TEST_HEADER)
    assert hooks == ["attn_testing_decode_paged_ctas", "attn_testing_fwd_f32_rows"]
    assert not set(hooks) & set(declared_functions())


def test_status_strings(lib):
    for code in range(6):
        s = A.attn_status_string(code)
        assert s and s != "unknown status"
    assert A.attn_status_string(99) == "unknown status"
    assert "sm_103a" in A.attn_version()


def _fwd(lib, q=1 << 20, k=1 << 20, v=1 << 20, o=1 << 20, B=1, Hq=1, Hkv=1, N=8, d=128,
         causal=1, scale=0.1):
    P = ctypes.c_void_p
    return lib.attn_fwd(P(q) if q else None, P(k) if k else None, P(v) if v else None,
                        P(o) if o else None, None, B, Hq, Hkv, N, d, causal, scale, None)


def test_fwd_argument_validation(lib):
    # null pointers, bad sizes, head grouping, scale, alignment: rejected on the host
    assert _fwd(lib, q=0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, o=0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, B=0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, N=0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, Hq=3, Hkv=2) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == A.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, q=(1 << 20) + 2) == A.ATTN_ERR_INVALID_ARG
    # valid but not implemented head dims
    assert _fwd(lib, d=96) == A.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, d=256) == A.ATTN_ERR_UNSUPPORTED


def test_varlen_and_decode_validation(lib):
    P = ctypes.c_void_p
    p = P(1 << 20)
    assert lib.attn_fwd_varlen(p, p, p, p, None, None, 2, 10, 8, 1, 1, 128, 1, 0.1,
                               None) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_varlen(p, p, p, p, None, p, 2, 10, 8, 4, 3, 128, 1, 0.1,
                               None) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_varlen(p, p, p, p, None, p, 2, 10, 8, 4, 2, 80, 1, 0.1,
                               None) == A.ATTN_ERR_UNSUPPORTED
    # decode: missing workspace, bad page size, too many query heads per kv head
    args = [p, p, p, p, p, p, None, 4, 32, 8, 128, 16, 100, 10, 0.1]
    assert lib.attn_decode_paged(*args, None, 0, None) == A.ATTN_ERR_INVALID_ARG
    bad_ps = list(args)
    bad_ps[11] = 32
    assert lib.attn_decode_paged(*bad_ps, p, 1 << 30, None) == A.ATTN_ERR_UNSUPPORTED
    bad_g = list(args)
    bad_g[8], bad_g[9] = 64, 4
    assert lib.attn_decode_paged(*bad_g, p, 1 << 30, None) == A.ATTN_ERR_UNSUPPORTED
    many_kv = list(args)       # 16 key/value heads: one consumer warp each would exceed 8
    many_kv[8], many_kv[9] = 32, 16
    assert lib.attn_decode_paged(*many_kv, p, 1 << 30, None) == A.ATTN_ERR_UNSUPPORTED
    assert lib.attn_decode_workspace_size(0, 32, 128, 10, 16) == 0
    # the scale rule is the same for every entry point: finite and > 0
    for bad in (0.0, -0.1, float("inf"), float("nan")):
        assert lib.attn_decode_paged(*args[:-1], bad, p, 1 << 30, None) == A.ATTN_ERR_INVALID_ARG
        assert lib.attn_fwd_f32(p, p, p, p, None, 1, 1, 1, 8, 64, 1, bad,
                                None) == A.ATTN_ERR_INVALID_ARG
        assert lib.attn_fwd_varlen(p, p, p, p, None, p, 2, 10, 8, 4, 2, 128, 1, bad,
                                   None) == A.ATTN_ERR_INVALID_ARG


def test_byte_cache_decode_validation(lib):
    """The FP8 and INT8 decodes need both per-head scale arrays and take d = 128 only;
    their other rules are attn_decode_paged's."""
    P = ctypes.c_void_p
    p = P(1 << 20)
    # q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, o, lse, B, Hq, Hkv, d,
    # page_size, num_pages, max_pages_per_seq, scale, workspace, bytes, stream
    for fn in (lib.attn_decode_paged_fp8, lib.attn_decode_paged_int8):
        ok = [p, p, p, p, p, p, p, p, None, 4, 32, 8, 128, 16, 100, 10, 0.1, p, 1 << 30, None]
        for i in (3, 4):                       # a missing scale array
            bad = list(ok)
            bad[i] = None
            assert fn(*bad) == A.ATTN_ERR_INVALID_ARG, (fn, i)
        d64 = list(ok)
        d64[12] = 64
        assert fn(*d64) == A.ATTN_ERR_UNSUPPORTED
        ps32 = list(ok)
        ps32[13] = 32
        assert fn(*ps32) == A.ATTN_ERR_UNSUPPORTED
        no_ws = list(ok)
        no_ws[17] = None
        assert fn(*no_ws) == A.ATTN_ERR_INVALID_ARG


def test_f32_head_dim_rule(lib):
    """attn_fwd_f32 implements 16 <= d <= 128 with d % 16 == 0, as its header states."""
    P = ctypes.c_void_p
    p = P(1 << 20)
    for d in (8, 24, 100, 144, 256):
        assert lib.attn_fwd_f32(p, p, p, p, None, 1, 1, 1, 8, d, 1, 0.1,
                                None) == A.ATTN_ERR_UNSUPPORTED, d
    text = open(HEADER).read()
    assert "16 <= d <= 128 and d % 16 == 0" in text


def test_f32_rows_hook_takes_the_two_tile_heights(lib):
    """attn_testing_fwd_f32_rows runs 16-, 4- or 2-row CTAs; any other height is refused
    before anything is launched, and the shared argument rules still apply."""
    P = ctypes.c_void_p
    p = P(1 << 20)
    fn = lib.attn_testing_fwd_f32_rows
    fn.argtypes = [P, P, P, P, P] + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int, P]
    fn.restype = ctypes.c_int
    for rows in (0, 1, 3, 8, 32, -4):
        assert fn(p, p, p, p, None, 1, 1, 1, 8, 64, 1, 0.1, rows, None) == A.ATTN_ERR_INVALID_ARG
    assert fn(None, p, p, p, None, 1, 1, 1, 8, 64, 1, 0.1, 4, None) == A.ATTN_ERR_INVALID_ARG
    assert fn(p, p, p, p, None, 1, 1, 1, 8, 24, 1, 0.1, 16, None) == A.ATTN_ERR_UNSUPPORTED


def test_workspace_size_signature():
    """attn_decode_workspace_size(B, Hq, d, max_pages_per_seq, page_size): five sizes."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"attn_decode_workspace_size\(([^)]*)\)", text)
    names = [a.split()[-1] for a in m.group(1).split(",")]
    assert names == ["B", "Hq", "d", "max_pages_per_seq", "page_size"]


def test_host_entry_validation(lib):
    # attn_fwd_host rejects bad arguments before any CUDA call (host pointers need no
    # alignment, so an odd address passes that check and fails nothing else)
    P = ctypes.c_void_p
    h = P((1 << 20) + 3)
    assert lib.attn_fwd_host(None, h, h, h, None, 1, 4, 2, 8, 128, 1, 0.1,
                             None) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_host(h, h, h, h, None, 1, 4, 3, 8, 128, 1, 0.1,
                             None) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_host(h, h, h, h, None, 1, 4, 2, 0, 128, 1, 0.1,
                             None) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_host(h, h, h, h, None, 1, 4, 2, 8, 128, 1, float("inf"),
                             None) == A.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_host(h, h, h, h, None, 1, 4, 2, 8, 96, 1, 0.1,
                             None) == A.ATTN_ERR_UNSUPPORTED


def test_binding_requires_library(tmp_path):
    """The binding raises rather than falling back when the library is absent."""
    import importlib
    mod = importlib.reload(A)
    try:
        with pytest.raises(OSError):
            mod.load_library(str(tmp_path / "missing.so"))
    finally:
        importlib.reload(A)


def test_cuda_failure_text_is_recorded(lib):
    # without a usable device, a valid call fails in the CUDA runtime: the status is
    # ATTN_ERR_CUDA and the failure's name is kept for the caller's thread
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this checks the failure path")
    assert _fwd(lib) == A.ATTN_ERR_CUDA
    text = A.attn_last_cuda_error()
    assert text.startswith("cuda") and "no CUDA error recorded" not in text, text
    with pytest.raises(A.AttnError, match=r"CUDA error \(status 3\) \[cuda"):
        A._check(A.ATTN_ERR_CUDA, "attn_fwd")


def test_binding_checks_tensors_before_calling_the_library():
    """The ctypes binding refuses CPU, mistyped, non-contiguous or mis-shaped tensors with a
    ValueError before any call into the library (so no device is needed to see it)."""
    import torch
    q = torch.zeros((1, 8, 4, 128), dtype=torch.bfloat16)
    k = torch.zeros((1, 8, 2, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        A.attn_fwd(q, k, k)                       # host tensors for the device entry point
    with pytest.raises(ValueError, match="CPU bfloat16"):
        A.attn_fwd_host(q.float(), k, k)          # wrong dtype for the host entry point
    with pytest.raises(ValueError, match="CPU bfloat16"):
        A.attn_fwd_host(q.transpose(1, 2), k, k)  # not contiguous
    with pytest.raises(ValueError, match="matching q"):
        A.attn_fwd_host(q, k[:, :4], k)           # k with another sequence length
