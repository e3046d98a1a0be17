"""attn_decode_paged_noalloc: the paged decode for callers that cannot allocate
device memory (a plugin host that only passes its input and output buffers, or a
server that reserved all device memory at start-up).  It must give the same
results as attn_decode_paged with a caller-provided workspace, call after call,
although every call reuses the library's one built-in scratch array.

Kept in its own file, collected last, so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import inputs
from parity import assert_close, errors

pytestmark = pytest.mark.gpu


def _dev(w):
    return [t.cuda() for t in (w.q, w.k_cache, w.v_cache, w.page_table, w.seq_lens)]


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.load_library()
    # two different problems in a row: the second call must not see the first one's
    # leftovers in the shared scratch array
    cases = [([1, 15, 17, 1023, 4000], 32, 8, 128, 501),
             ([2048, 3, 700], 16, 4, 64, 502)]
    for lens, Hq, Hkv, d, seed in cases:
        w = inputs.paged(lens, Hq, Hkv, d, seed, page_size=16, dtype=torch.bfloat16)
        args = _dev(w)
        o_ref, l_ref = A.attn_decode_paged(*args, w.scale)
        o, lse = A.attn_decode_paged_noalloc(*args, w.scale)
        torch.cuda.synchronize()
        assert A.attn_get_device_status() == 0
        e = errors(o.float().cpu().numpy(), o_ref.float().cpu().numpy(),
                   lse.cpu().numpy(), l_ref.cpu().numpy())
        assert_close(e, (lens, Hq, Hkv, d))


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = A.load_library()
    B, Hq, Hkv, d = 4096, 64, 8, 128   # needs far more than the built-in scratch
    assert A.attn_decode_workspace_size(B, Hq, d, 8, 16) > (8 << 20)
    p = torch.empty(16, dtype=torch.uint8, device="cuda")
    ptr = p.data_ptr()
    import ctypes
    rc = lib.attn_decode_paged_noalloc(*(ctypes.c_void_p(ptr) for _ in range(6)), None, B, Hq,
                                       Hkv, d, 16, 1, 8, 0.1, None)
    assert rc == A.ATTN_ERR_UNSUPPORTED
