"""GPU tests of the host-buffer prefill (attn_fwd_host): its result is bitwise the
device entry point's (each key/value head group is computed by the same kernel on
the same rows), for one to four head groups, ragged lengths, both head dims,
page-locked and pageable buffers, without an LSE output, across staging-area
growth and release; and one case against the fp64 oracle.  Invalid arguments
are rejected before any copy."""
import numpy as np
import pytest
import torch

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import inputs
from parity import assert_close, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.load_library()
    assert A.attn_get_device_status() == 0
    yield
    A.attn_release_host_staging()


def check_status():
    st = A.attn_get_device_status()
    assert st == 0, A.attn_status_string(st)


def device_result(w, causal):
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), causal, w.scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", [
    # causal: pieces along the sequence (256-row tile pairs)
    (1, 300, 8, 2, 128, True),    # two pieces, the second a ragged single tile
    (1, 1000, 6, 3, 128, True),   # four pieces, row-tile pairs (odd group size)
    (2, 700, 4, 2, 64, True),     # three pieces per sequence, two sequences
    (1, 17, 1, 1, 128, True),     # one piece
    (3, 64, 16, 8, 128, True),    # one piece, three sequences
    (1, 2048, 32, 8, 128, True),  # eight pieces, the N=16384 workload's heads
    (1, 4608, 8, 8, 64, True),    # sixteen pieces of two tiles
    # full attention: pieces are key/value head groups
    (2, 129, 4, 4, 64, False),    # four groups of one key/value head
    (1, 600, 8, 2, 128, False),   # two groups
    (1, 333, 6, 3, 128, False),   # three groups
    (2, 100, 16, 8, 128, False),  # four groups of two key/value heads
])
def test_host_equals_device(B, N, Hq, Hkv, d, causal):
    w = inputs.dense(B, N, Hq, Hkv, d, 8000 + N + Hq, torch.bfloat16, causal=causal)
    q, k, v = (t.pin_memory() for t in (w.q, w.k, w.v))
    o, lse = A.attn_fwd_host(q, k, v, causal, w.scale)
    check_status()
    o_dev, lse_dev = device_result(w, causal)
    assert torch.equal(o, o_dev)
    assert torch.equal(lse, lse_dev)


def test_host_workload_gqa_causal_n16384():
    """The benchmark's end-to-end call: B=1, N=16384, Hq=32, Hkv=8, causal."""
    w = inputs.make("gqa_causal_n16384")
    q, k, v = (t.pin_memory() for t in (w.q, w.k, w.v))
    o, lse = A.attn_fwd_host(q, k, v, True, w.scale)
    check_status()
    o_dev, lse_dev = device_result(w, True)
    assert torch.equal(o, o_dev)
    assert torch.equal(lse, lse_dev)


def test_host_pageable_buffers_and_no_lse():
    w = inputs.dense(2, 200, 8, 4, 128, 8100, torch.bfloat16)
    o, lse = A.attn_fwd_host(w.q, w.k, w.v, True, w.scale, want_lse=False)
    check_status()
    assert lse is None
    o_dev, _ = device_result(w, True)
    assert torch.equal(o, o_dev)


def test_host_staging_grows_shrinks_and_releases():
    for N in (64, 3000, 100):
        w = inputs.dense(1, N, 4, 2, 128, 8200 + N, torch.bfloat16)
        o, lse = A.attn_fwd_host(w.q.pin_memory(), w.k.pin_memory(), w.v.pin_memory(), True,
                                 w.scale)
        check_status()
        o_dev, lse_dev = device_result(w, True)
        assert torch.equal(o, o_dev) and torch.equal(lse, lse_dev)
        A.attn_release_host_staging()


def test_host_against_oracle(oracle):
    w = inputs.dense(1, 333, 8, 2, 128, 8300, torch.bfloat16)
    o, lse = A.attn_fwd_host(w.q, w.k, w.v, True, w.scale)
    check_status()
    o_ref, lse_ref = oracle.attn_fwd(w.q.float().numpy(), w.k.float().numpy(),
                                     w.v.float().numpy(), True, w.scale)
    assert_close(errors(o.float().numpy(), o_ref, lse.numpy(), lse_ref), "host")


def test_host_rejects_bad_arguments():
    w = inputs.dense(1, 16, 4, 2, 128, 8400, torch.bfloat16)
    with pytest.raises(ValueError):
        A.attn_fwd_host(w.q.cuda(), w.k, w.v)          # device tensor
    q96 = torch.zeros((1, 16, 4, 96), dtype=torch.bfloat16)
    k96 = torch.zeros((1, 16, 2, 96), dtype=torch.bfloat16)
    with pytest.raises(A.AttnError) as e:
        A.attn_fwd_host(q96, k96, k96)                 # head dim 96: unsupported
    assert e.value.code == A.ATTN_ERR_UNSUPPORTED
    k3 = torch.zeros((1, 16, 3, 128), dtype=torch.bfloat16)
    q4 = torch.zeros((1, 16, 4, 128), dtype=torch.bfloat16)
    with pytest.raises(A.AttnError) as e:
        A.attn_fwd_host(q4, k3, k3)                    # Hq % Hkv != 0
    assert e.value.code == A.ATTN_ERR_INVALID_ARG
