"""GPU parity for the two-pass forward (attn_fwd_two_pass: row statistics first,
then the output, as the FlashAttention-1 section of "Donanıma Duyarlı Algoritma
Tasarımı: FlashAttention" orders it) against the fp64 oracle, and against the
one-pass kernel on the same inputs.  Tolerances are in tests/parity.py."""
import ctypes

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


def f32(t):
    return t.float().cpu().numpy()


def check_status():
    st = A.attn_get_device_status()
    assert st == 0, A.attn_status_string(st)


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", [
    (1, 1, 1, 1, 128, True), (1, 300, 4, 2, 128, True), (2, 129, 2, 1, 64, False),
    (1, 1000, 8, 2, 128, False), (3, 513, 6, 3, 64, True), (1, 256, 2, 2, 128, True),
])
def test_two_pass_small(oracle, B, N, Hq, Hkv, d, causal):
    w = inputs.dense(B, N, Hq, Hkv, d, 7000 + B + N + Hq + d, torch.bfloat16, causal=causal)
    o, lse = A.attn_fwd_two_pass(w.q.cuda(), w.k.cuda(), w.v.cuda(), causal, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_fwd(f32(w.q), f32(w.k), f32(w.v), causal, w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (B, N, Hq, Hkv, d, causal))


def test_two_pass_large_scores(oracle):
    """Scores with standard deviation 6: the first pass's running maximum moves often;
    the second pass uses the final statistics directly."""
    w = inputs.dense(1, 400, 2, 2, 128, 7100, torch.float32)
    q = (w.q * 6.0).to(torch.bfloat16)
    k = w.k.to(torch.bfloat16)
    v = (w.v * 0.25).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = A.attn_fwd_two_pass(q.cuda(), k.cuda(), v.cuda(), causal, w.scale)
        torch.cuda.synchronize()
        check_status()
        o_ref, lse_ref = oracle.attn_fwd(f32(q), f32(k), f32(v), causal, w.scale)
        assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), ("large", causal))


def test_two_pass_agrees_with_one_pass():
    """Both orders round P to bf16 at different points (against the running maximum, or
    against the final statistics), so each output is within the parity tolerance of the
    exact one and the two within twice that of each other; the first pass forms the same
    row sums as the one-pass kernel, so the LSE agrees bitwise."""
    w = inputs.dense(2, 777, 8, 2, 128, 7200, torch.bfloat16)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o1, l1 = A.attn_fwd(q, k, v, True, w.scale)
    o2, l2 = A.attn_fwd_two_pass(q, k, v, True, w.scale)
    torch.cuda.synchronize()
    check_status()
    e = errors(f32(o2), f32(o1), f32(l2), f32(l1))
    assert e["max_o"] <= 2e-2 and e["mean_o"] <= 1e-3 and e["max_lse"] == 0.0, e


def test_two_pass_requires_lse():
    w = inputs.dense(1, 16, 1, 1, 128, 7300, torch.bfloat16)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o = torch.empty_like(q)
    P = ctypes.c_void_p
    rc = A.load_library().attn_fwd_two_pass(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()),
                                            P(o.data_ptr()), None, 1, 1, 1, 16, 128, 1,
                                            ctypes.c_float(w.scale), None)
    assert rc == A.ATTN_ERR_INVALID_ARG


def test_workload_gqa_two_pass_sampled(oracle):
    """The N=16384 GQA causal workload in the two-pass order, on sampled rows."""
    w = inputs.make("gqa_causal_n16384_two_pass")
    o, lse = A.attn_fwd_two_pass(w.q.cuda(), w.k.cuda(), w.v.cuda(), True, w.scale)
    torch.cuda.synchronize()
    check_status()
    B, N, Hq, d = w.q.shape
    rng = np.random.default_rng(9)
    i = np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 124)])
    h = rng.integers(0, Hq, len(i))
    rows = np.stack([np.zeros_like(i), h, i], 1).astype(np.int32)
    o_ref, lse_ref = oracle.attn_rows(f32(w.q), f32(w.k), f32(w.v), rows, True, w.scale)
    assert_close(errors(f32(o)[0, i, h], o_ref, f32(lse)[0, h, i], lse_ref), "two-pass N=16384")
