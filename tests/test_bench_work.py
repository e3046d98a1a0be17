"""The algorithmic work that bench.py divides by (FLOPs of a prefill, bytes of a decode),
checked on small generated inputs against brute-force counts of allowed (query, key)
pairs and cached tokens, and against the workloads' stated figures."""
import numpy as np
import torch

import bench
from attn_fwd_07_b300 import inputs


def pairs_dense(N, causal, wl=-1, wr=-1):
    """Allowed (query, key) pairs of one N-token sequence, counted one by one."""
    n = 0
    for i in range(N):
        for j in range(N):
            if causal and j > i:
                continue
            if wl >= 0 and j < i - wl:
                continue
            if wr >= 0 and j > i + wr:
                continue
            n += 1
    return n


def test_dense_convention():
    """Full: 4*B*Hq*N^2*d; causal: half of it (the stated convention, not N(N+1)/2)."""
    for causal in (False, True):
        w = inputs.dense(2, 40, 4, 2, 64, 1, causal=causal)
        want = 4.0 * 2 * 4 * 40 * 40 * 64 * (0.5 if causal else 1.0)
        assert bench.prefill_flops(w) == want


def test_workload_3_figure():
    """2*B*Hq*N^2*d = 2.199e12 for B=1, Hq=32, N=16384, d=128 (the headline figure),
    from the formula alone (the workload's tensors are not generated)."""
    class W:
        causal = True
        q = torch.empty((1, 16384, 32, 128), dtype=torch.bfloat16, device="meta")
    assert bench.prefill_flops(W()) == 2.0 * 32 * 16384 ** 2 * 128
    assert abs(bench.prefill_flops(W()) - 2.199e12) < 1e9


def test_window_counts_allowed_pairs_exactly():
    for wl, wr in ((7, 3), (0, 0), (-1, 5), (12, -1), (100, 100)):
        w = inputs.dense(1, 37, 2, 2, 64, 2, causal=False)
        w.window = (wl, wr)
        assert bench.prefill_flops(w) == 4.0 * 2 * 64 * pairs_dense(37, False, wl, wr)


def test_varlen_sums_squares():
    w = inputs.varlen([5, 1, 33, 16], 4, 2, 64, 3, causal=True)
    assert bench.prefill_flops(w) == 4.0 * 4 * 64 * 0.5 * (25 + 1 + 33 * 33 + 256)


def test_chunk_counts_allowed_pairs_exactly():
    """A chunk of q_len queries at the end of ctx cached tokens: causal query i sees the
    first ctx - q_len + i + 1 keys; full attention sees all ctx."""
    ctx, ql = [40, 17, 100], [7, 17, 1]
    for causal in (True, False):
        c = inputs.chunked(ctx, ql, 4, 2, 64, 4, causal=causal)
        pairs = sum(sum((n - m + i + 1) if causal else n for i in range(m))
                    for n, m in zip(ctx, ql))
        assert bench.prefill_flops(c) == 4.0 * 4 * 64 * pairs


def test_decode_bytes_per_token():
    """K and V rows of every cached token read once: 2 * Hkv * d * element size."""
    lens = [1, 15, 16, 17, 300, 0]
    p = inputs.paged(lens, 8, 4, 128, 5)
    assert bench.decode_bytes(p) == 2.0 * 4 * 128 * 2 * sum(lens)
    f = inputs.paged_fp8(lens, 8, 4, 128, 5)
    assert bench.decode_bytes(f) == 2.0 * 4 * 128 * 1 * sum(lens)
    i8 = inputs.paged_int8(lens, 8, 4, 128, 5)
    assert bench.decode_bytes(i8) == 2.0 * 4 * 128 * 1 * sum(lens)


def test_every_workload_has_a_config_and_a_kernel_name():
    """Each named workload maps to a config key and, on the device, to a kernel whose
    sources the fingerprint covers (no workload is left without its traffic lookup)."""
    kinds = {w.kind for w in inputs.WORKLOADS.values()}
    assert {"dense", "varlen", "decode", "decode_fp8", "decode_int8", "chunk", "window",
            "two_pass"} <= kinds
    for k in ("decode_split_kernel<0>", "decode_split_kernel<1>", "decode_split_kernel<2>",
              "prefill_tc_kernel", "prefill_simt_kernel", "prefill_simt_rows_kernel<4>",
              "prefill_simt_rows_kernel<2>"):
        assert len(bench.kernel_fingerprint(k)) == 16
