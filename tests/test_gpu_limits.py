"""GPU parity at the edges of the supported sizes, against the fp64 oracle: a 65,536-token
causal prefill with the largest query-head group (8 per key/value head) on sampled rows, the
decode with the largest group and a 70,000-token sequence beside a 1-token one, and 300 packed
sequences of 0 to 300 tokens.  Tolerances are in tests/parity.py."""
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


def test_prefill_65536_tokens_group_of_8(oracle):
    """B=1, N=65536, Hq=8, Hkv=1, d=128, causal: 512 query tiles, 4 head pairs; rows at the
    start, at tile edges and at the end, and random ones."""
    w = inputs.dense(1, 65536, 8, 1, 128, 9200, torch.bfloat16, causal=True)
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), True, w.scale)
    torch.cuda.synchronize()
    check_status()
    N = 65536
    rng = np.random.default_rng(12)
    i = np.concatenate([[0, 1, 127, 128, 32767, 32768, N - 129, N - 128, N - 1],
                        rng.integers(0, N, 55)])
    h = rng.integers(0, 8, len(i))
    rows = np.stack([np.zeros_like(i), h, i], 1).astype(np.int32)
    o_ref, lse_ref = oracle.attn_rows(f32(w.q), f32(w.k), f32(w.v), rows, True, w.scale)
    assert_close(errors(f32(o)[0, i, h], o_ref, f32(lse)[0, h, i], lse_ref), "N=65536")


def test_decode_group_of_8_and_a_70000_token_sequence(oracle):
    p = inputs.paged([1, 70000, 3000], 64, 8, 128, 9300)
    args = [t.cuda() for t in (p.q, p.k_cache, p.v_cache, p.page_table, p.seq_lens)]
    o, lse = A.attn_decode_paged(*args, p.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.decode_paged(f32(p.q), f32(p.k_cache), f32(p.v_cache),
                                         p.page_table.numpy(), p.seq_lens.numpy(), p.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), "decode 70000")


def test_varlen_300_sequences(oracle):
    rng = np.random.default_rng(13)
    lens = rng.integers(0, 301, 300)
    lens[[0, 17, 299]] = 0
    lens[[1, 2]] = [1, 300]
    # values halved (factor 0.5 for Q, K and V): a sequence's second and third rows average
    # two or three V rows, and at |O| >= 4 the bf16 output itself can be 0.0156 from the
    # exact value (one such row rounded correctly to 4.0625 from 4.0758 at full scale)
    w = inputs.varlen(lens, 4, 2, 128, 9400, torch.bfloat16, factor=0.5, causal=True)
    o, lse = A.attn_fwd_varlen(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.cu_seqlens.cuda(),
                               int(lens.max()), True, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_varlen(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(), True,
                                        w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), "300 sequences")
