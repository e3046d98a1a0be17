"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element, at sizes that span several tiles and a
ragged tail, at the five workloads' full sizes (sampled rows where the oracle
would take minutes), and on edge cases.  Tolerances are in tests/parity.py.
"""
import ctypes
import math

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


# ---------------------------------------------------------------- dense bf16 (tensor cores)

DENSE_CASES = [
    # B, N, Hq, Hkv, d, causal
    (1, 1, 1, 1, 128, False), (1, 1, 1, 1, 128, True), (1, 2, 1, 1, 64, True),
    (1, 63, 2, 1, 128, True), (1, 64, 2, 2, 64, False), (2, 65, 2, 1, 128, False),
    (1, 127, 4, 2, 128, True), (1, 128, 1, 1, 128, True), (1, 128, 1, 1, 64, False),
    (2, 129, 4, 1, 128, True), (1, 255, 2, 2, 64, True), (1, 256, 4, 4, 128, False),
    (1, 300, 8, 2, 128, True), (2, 300, 2, 1, 64, False), (1, 1000, 4, 1, 128, True),
    (1, 1000, 2, 2, 64, True), (1, 777, 2, 1, 128, False), (3, 513, 6, 3, 64, True),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", DENSE_CASES)
def test_prefill_bf16_small(oracle, B, N, Hq, Hkv, d, causal):
    seed = 1000 + B * 7 + N * 3 + Hq * 5 + d + int(causal)
    w = inputs.dense(B, N, Hq, Hkv, d, seed, torch.bfloat16, causal=causal)
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), causal, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_fwd(f32(w.q), f32(w.k), f32(w.v), causal, w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (B, N, Hq, Hkv, d, causal))


def test_prefill_bf16_deterministic():
    w = inputs.dense(2, 700, 4, 2, 128, 77, torch.bfloat16)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o1, l1 = A.attn_fwd(q, k, v, True, w.scale)
    o2, l2 = A.attn_fwd(q, k, v, True, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prefill_gqa_equals_repeated_kv_heads():
    w = inputs.dense(1, 333, 8, 2, 128, 78, torch.bfloat16)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o1, l1 = A.attn_fwd(q, k, v, True, w.scale)
    kr = k.repeat_interleave(4, dim=2).contiguous()
    vr = v.repeat_interleave(4, dim=2).contiguous()
    o2, l2 = A.attn_fwd(q, kr, vr, True, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("kind", ["large_scores", "equal_keys", "one_hot_peak"])
def test_prefill_adversarial(oracle, kind):
    """Scores far from zero (rescaling path), identical keys (uniform weights),
    and a single dominant key per row."""
    B, N, H, d = 1, 400, 2, 128
    w = inputs.dense(B, N, H, H, d, 90, torch.float32)
    q, k, v = w.q.clone(), w.k.clone(), w.v.clone()
    if kind == "large_scores":
        # scores with standard deviation 6 (maxima growing along the row, very
        # peaked rows).  V is scaled so that |O| stays below 2: the absolute
        # tolerance is meant for outputs of that size (a bf16 output at |O| in
        # [2, 4) already carries up to 0.0078 of rounding alone).
        q *= 6.0
        v *= 0.25
    elif kind == "equal_keys":
        k[:] = k[:, :1]
    else:
        k[:, 77] = q[:, 77] * 4.0
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    for causal in (False, True):
        o, lse = A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal, w.scale)
        torch.cuda.synchronize()
        check_status()
        o_ref, lse_ref = oracle.attn_fwd(f32(q), f32(k), f32(v), causal, w.scale)
        assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (kind, causal))


@pytest.mark.parametrize("keys", [(40,), (100,), (150,), (230,), (300,), (480,), (150, 480),
                                  (230, 480), (229, 230)])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (1, 1)])
def test_prefill_maximum_jumps_inside_a_key_tile(oracle, keys, Hq, Hkv):
    """Every query shares a direction u; the listed keys are 32 u, so their scores sit
    about 33 (log2 units) above the rest.  A key in the first or second 64-key half of
    a key tile that is not the row's first moves the row maximum in the middle of the
    tile (the exponent reference is exceeded by far more than the half-tile bound), a
    key in the first tile sets it; two keys move it twice.  Both CTA pairings (two
    heads of a group, two row tiles)."""
    B, N, d = 1, 512, 128
    w = inputs.dense(B, N, Hq, Hkv, d, 95, torch.float32)
    u = torch.full((d,), 0.25)
    q = w.q * 0.3 + u
    k = w.k.clone()
    for key in keys:
        k[:, key] = u * 32.0
    # V halved so that |O| (about one V row here) stays below 2.2
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, w.v * 0.5))
    for causal in (False, True):
        o, lse = A.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal, w.scale)
        torch.cuda.synchronize()
        check_status()
        o_ref, lse_ref = oracle.attn_fwd(f32(q), f32(k), f32(v), causal, w.scale)
        assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (keys, Hq, causal))


# ---------------------------------------------------------------- fp32 (CUDA cores)

@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", [
    (1, 1, 1, 1, 64, False), (1, 63, 2, 1, 64, True), (1, 65, 1, 1, 128, False),
    (2, 129, 4, 2, 64, True), (1, 255, 2, 2, 32, False), (1, 300, 4, 1, 128, True),
    # every head dimension the kernel takes: a row's 64 threads own output columns c and
    # c + 64 below d, two, one or none each
    (1, 70, 2, 1, 16, True), (1, 100, 1, 1, 48, False), (2, 90, 2, 2, 80, True),
    (1, 130, 3, 1, 96, False), (1, 77, 2, 2, 112, True),
    # CTAs of 4 query rows: sequences shorter than one, ragged last CTAs, and many key
    # tiles below the causal diagonal
    (1, 2, 1, 1, 64, True), (3, 5, 2, 1, 128, True), (2, 7, 2, 2, 16, False),
    (1, 1000, 2, 1, 128, True), (1, 513, 1, 1, 64, False),
])
def test_prefill_f32_small(oracle, B, N, Hq, Hkv, d, causal):
    w = inputs.dense(B, N, Hq, Hkv, d, 2000 + N + d, torch.float32, causal=causal)
    o, lse = A.attn_fwd_f32(w.q.cuda(), w.k.cuda(), w.v.cuda(), causal, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_fwd(f32(w.q), f32(w.k), f32(w.v), causal, w.scale)
    e = errors(f32(o), o_ref, f32(lse), lse_ref)
    assert_close(e, (B, N, Hq, Hkv, d, causal))
    assert e["max_o"] < 1e-4 and e["max_lse"] < 1e-4, e  # fp32 arithmetic throughout


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", [
    (1, 256, 1, 1, 64, False), (1, 1, 1, 1, 16, True), (2, 67, 4, 2, 128, True),
    (1, 300, 2, 1, 96, False), (3, 130, 2, 2, 48, True), (1, 1100, 1, 1, 80, True),
])
def test_prefill_f32_every_tile_height(oracle, B, N, Hq, Hkv, d, causal):
    """16-, 4- and 2-row CTAs (through the test hook) each match the oracle, and
    attn_fwd_f32 returns, bit for bit, the result of the height its launch-size rule
    picks: with C CTAs of 16 rows, 2 rows when 8 C <= #SM, 4 rows when 2 C <= #SM."""
    lib = A.load_library()
    P = ctypes.c_void_p
    fn = lib.attn_testing_fwd_f32_rows
    fn.argtypes = [P, P, P, P, P] + [ctypes.c_int] * 6 + [ctypes.c_float, ctypes.c_int, P]
    fn.restype = ctypes.c_int
    w = inputs.dense(B, N, Hq, Hkv, d, 2100 + N + d, torch.float32, causal=causal)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o_ref, lse_ref = oracle.attn_fwd(f32(w.q), f32(w.k), f32(w.v), causal, w.scale)
    got = {}
    for rows in (16, 4, 2):
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
        rc = fn(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()),
                P(lse.data_ptr()), B, Hq, Hkv, N, d, int(causal), w.scale, rows,
                P(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, A.attn_status_string(rc)
        torch.cuda.synchronize()
        check_status()
        e = errors(f32(o), o_ref, f32(lse), lse_ref)
        assert_close(e, (rows, B, N, Hq, Hkv, d, causal))
        assert e["max_o"] < 1e-4 and e["max_lse"] < 1e-4, (rows, e)
        got[rows] = (o, lse)
    o, lse = A.attn_fwd_f32(q, k, v, causal, w.scale)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas16 = ((N + 15) // 16) * Hq * B
    pick = 2 if 8 * ctas16 <= sms else 4 if 2 * ctas16 <= sms else 16
    assert torch.equal(o, got[pick][0]) and torch.equal(lse, got[pick][1]), pick


# ---------------------------------------------------------------- varlen

@pytest.mark.parametrize("lens,d,causal", [
    ([1, 17, 128, 129, 513], 128, True),
    ([300, 0, 1, 64, 200], 64, True),
    ([257, 33], 128, False),
])
def test_varlen_small(oracle, lens, d, causal):
    Hq, Hkv = 4, 2
    w = inputs.varlen(lens, Hq, Hkv, d, 3000 + sum(lens), torch.bfloat16, causal=causal)
    o, lse = A.attn_fwd_varlen(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.cu_seqlens.cuda(),
                               max(lens), causal, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_varlen(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(),
                                        causal, w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (lens, d, causal))


# ---------------------------------------------------------------- decode

def decode_oracle_rows(oracle, w, seqs):
    return oracle.decode_paged(f32(w.q), f32(w.k_cache), f32(w.v_cache), w.page_table.numpy(),
                               w.seq_lens.numpy(), w.scale, seqs=seqs)


def run_decode(w, **kw):
    return A.attn_decode_paged(w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda(),
                               w.page_table.cuda(), w.seq_lens.cuda(), w.scale, **kw)


@pytest.mark.parametrize("lens,Hq,Hkv,d", [
    ([1, 15, 16, 17, 1023], 32, 8, 128),
    ([0, 5, 2048, 33], 8, 8, 64),
    ([4096], 16, 4, 128),
    ([1] * 40 + [3000], 32, 8, 128),
])
def test_decode_small(oracle, lens, Hq, Hkv, d):
    w = inputs.paged(lens, Hq, Hkv, d, 4000 + sum(lens), page_size=16, dtype=torch.bfloat16)
    o, lse = run_decode(w)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = decode_oracle_rows(oracle, w, np.arange(len(lens)))
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (lens, Hq, Hkv, d))


def test_decode_page_permutation_is_bitwise_invariant():
    lens = [700, 31, 5000, 16]
    w = inputs.paged(lens, 32, 8, 128, 4100, page_size=16, dtype=torch.bfloat16)
    o1, l1 = run_decode(w)
    P = w.k_cache.shape[0]
    perm = torch.from_numpy(np.random.default_rng(4101).permutation(P))
    inv = torch.argsort(perm)
    pt = w.page_table.clone()
    mask = pt >= 0
    pt[mask] = inv[pt[mask].long()].to(torch.int32)
    w2 = inputs.Paged(w.q, w.k_cache[perm].contiguous(), w.v_cache[perm].contiguous(), pt,
                      w.seq_lens, w.scale)
    o2, l2 = run_decode(w2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_matches_last_row_of_causal_prefill():
    """Two paths of the library agree: decode of token N-1 against a contiguous
    cache equals row N-1 of causal prefill over the same keys."""
    N, Hq, Hkv, d = 1000, 8, 2, 128
    w = inputs.dense(1, N, Hq, Hkv, d, 4200, torch.bfloat16)
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), True, w.scale)
    npg = (N + 15) // 16
    kc = torch.zeros(npg * 16, Hkv, d, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kc[:N] = w.k[0]
    vc[:N] = w.v[0]
    pw = inputs.Paged(w.q[0, N - 1:N].contiguous(), kc.view(npg, 16, Hkv, d),
                      vc.view(npg, 16, Hkv, d), torch.arange(npg, dtype=torch.int32)[None],
                      torch.tensor([N], dtype=torch.int32), w.scale)
    od, ld = run_decode(pw)
    torch.cuda.synchronize()
    e = errors(f32(od[0]), f32(o[0, N - 1]), f32(ld[0]), f32(lse[0, :, N - 1]))
    assert e["max_o"] <= 2e-2 and e["max_lse"] <= 2e-3, e


def test_decode_bad_page_id_is_reported_not_read(oracle):
    """A page id outside the pool is never dereferenced: its tokens count as
    masked, the other sequences are unaffected, and the device status reports it."""
    lens = [40, 100]
    w = inputs.paged(lens, 8, 2, 128, 4300, page_size=16, dtype=torch.bfloat16)
    pt = w.page_table.clone()
    pt[1, 2] = 10 ** 6
    w2 = inputs.Paged(w.q, w.k_cache, w.v_cache, pt, w.seq_lens, w.scale)
    o, lse = run_decode(w2)
    st = A.attn_get_device_status()
    assert st == A.ATTN_ERR_DEVICE_BOUNDS
    o_ref, lse_ref = decode_oracle_rows(oracle, w, [0])
    assert_close(errors(f32(o[:1]), o_ref, f32(lse[:1]), lse_ref))
    assert A.attn_get_device_status() == 0


# ---------------------------------------------------------------- the five workloads

def test_workload_single_head_f32(oracle):
    w = inputs.make("single_head_f32")
    o, lse = A.attn_fwd_f32(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.causal, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_fwd(f32(w.q), f32(w.k), f32(w.v), w.causal, w.scale)
    e = errors(f32(o), o_ref, f32(lse), lse_ref)
    assert_close(e)
    assert e["max_o"] < 1e-4, e


def test_workload_batched_causal_full(oracle):
    """B=4 H=16 N=2048 d=128 causal: every output element against the oracle."""
    w = inputs.make("batched_causal_b4h16n2048")
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.causal, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_fwd(f32(w.q), f32(w.k), f32(w.v), w.causal, w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref))


def sampled_rows(B, Hq, N, n_random, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = []
    for b in range(B):
        for h in sorted(set([0, Hq - 1] + list(rng.integers(0, Hq, 2)))):
            for i in sorted(set([x for x in fixed if 0 <= x < N] +
                                list(rng.integers(0, N, n_random)))):
                rows.append((b, h, int(i)))
    return np.array(rows, np.int32)


def test_workload_gqa_n16384_sampled(oracle):
    """B=1 Hq=32 Hkv=8 N=16384 causal, as timed by the benchmark: sampled rows."""
    w = inputs.make("gqa_causal_n16384")
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.causal, w.scale)
    torch.cuda.synchronize()
    check_status()
    B, N, Hq, _ = w.q.shape
    rows = sampled_rows(B, Hq, N, 24, 5)
    o_ref, lse_ref = oracle.attn_rows(f32(w.q), f32(w.k), f32(w.v), rows, True, w.scale)
    og = f32(o)[rows[:, 0], rows[:, 2], rows[:, 1]]
    lg = f32(lse)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(errors(og, o_ref, lg, lse_ref))
    # whole-output properties: finite, and the LSE of causal row 0 is its single score
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


def test_workload_varlen_sampled(oracle):
    w = inputs.make("varlen_causal_8seq")
    lens = w.lens
    o, lse = A.attn_fwd_varlen(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.cu_seqlens.cuda(),
                               int(lens.max()), True, w.scale)
    torch.cuda.synchronize()
    check_status()
    cu = w.cu_seqlens.numpy()
    q, k, v = f32(w.q), f32(w.k), f32(w.v)
    og_all, lg_all = f32(o), f32(lse)
    rng = np.random.default_rng(6)
    for s, L in enumerate(lens):
        a, b = int(cu[s]), int(cu[s + 1])
        idx = sorted(set([0, 1, 127, 128, L - 1] + list(rng.integers(0, L, 12))))
        rows = np.array([(0, h, i) for h in (0, 13, 31) for i in idx], np.int32)
        o_ref, l_ref = oracle.attn_rows(q[None, a:b], k[None, a:b], v[None, a:b], rows, True,
                                        w.scale)
        og = og_all[a + rows[:, 2], rows[:, 1]]
        lg = lg_all[rows[:, 1], a + rows[:, 2]]
        assert_close(errors(og, o_ref, lg, l_ref), ("seq", s, L))


def test_workload_decode_sampled(oracle):
    """B=64 decode, lengths U[1024,32768], permuted 16-token pages: 8 sampled
    sequences, all heads, plus finiteness of the rest."""
    w = inputs.make("decode_paged_b64")
    o, lse = run_decode(w)
    torch.cuda.synchronize()
    check_status()
    lens = w.seq_lens.numpy()
    seqs = sorted(set([int(lens.argmin()), int(lens.argmax()), 0, 63] +
                      list(np.random.default_rng(7).integers(0, 64, 4))))
    # gather only the sampled sequences' pages into a compact cache for the oracle
    ps = w.page_size
    pages = [w.page_table[b, :(int(lens[b]) + ps - 1) // ps].numpy() for b in seqs]
    allp = np.concatenate(pages)
    kc, vc = f32(w.k_cache[torch.from_numpy(allp).long()]), f32(w.v_cache[torch.from_numpy(allp).long()])
    maxp = max(len(p) for p in pages)
    pt = np.full((len(seqs), maxp), -1, np.int32)
    off = 0
    for r, p in enumerate(pages):
        pt[r, :len(p)] = np.arange(off, off + len(p))
        off += len(p)
    q = f32(w.q)[seqs]
    o_ref, lse_ref = oracle.decode_paged(q, kc, vc, pt, lens[seqs], w.scale)
    assert_close(errors(f32(o)[seqs], o_ref, f32(lse)[seqs], lse_ref))
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
