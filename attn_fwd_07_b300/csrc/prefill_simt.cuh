// prefill_simt.cuh -- fp32 prefill attention on the CUDA cores (no tensor
// cores), for fp32 inputs.
//
// A CTA owns a tile of query rows of one (sequence, query head) and streams the
// sequence's keys and values through shared memory 64 at a time, keeping the
// online-softmax state per row ("Donanıma Duyarlı Algoritma Tasarımı:
// FlashAttention", section "Online Softmax Prensibi"): a running maximum M and
// sum L, and the output rescaled by exp(M_old - M_new) whenever the maximum
// grows, so that no score row is ever written to device memory.  Exponentials
// are taken base 2 with log2(e) folded into the scale; the output is divided by
// L once at the end and LSE = (M + log2 L) * ln 2.
//
// Two thread maps, the tile height chosen per launch (the page's item on block
// sizes chosen per hardware and sequence length, section "FlashAttention-2:
// Optimizasyonlar ve İyileştirmeler"):
// - prefill_simt_kernel: 16 rows per CTA, 16 threads per row.  Each K/V tile
//   loaded into shared memory serves 16 rows: the choice when the launch has
//   enough CTAs to fill the GPU.
// - prefill_simt_rows_kernel<4> and <2>: 4 or 2 rows per CTA, 64 or 128 threads
//   per row, for launches that would leave most SMs idle with 16-row tiles (N = 256
//   on one head is 16 such CTAs, 64 of 4 rows or 128 of 2 rows).
#pragma once

#include "ptx.cuh"

namespace attn07 {

constexpr int kSimtBM = 16;   // query rows per CTA (prefill_simt_kernel)
constexpr int kSimtBN = 64;   // keys per tile
constexpr int kSimtTPR = 16;  // threads per query row (prefill_simt_kernel)
constexpr int kSimtThreads = kSimtBM * kSimtTPR;
constexpr int kSimtMaxD = 128;

struct SimtParams {
    const float *q;
    const float *k;
    const float *v;
    float *o;
    float *lse;
    const int32_t *cu_seqlens;  // null: dense batch of fixed-length sequences
    int N;                      // dense: tokens per sequence
    int total;                  // varlen: total tokens (lse row stride)
    int Hq, Hkv, d;
    int causal;
    float scale_log2;           // scale * log2(e)
};

// 16 rows per CTA, 256 threads, sixteen per query row.  Thread (row r, lane
// c16 of its row) computes the scores of keys c16, c16+16, c16+32, c16+48 of each
// 64-key tile and owns the output columns 4 ch .. 4 ch + 3 of its row for ch = c16
// and c16 + 16 (those below d / 4); a row's sixteen threads are one half of a warp,
// so the row maximum and sum are half-warp shuffles.
__global__ void __launch_bounds__(kSimtThreads)
prefill_simt_kernel(const SimtParams p) {
    extern __shared__ __align__(16) float smem_f[];
    const int dp = p.d + 4;  // padded row length (floats)
    float *Qs = smem_f;                          // [16][dp]
    float *Ks = Qs + kSimtBM * dp;               // [64][dp]
    float *Vs = Ks + kSimtBN * dp;               // [64][dp]
    float *Ps = Vs + kSimtBN * dp;               // [16][68]

    const int tile = blockIdx.x;
    const int h = blockIdx.y;
    const int seq = blockIdx.z;
    const int g = h / (p.Hq / p.Hkv);

    int start, len;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[seq];
        len = p.cu_seqlens[seq + 1] - start;
    } else {
        start = seq * p.N;
        len = p.N;
    }
    const int row0 = tile * kSimtBM;
    if (row0 >= len) return;

    const int tid = threadIdx.x;
    const int r = tid / kSimtTPR;   // query row in tile
    const int c16 = tid % kSimtTPR; // lane within the row
    const int d = p.d;
    const int nvec = d >> 2;        // float4 per row (at most 32: two per thread)

    // Q tile, pre-scaled by scale*log2(e) so scores come out in log2 units.
    for (int idx = tid; idx < kSimtBM * nvec; idx += kSimtThreads) {
        const int rr = idx / nvec, cv = idx % nvec;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + rr < len) {
            val = *reinterpret_cast<const float4 *>(
                p.q + ((int64_t)(start + row0 + rr) * p.Hq + h) * d + cv * 4);
            val.x *= p.scale_log2; val.y *= p.scale_log2;
            val.z *= p.scale_log2; val.w *= p.scale_log2;
        }
        *reinterpret_cast<float4 *>(Qs + rr * dp + cv * 4) = val;
    }

    float m = -INFINITY, l = 0.f;
    float acc[8];  // columns 4 (c16 + 16 i) + e, i < 2, e < 4
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;

    const int qi = row0 + r;  // this thread's query position
    int kv_end = len;
    if (p.causal) kv_end = min(len, row0 + kSimtBM);
    constexpr int KPT = kSimtBN / kSimtTPR;  // keys per thread per tile

    // the K and V tiles pass through registers: each thread's share of the next tile
    // is loaded from device memory while the current one is computed on
    constexpr int kMaxVec = kSimtBN * kSimtMaxD / 4 / kSimtThreads;  // float4 per thread
    float4 pk[kMaxVec], pv[kMaxVec];
    auto fetch = [&](int t0) {
#pragma unroll
        for (int i = 0; i < kMaxVec; ++i) {
            const int idx = tid + kSimtThreads * i;
            const int rr = idx / nvec, cv = idx % nvec;
            pk[i] = pv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < kSimtBN * nvec && t0 + rr < len) {
                const int64_t off = ((int64_t)(start + t0 + rr) * p.Hkv + g) * d + cv * 4;
                pk[i] = *reinterpret_cast<const float4 *>(p.k + off);
                pv[i] = *reinterpret_cast<const float4 *>(p.v + off);
            }
        }
    };
    fetch(0);
    for (int kv0 = 0; kv0 < kv_end; kv0 += kSimtBN) {
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kMaxVec; ++i) {
            const int idx = tid + kSimtThreads * i;
            if (idx < kSimtBN * nvec) {
                const int rr = idx / nvec, cv = idx % nvec;
                *reinterpret_cast<float4 *>(Ks + rr * dp + cv * 4) = pk[i];
                *reinterpret_cast<float4 *>(Vs + rr * dp + cv * 4) = pv[i];
            }
        }
        __syncthreads();
        if (kv0 + kSimtBN < kv_end) fetch(kv0 + kSimtBN);

        // scores of keys c16 + 16*jj: four independent dot products over d
        float s[KPT] = {0.f, 0.f, 0.f, 0.f};
        const float *qr = Qs + r * dp;
#pragma unroll 4
        for (int c = 0; c < d; c += 4) {
            const float4 qa = *reinterpret_cast<const float4 *>(qr + c);
#pragma unroll
            for (int jj = 0; jj < KPT; ++jj) {
                const float4 ka =
                    *reinterpret_cast<const float4 *>(Ks + (c16 + kSimtTPR * jj) * dp + c);
                s[jj] = fmaf(qa.x, ka.x, s[jj]);
                s[jj] = fmaf(qa.y, ka.y, s[jj]);
                s[jj] = fmaf(qa.z, ka.z, s[jj]);
                s[jj] = fmaf(qa.w, ka.w, s[jj]);
            }
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < KPT; ++jj) {
            const int kj = kv0 + c16 + kSimtTPR * jj;
            const bool ok = kj < len && (!p.causal || kj <= qi);
            s[jj] = ok ? s[jj] : -INFINITY;
            tmax = fmaxf(tmax, s[jj]);
        }
#pragma unroll
        for (int o = kSimtTPR / 2; o > 0; o >>= 1)
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
        const float m_new = fmaxf(m, tmax);
        // a row with no allowed key yet keeps m = -inf; shift by 0 then
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m - m_use);
        float tsum = 0.f;
#pragma unroll
        for (int jj = 0; jj < KPT; ++jj) {
            const float pj = ex2(s[jj] - m_use);
            tsum += pj;
            Ps[r * (kSimtBN + 4) + c16 + kSimtTPR * jj] = pj;
        }
#pragma unroll
        for (int o = kSimtTPR / 2; o > 0; o >>= 1)
            tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
        l = l * alpha + tsum;
        m = m_new;
        __syncwarp();  // (a row's P is written and read by its own half-warp)
        // O = O * alpha + P V over this thread's columns
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] *= alpha;
        const int jmax = min(kSimtBN, kv_end - kv0);
#pragma unroll 4
        for (int j = 0; j < jmax; ++j) {
            const float pj = Ps[r * (kSimtBN + 4) + j];
            const float *vr = Vs + j * dp;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int ch = c16 + kSimtTPR * i;
                if (ch < nvec) {
                    const float4 va = *reinterpret_cast<const float4 *>(vr + 4 * ch);
                    acc[4 * i] = fmaf(pj, va.x, acc[4 * i]);
                    acc[4 * i + 1] = fmaf(pj, va.y, acc[4 * i + 1]);
                    acc[4 * i + 2] = fmaf(pj, va.z, acc[4 * i + 2]);
                    acc[4 * i + 3] = fmaf(pj, va.w, acc[4 * i + 3]);
                }
            }
        }
    }

    if (qi < len) {
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        float *orow = p.o + ((int64_t)(start + qi) * p.Hq + h) * d;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int ch = c16 + kSimtTPR * i;
            if (ch < nvec) {
                *reinterpret_cast<float4 *>(orow + 4 * ch) =
                    make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv,
                                acc[4 * i + 3] * inv);
            }
        }
        if (p.lse && c16 == 0) {
            const float lse = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
            int64_t idx;
            if (p.cu_seqlens) idx = (int64_t)h * p.total + start + qi;
            else idx = ((int64_t)seq * p.Hq + h) * p.N + qi;
            p.lse[idx] = lse;
        }
    }
}

inline size_t prefill_simt_smem_bytes(int d) {
    return sizeof(float) * ((size_t)(kSimtBM + 2 * kSimtBN) * (d + 4) + kSimtBM * (kSimtBN + 4));
}

// ROWS = 4 or 2 rows per CTA, 256 threads, TPR = 64 or 128 per query row (two or
// four warps).  Thread (row r, lane c of its row):
// - scores: one key of each 64-key tile per S = TPR / 64 threads.  Each of a key's
//   threads takes every S-th float4 of the dot product over d (the row's Q a
//   warp-wide broadcast, the key rows conflict-free with the padded row length),
//   and a shuffle adds the S partial sums.
// - output: with 64 threads per row, columns c and c + 64 (those below d) over all
//   keys of the tile; with 128, column c over all keys when d > 64, else column
//   c % 64 over one half of the tile's keys (the halves added once at the end).
//   A warp's value loads are 32 consecutive words of one value row.
// The row maximum and sum are warp shuffles, then one exchange between the row's
// warps through shared memory.  (One CTA per SM: the registers hold a K/V tile's
// share and its slots' offsets.)
template <int ROWS>
__global__ void __launch_bounds__(kSimtThreads, 1)
prefill_simt_rows_kernel(const SimtParams p) {
    constexpr int TPR = kSimtThreads / ROWS;  // threads per query row
    constexpr int S = TPR / kSimtBN;          // threads per key in the scores
    constexpr int NW = TPR / 32;              // warps per row
    static_assert(S == 1 || S == 2, "64 or 128 threads per row");
    extern __shared__ __align__(16) float smem_f[];
    const int dp = p.d + 4;  // padded row length (floats)
    float *Qs = smem_f;                          // [ROWS][dp]
    float *Ks = Qs + ROWS * dp;                  // [64][dp]
    float *Vs = Ks + kSimtBN * dp;               // [64][dp]
    float *Ps = Vs + kSimtBN * dp;               // [ROWS][64]
    float *red = Ps + ROWS * kSimtBN;            // [2][ROWS][NW]: row maxima, row sums per warp
    float *half_o = red + 2 * ROWS * NW;         // [ROWS][64]: the second key half's output

    const int tile = blockIdx.x;
    const int h = blockIdx.y;
    const int seq = blockIdx.z;
    const int g = h / (p.Hq / p.Hkv);

    int start, len;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[seq];
        len = p.cu_seqlens[seq + 1] - start;
    } else {
        start = seq * p.N;
        len = p.N;
    }
    const int row0 = tile * ROWS;
    if (row0 >= len) return;

    const int tid = threadIdx.x;
    const int r = tid / TPR;         // query row in tile
    const int c = tid % TPR;         // lane within the row
    const int wr = c >> 5;           // the row's warp
    const int lane = tid & 31;
    // key of the scores and part of its dot product: with two parts, lanes l and l + 16
    // of a warp share a key, so that each 8-lane phase of a 16-byte shared-memory load
    // reads 8 different key rows (no bank conflict)
    const int kc = S == 1 ? c : (c >> 5) * 16 + (lane & 15);
    const int kp = S == 1 ? 0 : lane >> 4;
    const int d = p.d;
    const int nvec = d >> 2;         // float4 per row
    // output: column col over keys [jlo_o, jlo_o + jn_o) of each tile (second column
    // col + 64 with 64 threads per row)
    const bool split_keys = S == 2 && d <= 64;
    const int col = split_keys ? (c & 63) : c;
    const int jlo_o = split_keys ? 32 * (c >> 6) : 0;
    const int jn_o = split_keys ? 32 : kSimtBN;

    // Q tile, pre-scaled by scale*log2(e) so scores come out in log2 units.
    for (int idx = tid; idx < ROWS * nvec; idx += kSimtThreads) {
        const int rr = idx / nvec, cv = idx % nvec;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row0 + rr < len) {
            val = *reinterpret_cast<const float4 *>(
                p.q + ((int64_t)(start + row0 + rr) * p.Hq + h) * d + cv * 4);
            val.x *= p.scale_log2; val.y *= p.scale_log2;
            val.z *= p.scale_log2; val.w *= p.scale_log2;
        }
        *reinterpret_cast<float4 *>(Qs + rr * dp + cv * 4) = val;
    }

    float m = -INFINITY, l = 0.f;
    float acc0 = 0.f, acc1 = 0.f;  // output columns col and col + 64

    const int qi = row0 + r;  // this thread's query position
    int kv_end = len;
    if (p.causal) kv_end = min(len, row0 + ROWS);

    // the K and V tiles pass through registers: each thread's share of the next tile
    // is loaded from device memory while the current one is computed on (rows past
    // the sequence are zeros).  A thread's share is the same float4 slots of every
    // tile: their rows, shared-memory offsets and device offsets (relative to the
    // tile's first row) are computed once.
    constexpr int kMaxVec = kSimtBN * kSimtMaxD / 4 / kSimtThreads;  // float4 per thread
    float4 pk[kMaxVec], pv[kMaxVec];
    int vrow[kMaxVec], soff[kMaxVec], goff[kMaxVec];
#pragma unroll
    for (int i = 0; i < kMaxVec; ++i) {
        const int idx = tid + kSimtThreads * i;
        vrow[i] = kSimtBN;  // (no slot)
        soff[i] = goff[i] = 0;
        if (idx < kSimtBN * nvec) {
            const int rr = idx / nvec, cv = idx - rr * nvec;
            vrow[i] = rr;
            soff[i] = rr * dp + cv * 4;
            goff[i] = rr * p.Hkv * d + cv * 4;
        }
    }
    auto fetch = [&](int t0) {
        const int lim = min(kSimtBN, len - t0);
        const int64_t base = ((int64_t)(start + t0) * p.Hkv + g) * d;
#pragma unroll
        for (int i = 0; i < kMaxVec; ++i) {
            if (vrow[i] < lim) {
                pk[i] = *reinterpret_cast<const float4 *>(p.k + base + goff[i]);
                pv[i] = *reinterpret_cast<const float4 *>(p.v + base + goff[i]);
            } else {
                pk[i] = pv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
    fetch(0);
    for (int kv0 = 0; kv0 < kv_end; kv0 += kSimtBN) {
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kMaxVec; ++i) {
            if (vrow[i] < kSimtBN) {
                *reinterpret_cast<float4 *>(Ks + soff[i]) = pk[i];
                *reinterpret_cast<float4 *>(Vs + soff[i]) = pv[i];
            }
        }
        __syncthreads();
        if (kv0 + kSimtBN < kv_end) fetch(kv0 + kSimtBN);

        // score of key kc: four partial sums (one per float4 component) over this
        // thread's float4 groups, then the key's S parts added
        const float *qr = Qs + r * dp;
        const float *kr = Ks + kc * dp;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
        for (int cc = 4 * kp; cc < d; cc += 4 * S) {
            const float4 qa = *reinterpret_cast<const float4 *>(qr + cc);
            const float4 ka = *reinterpret_cast<const float4 *>(kr + cc);
            a0 = fmaf(qa.x, ka.x, a0);
            a1 = fmaf(qa.y, ka.y, a1);
            a2 = fmaf(qa.z, ka.z, a2);
            a3 = fmaf(qa.w, ka.w, a3);
        }
        float sc = (a0 + a1) + (a2 + a3);
        if constexpr (S == 2) sc += __shfl_xor_sync(0xffffffffu, sc, 16);
        const int kj = kv0 + kc;
        const bool ok = kj < len && (!p.causal || kj <= qi);
        const float s = ok ? sc : -INFINITY;

        // row maximum: the warp's, then the row's warps' through shared memory
        float tmax = s;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
        if (lane == 0) red[r * NW + wr] = tmax;
        __syncthreads();
        tmax = red[r * NW];
#pragma unroll
        for (int w = 1; w < NW; ++w) tmax = fmaxf(tmax, red[r * NW + w]);
        const float m_new = fmaxf(m, tmax);
        // a row with no allowed key yet keeps m = -inf; shift by 0 then
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m - m_use);
        const float pj = ex2(s - m_use);  // 0 for a masked key
        if (kp == 0) Ps[r * kSimtBN + kc] = pj;
        // (each key counted once: by the first of its S threads)
        float tsum = kp == 0 ? pj : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
        if (lane == 0) red[ROWS * NW + r * NW + wr] = tsum;
        __syncthreads();
        float rsum = red[ROWS * NW + r * NW];
#pragma unroll
        for (int w = 1; w < NW; ++w) rsum += red[ROWS * NW + r * NW + w];
        l = l * alpha + rsum;
        m = m_new;

        // O = O * alpha + P V over this thread's columns and keys.  Keys from the
        // tile's end up to the next multiple of 4 have P = 0 and finite (or
        // zero-filled) values.
        acc0 *= alpha;
        acc1 *= alpha;
        const int jmax = (min(kSimtBN, kv_end - kv0) + 3) & ~3;
        const int j1 = min(jlo_o + jn_o, jmax);
        const float *pr = Ps + r * kSimtBN;
        if (S == 1 && col + 64 < d) {
#pragma unroll 2
            for (int j = jlo_o; j < j1; j += 4) {
                const float4 p4 = *reinterpret_cast<const float4 *>(pr + j);
                const float *vr = Vs + j * dp + col;
                acc0 = fmaf(p4.x, vr[0], acc0);
                acc1 = fmaf(p4.x, vr[64], acc1);
                acc0 = fmaf(p4.y, vr[dp], acc0);
                acc1 = fmaf(p4.y, vr[dp + 64], acc1);
                acc0 = fmaf(p4.z, vr[2 * dp], acc0);
                acc1 = fmaf(p4.z, vr[2 * dp + 64], acc1);
                acc0 = fmaf(p4.w, vr[3 * dp], acc0);
                acc1 = fmaf(p4.w, vr[3 * dp + 64], acc1);
            }
        } else if (col < d) {
            // (two chains, even and odd keys)
#pragma unroll 2
            for (int j = jlo_o; j < j1; j += 4) {
                const float4 p4 = *reinterpret_cast<const float4 *>(pr + j);
                const float *vr = Vs + j * dp + col;
                acc0 = fmaf(p4.x, vr[0], acc0);
                acc1 = fmaf(p4.y, vr[dp], acc1);
                acc0 = fmaf(p4.z, vr[2 * dp], acc0);
                acc1 = fmaf(p4.w, vr[3 * dp], acc1);
            }
        }
    }

    // one column's partial outputs added: the even and odd key chains, and (keys split
    // between two threads) the second half's through shared memory
    float out0 = acc0, out1 = acc1;
    if (!(S == 1 && col + 64 < d)) {
        out0 = acc0 + acc1;
        out1 = 0.f;
    }
    if (split_keys) {
        if (jlo_o != 0 && col < d) half_o[r * kSimtBN + col] = out0;
        __syncthreads();
        if (jlo_o == 0 && col < d) out0 += half_o[r * kSimtBN + col];
    }
    if (qi < len && jlo_o == 0) {
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        float *orow = p.o + ((int64_t)(start + qi) * p.Hq + h) * d;
        if (col < d) orow[col] = out0 * inv;
        if (S == 1 && col + 64 < d) orow[col + 64] = out1 * inv;
        if (p.lse && c == 0) {
            const float lse = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
            int64_t idx;
            if (p.cu_seqlens) idx = (int64_t)h * p.total + start + qi;
            else idx = ((int64_t)seq * p.Hq + h) * p.N + qi;
            p.lse[idx] = lse;
        }
    }
}

inline size_t prefill_simt_rows_smem_bytes(int rows, int d) {
    const int nw = kSimtThreads / rows / 32;
    return sizeof(float) * ((size_t)(rows + 2 * kSimtBN) * (d + 4) + 2 * (size_t)rows * kSimtBN +
                            2 * (size_t)rows * nw);
}

}  // namespace attn07
