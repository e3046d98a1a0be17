// prefill_simt.cuh -- fp32 prefill attention on the CUDA cores (no tensor
// cores), for fp32 inputs.
//
// One CTA owns a tile of 64 query rows of one (sequence, query head) and
// streams the sequence's keys and values through shared memory 64 at a time,
// keeping the online-softmax state per row ("Donanıma Duyarlı Algoritma
// Tasarımı: FlashAttention", section "Online Softmax Prensibi"): a running
// maximum M and sum L, and the output rescaled by exp(M_old - M_new) whenever
// the maximum grows, so that no score row is ever written to device memory.
// Exponentials are taken base 2 with log2(e) folded into the scale; the output
// is divided by L once at the end and LSE = (M + log2 L) * ln 2.
//
// Thread map: 256 threads, four per query row.  Thread (row r, quarter c)
// computes the scores of keys c, c+4, ... of each 64-key tile, and owns the
// output columns [c*d/4, (c+1)*d/4) of its row.
#pragma once

#include "ptx.cuh"

namespace attn07 {

constexpr int kSimtBM = 64;   // query rows per CTA
constexpr int kSimtBN = 64;   // keys per tile
constexpr int kSimtThreads = 256;
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

__global__ void __launch_bounds__(kSimtThreads)
prefill_simt_kernel(const SimtParams p) {
    extern __shared__ __align__(16) float smem_f[];
    const int dp = p.d + 4;  // padded row length (floats)
    float *Qs = smem_f;                          // [64][dp]
    float *Ks = Qs + kSimtBM * dp;               // [64][dp]
    float *Vs = Ks + kSimtBN * dp;               // [64][dp]
    float *Ps = Vs + kSimtBN * dp;               // [64][68]

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
    const int r = tid >> 2;     // query row in tile
    const int c4 = tid & 3;     // quarter
    const int d = p.d;
    const int dq = d >> 2;      // output columns per thread
    const int nvec = d >> 2;    // float4 per row

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
    float acc[kSimtMaxD / 4];
#pragma unroll
    for (int c = 0; c < kSimtMaxD / 4; ++c) acc[c] = 0.f;

    const int qi = row0 + r;  // this thread's query position
    int kv_end = len;
    if (p.causal) kv_end = min(len, row0 + kSimtBM);

    for (int kv0 = 0; kv0 < kv_end; kv0 += kSimtBN) {
        __syncthreads();
        for (int idx = tid; idx < kSimtBN * nvec; idx += kSimtThreads) {
            const int rr = idx / nvec, cv = idx % nvec;
            float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
            if (kv0 + rr < len) {
                const int64_t off = ((int64_t)(start + kv0 + rr) * p.Hkv + g) * d + cv * 4;
                kk = *reinterpret_cast<const float4 *>(p.k + off);
                vv = *reinterpret_cast<const float4 *>(p.v + off);
            }
            *reinterpret_cast<float4 *>(Ks + rr * dp + cv * 4) = kk;
            *reinterpret_cast<float4 *>(Vs + rr * dp + cv * 4) = vv;
        }
        __syncthreads();

        // scores of keys c4 + 4*jj
        float s[kSimtBN / 4];
        float tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kSimtBN / 4; ++jj) {
            const int j = c4 + 4 * jj;
            const float *qr = Qs + r * dp;
            const float *kr = Ks + j * dp;
            float a = 0.f;
            for (int c = 0; c < d; c += 4) {
                const float4 qa = *reinterpret_cast<const float4 *>(qr + c);
                const float4 ka = *reinterpret_cast<const float4 *>(kr + c);
                a = fmaf(qa.x, ka.x, a);
                a = fmaf(qa.y, ka.y, a);
                a = fmaf(qa.z, ka.z, a);
                a = fmaf(qa.w, ka.w, a);
            }
            const int kj = kv0 + j;
            const bool ok = kj < len && (!p.causal || kj <= qi);
            s[jj] = ok ? a : -INFINITY;
            tmax = fmaxf(tmax, s[jj]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m, tmax);
        // a row with no allowed key yet keeps m = -inf; shift by 0 then
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2(m - m_use);
        float tsum = 0.f;
#pragma unroll
        for (int jj = 0; jj < kSimtBN / 4; ++jj) {
            const float pj = ex2(s[jj] - m_use);
            tsum += pj;
            Ps[r * (kSimtBN + 4) + c4 + 4 * jj] = pj;
        }
        tsum += __shfl_xor_sync(0xffffffffu, tsum, 1);
        tsum += __shfl_xor_sync(0xffffffffu, tsum, 2);
        l = l * alpha + tsum;
        m = m_new;
        __syncwarp();
        // O = O * alpha + P V over this thread's columns
        const int cbase = c4 * dq;
#pragma unroll
        for (int c = 0; c < kSimtMaxD / 4; ++c)
            if (c < dq) acc[c] *= alpha;
        const int jmax = min(kSimtBN, kv_end - kv0);
        for (int j = 0; j < jmax; ++j) {
            const float pj = Ps[r * (kSimtBN + 4) + j];
            const float *vr = Vs + j * dp + cbase;
#pragma unroll
            for (int c = 0; c < kSimtMaxD / 4; c += 4) {
                if (c < dq) {
                    const float4 va = *reinterpret_cast<const float4 *>(vr + c);
                    acc[c] = fmaf(pj, va.x, acc[c]);
                    acc[c + 1] = fmaf(pj, va.y, acc[c + 1]);
                    acc[c + 2] = fmaf(pj, va.z, acc[c + 2]);
                    acc[c + 3] = fmaf(pj, va.w, acc[c + 3]);
                }
            }
        }
    }

    if (qi < len) {
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        float *orow = p.o + ((int64_t)(start + qi) * p.Hq + h) * d + c4 * dq;
#pragma unroll
        for (int c = 0; c < kSimtMaxD / 4; c += 4) {
            if (c < dq) {
                *reinterpret_cast<float4 *>(orow + c) =
                    make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv);
            }
        }
        if (p.lse && c4 == 0) {
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

}  // namespace attn07
