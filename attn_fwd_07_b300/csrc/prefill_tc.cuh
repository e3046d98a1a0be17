// prefill_tc.cuh -- bf16 prefill attention on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for sm_103a.
//
// Method ("Donanıma Duyarlı Algoritma Tasarımı: FlashAttention",
// fatihsoysal.com): the attention formula of section "Transformer Mimarisi ve
// Self-Attention Mekanizması" is computed tile by tile in on-chip memory
// (section "FlashAttention'ın Temelleri"), with the online softmax of section
// "Online Softmax Prensibi" (running row maximum M and sum L), so the N x N
// score matrix never reaches device memory.  As in section "FlashAttention-2:
// Optimizasyonlar ve İyileştirmeler", each CTA owns a block of 128 query rows
// of one (sequence, query head) and streams all of that head's keys and values,
// loading the next block while the current one is computed.
//
// Work of one CTA (one 128-row query tile):
//   warp 4  (TMA)      loads the Q tile once, then K_j and V_j (128 keys each)
//                      into two 3-stage shared-memory rings (128-byte swizzle)
//   warp 5  (MMA)      one thread issues tcgen05.mma:
//                        S_j = Q K_j^T       (128x128, K = d) into TMEM buffer j%2
//                        O  += P_j V_j       (P_j read from TMEM, 128 x d, K = 128)
//                      issuing S_{j+1} before waiting for P_j, so the tensor core
//                      computes the next scores while the softmax warps work
//   warps 0-3 (softmax) one thread per query row: load the row of S_j from TMEM,
//                      mask (causal diagonal / sequence end), update the running
//                      maximum, P = 2^(S*scale*log2e - M) rounded to bf16, add the
//                      row sum of the rounded P into L, write P into TMEM, then the
//                      epilogue O / L -> bf16.
//
// Rescaling: the row maximum used for the exponent is only moved when the new
// maximum exceeds it by more than 8 (log2 units).  Until then P may reach
// 2^8, which fp32 and bf16 hold exactly in range; the output and the sum are
// always scaled consistently, so the result is the same exact softmax.  When it
// moves, O (in TMEM) and L are multiplied by 2^(M_old - M_new), which is the
// output rescaling that accompanies the online softmax.
//
// Tensor memory (512 columns of 128 lanes x 32 bit):
//   [0,128) S buffer 0, [128,256) S buffer 1, [256,256+d) O,
//   [384,448) P buffer 0, [448,512) P buffer 1 (128 bf16 per row, packed in pairs)
#pragma once

#include "ptx.cuh"

namespace attn07 {

struct PrefillParams {
    __nv_bfloat16 *o;
    float *lse;
    const int32_t *cu_seqlens;  // varlen: [num_seqs + 1]; null for the dense batch
    unsigned *status;
    int N;          // dense: tokens per sequence
    int nseq;       // dense: B; varlen: num_seqs
    int total;      // varlen: total tokens
    int Hq, Hkv;
    int ntiles;     // query tiles per sequence (of the longest sequence)
    int causal;
    float scale_log2;
};

template <int D>
struct PrefillCfg {
    static constexpr int BM = 128;
    static constexpr int BN = 128;
    static constexpr int NH = D / 64;                     // 64-column halves of a row
    static constexpr uint32_t HALF = 128u * 128u;         // one [128 rows][64] bf16 half: 16 KB
    static constexpr uint32_t TILE = NH * HALF;
    static constexpr int SK = (D == 128) ? 3 : 4;         // K ring stages
    static constexpr int SV = SK;                         // V ring stages
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = TILE;
    static constexpr uint32_t OFF_V = OFF_K + SK * TILE;
    static constexpr uint32_t OFF_CTRL = OFF_V + SV * TILE;
    static constexpr uint32_t CTRL_BYTES = 512;
    static constexpr size_t SMEM = 1024 + OFF_CTRL + CTRL_BYTES;
    // TMEM columns
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256, COL_P0 = 384, COL_P1 = 448;
    static constexpr int THREADS = 192;
};

// barrier slots inside the control block (8 bytes each)
enum : uint32_t {
    BAR_Q = 0,
    BAR_KFULL = 1,    // +s, s < 4
    BAR_KEMPTY = 5,   // +s
    BAR_VFULL = 9,    // +s
    BAR_VEMPTY = 13,  // +s
    BAR_SFULL = 17,   // +b, b < 2
    BAR_SEMPTY = 19,
    BAR_PFULL = 21,
    BAR_PVDONE = 23,
    BAR_DRAIN = 25,
    BAR_COUNT = 26
};

template <int D>
__global__ void __launch_bounds__(192, 1)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t pf_smem_raw[];

    // ---- work item: heaviest query tiles first, heads fastest
    const int units = p.Hq * p.nseq;
    const int tile = p.ntiles - 1 - (int)(blockIdx.x / units);
    const int rem = (int)(blockIdx.x % units);
    const int h = rem % p.Hq;
    const int sq = rem / p.Hq;
    const int g = h / (p.Hq / p.Hkv);
    int tok0, len, batch;
    if (p.cu_seqlens) {
        tok0 = p.cu_seqlens[sq];
        len = p.cu_seqlens[sq + 1] - tok0;
        batch = 0;
    } else {
        tok0 = 0;
        len = p.N;
        batch = sq;
    }
    if (tile < 0 || tile * C::BM >= len) return;  // uniform: nothing to do
    const int nkv_all = (len + C::BN - 1) / C::BN;
    const int n_kv = p.causal ? min(tile + 1, nkv_all) : nkv_all;

    const uint32_t raw = smem_u32(pf_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = pf_smem_raw + (base - raw);
    const uint32_t ctrl = base + C::OFF_CTRL;
    uint8_t *ctrl_ptr = base_ptr + C::OFF_CTRL;
    auto bar = [&](uint32_t i) { return ctrl + 8u * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(ctrl_ptr + 8 * BAR_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl_ptr + 8 * BAR_COUNT + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 128) {
        mbar_init(bar(BAR_Q), 1);
        for (int s = 0; s < C::SK; ++s) {
            mbar_init(bar(BAR_KFULL + s), 1);
            mbar_init(bar(BAR_KEMPTY + s), 1);
        }
        for (int s = 0; s < C::SV; ++s) {
            mbar_init(bar(BAR_VFULL + s), 1);
            mbar_init(bar(BAR_VEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(BAR_SFULL + b), 1);
            mbar_init(bar(BAR_SEMPTY + b), 4);
            mbar_init(bar(BAR_PFULL + b), 4);
            mbar_init(bar(BAR_PVDONE + b), 1);
        }
        mbar_init(bar(BAR_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(ctrl + 8 * BAR_COUNT, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ============================ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            const int qrow = tok0 + tile * C::BM;
            mbar_arrive_expect_tx(bar(BAR_Q), C::TILE);
#pragma unroll
            for (int hf = 0; hf < C::NH; ++hf)
                tma_load_4d(base + C::OFF_Q + hf * C::HALF, &tmQ, bar(BAR_Q), hf * 64, h, qrow,
                            batch, pol_q);
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int kvrow = tok0 + j * C::BN;
                const int sk = j % C::SK;
                if (!mbar_wait(bar(BAR_KEMPTY + sk), ((uint32_t)(j / C::SK) & 1u) ^ 1u, p.status,
                               abort_flag))
                    break;
                mbar_arrive_expect_tx(bar(BAR_KFULL + sk), C::TILE);
#pragma unroll
                for (int hf = 0; hf < C::NH; ++hf)
                    tma_load_4d(base + C::OFF_K + sk * C::TILE + hf * C::HALF, &tmK,
                                bar(BAR_KFULL + sk), hf * 64, g, kvrow, batch, pol_kv);
                issued_k = j + 1;
                const int sv = j % C::SV;
                if (!mbar_wait(bar(BAR_VEMPTY + sv), ((uint32_t)(j / C::SV) & 1u) ^ 1u, p.status,
                               abort_flag))
                    break;
                mbar_arrive_expect_tx(bar(BAR_VFULL + sv), C::TILE);
#pragma unroll
                for (int hf = 0; hf < C::NH; ++hf)
                    tma_load_4d(base + C::OFF_V + sv * C::TILE + hf * C::HALF, &tmV,
                                bar(BAR_VFULL + sv), hf * 64, g, kvrow, batch, pol_kv);
                issued_v = j + 1;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                for (int j = max(0, issued_k - C::SK); j < issued_k; ++j)
                    mbar_wait(bar(BAR_KFULL + j % C::SK), (uint32_t)(j / C::SK) & 1u, p.status,
                              nullptr);
                for (int j = max(0, issued_v - C::SV); j < issued_v; ++j)
                    mbar_wait(bar(BAR_VFULL + j % C::SV), (uint32_t)(j / C::SV) & 1u, p.status,
                              nullptr);
                mbar_wait(bar(BAR_Q), 0u, p.status, nullptr);
            }
        }
    } else if (warp == 5) {
        // ============================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 64, 0, 1);
            bool ok = mbar_wait(bar(BAR_Q), 0u, p.status, abort_flag);
            auto issue_qk = [&](int j) -> bool {
                const int sk = j % C::SK;
                const int sb = j & 1;
                if (!mbar_wait(bar(BAR_KFULL + sk), (uint32_t)(j / C::SK) & 1u, p.status,
                               abort_flag))
                    return false;
                if (!mbar_wait(bar(BAR_SEMPTY + sb), ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status,
                               abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t qb = base + C::OFF_Q;
                const uint32_t kb = base + C::OFF_K + sk * C::TILE;
                const uint32_t dcol = tmem + (sb ? C::COL_S1 : C::COL_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * C::HALF + (uint32_t)(kk & 3) * 32u;
                    tc_mma_ss(dcol, smem_desc_sw128(qb + off, 1024, 1024),
                              smem_desc_sw128(kb + off, 1024, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(BAR_SFULL + sb));
                tc_commit(bar(BAR_KEMPTY + sk));
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv && !issue_qk(j + 1)) break;
                const int sb = j & 1;
                const int sv = j % C::SV;
                if (!mbar_wait(bar(BAR_PFULL + sb), (uint32_t)(j >> 1) & 1u, p.status, abort_flag))
                    break;
                if (!mbar_wait(bar(BAR_VFULL + sv), (uint32_t)(j / C::SV) & 1u, p.status,
                               abort_flag))
                    break;
                tc_fence_after();
                const uint32_t vb = base + C::OFF_V + sv * C::TILE;
                const uint32_t pcol = tmem + (sb ? C::COL_P1 : C::COL_P0);
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
#pragma unroll
                    for (int hf = 0; hf < C::NH; ++hf) {
                        tc_mma_ts(tmem + C::COL_O + hf * 64, pcol + kk * 8,
                                  smem_desc_sw128(vb + hf * C::HALF + kk * 2048u, 1024, 1024),
                                  idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                tc_commit(bar(BAR_PVDONE + sb));
                tc_commit(bar(BAR_VEMPTY + sv));
            }
            // all issued MMAs complete before TMEM is released
            tc_commit(bar(BAR_DRAIN));
            mbar_wait(bar(BAR_DRAIN), 0u, p.status, nullptr);
        }
    } else {
        // ============================ softmax warps 0-3: thread = query row
        const int r = threadIdx.x;                 // row in tile, 0..127
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int qpos = tile * C::BM + r;         // position within the sequence
        float m_ref = -INFINITY;                   // log2 units, scaled
        float l = 0.f;                             // sum of P (fp32) -> LSE
        float lr = 0.f;                            // sum of bf16-rounded P -> normalises O
        const float sl2 = p.scale_log2;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            ok = mbar_wait(bar(BAR_SFULL + sb), (uint32_t)(j >> 1) & 1u, p.status, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[128];
            const uint32_t scol = tmem + lane_base + (sb ? C::COL_S1 : C::COL_S0);
            tmem_ld32(scol + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
            tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_SEMPTY + sb));

            float *s = reinterpret_cast<float *>(sr);
            const int kv0 = j * C::BN;
            const bool tail = kv0 + C::BN > len;
            const bool diag = p.causal && (kv0 + C::BN > tile * C::BM);
            if (tail || diag) {
                const int lim = p.causal ? min(len - 1, qpos) : (len - 1);  // last allowed key
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (kv0 + c > lim) s[c] = -INFINITY;
            }
            // row maximum: eight independent 3-input max chains
            float mxa[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mxa[i] = fmax3(s[i], s[i + 8], s[i + 16]);
#pragma unroll
            for (int c = 24; c + 16 <= 120; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) mxa[i] = fmax3(mxa[i], s[c + i], s[c + 8 + i]);
#pragma unroll
            for (int i = 0; i < 8; ++i) mxa[i] = fmaxf(mxa[i], s[120 + i]);
            const float mx = fmax3(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5]),
                                   fmaxf(mxa[6], mxa[7]));
            const float m_new = fmaxf(m_ref, mx * sl2);
            const bool need = m_new > m_ref + 8.0f;
            if (need && j == 0) {
                m_ref = m_new;
            }
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                const float alpha = need ? ex2(m_ref - m_new) : 1.0f;
                if (need) {
                    l *= alpha;
                    lr *= alpha;
                    m_ref = m_new;
                }
                // O must hold PV_{j-1} before it is rescaled
                const int pj = j - 1;
                ok = mbar_wait(bar(BAR_PVDONE + (pj & 1)), (uint32_t)(pj >> 1) & 1u, p.status,
                               abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t orr[32];
                    tmem_ld32(tmem + lane_base + C::COL_O + c, orr);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                    tmem_st16(tmem + lane_base + C::COL_O + c,
                              *reinterpret_cast<uint32_t(*)[16]>(&orr[0]));
                    tmem_st16(tmem + lane_base + C::COL_O + c + 16,
                              *reinterpret_cast<uint32_t(*)[16]>(&orr[16]));
                }
                tc_wait_st();
            }
            const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
            uint32_t pk[64];
            // P = 2^(s*scale*log2e - M); the exact row sum feeds the log-sum-exp, and the
            // row sum of the bf16-rounded P (the values the PV product uses) normalises O,
            // so O / L stays an exact convex combination of V rows
            float le[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            float lq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
                float t0, t1;
                ffma2(t0, t1, s[c], s[c + 1], sl2, sl2, -m_use, -m_use);
                const float p0 = ex2(t0);
                const float p1 = ex2(t1);
                const uint32_t pp = pack_bf16(p0, p1);
                const int a = (c >> 1) & 3;
                fadd2(le[2 * a], le[2 * a + 1], p0, p1);
                add_bf16x2_to(lq[a], pp);
                pk[c >> 1] = pp;
            }
            l += ((le[0] + le[1]) + (le[2] + le[3])) + ((le[4] + le[5]) + (le[6] + le[7]));
            lr += (lq[0] + lq[1]) + (lq[2] + lq[3]);
            if (j >= 2) {
                // P buffer sb was last read by PV_{j-2}
                ok = mbar_wait(bar(BAR_PVDONE + sb), (uint32_t)((j - 2) >> 1) & 1u, p.status,
                               abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            const uint32_t pcol = tmem + lane_base + (sb ? C::COL_P1 : C::COL_P0);
            tmem_st16(pcol + 0, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
            tmem_st16(pcol + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
            tmem_st16(pcol + 32, *reinterpret_cast<uint32_t(*)[16]>(&pk[32]));
            tmem_st16(pcol + 48, *reinterpret_cast<uint32_t(*)[16]>(&pk[48]));
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_PFULL + sb));
        }
        if (ok) {
            // ---- epilogue: O / L -> bf16, LSE
            const int last = n_kv - 1;
            ok = mbar_wait(bar(BAR_PVDONE + (last & 1)), (uint32_t)(last >> 1) & 1u, p.status,
                           abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                const bool row_ok = qpos < len;
                const float inv = (lr > 0.f) ? 1.f / lr : 0.f;
                const long long tok = (long long)tok0 + qpos;
                __nv_bfloat16 *orow =
                    p.o + ((p.cu_seqlens ? tok : (long long)batch * p.N + qpos) * p.Hq + h) * D;
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t orr[32];
                    tmem_ld32(tmem + lane_base + C::COL_O + c, orr);
                    tc_wait_ld();
                    uint32_t pkd[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pkd[e] = pack_bf16(__uint_as_float(orr[2 * e]) * inv,
                                           __uint_as_float(orr[2 * e + 1]) * inv);
                    if (row_ok) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pkd[4 * e], pkd[4 * e + 1], pkd[4 * e + 2],
                                                pkd[4 * e + 3]);
                    }
                }
                if (row_ok && p.lse) {
                    const float lse = (l > 0.f) ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
                    const long long idx = p.cu_seqlens ? (long long)h * p.total + tok
                                                       : ((long long)batch * p.Hq + h) * p.N + qpos;
                    p.lse[idx] = lse;
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace attn07
