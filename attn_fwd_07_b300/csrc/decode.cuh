// decode.cuh -- decode attention against a paged key/value cache.
//
// What it computes: for every sequence b, one new query per query head
// attends to all seq_lens[b] cached keys/values of its key/value head
// (yapayzekasozluk.tr "attention" tag page, entry "KV Cache": cached keys and
// values, grouped query heads sharing a key/value head, the cache held in
// fixed-size pages).
//
// How (two kernels):
//   decode_split_kernel  The cache pages of all sequences, taken in order
//       (sequence 0's pages, then sequence 1's, ...), are cut into gridDim.x
//       equal contiguous ranges, one per CTA, so every CTA streams the same
//       number of pages whatever the length mix.  Within its range a CTA walks
//       one or more "segments" (the part of one sequence inside the range) and
//       keeps the online-softmax state ("Donanıma Duyarlı Algoritma Tasarımı:
//       FlashAttention", section "Online Softmax Prensibi": running maximum,
//       running sum, output rescaled when the maximum grows) per query head.
//       At the end of a segment it writes the normalised partial output and
//       its log-sum-exp to workspace slot (b + CTA index); along the
//       monotone staircase of (sequence, CTA) pairs that touch, b + c is
//       strictly increasing, so slots never collide and B + gridDim.x slots
//       suffice.
//   decode_merge_kernel  For each sequence, combines its partials by their
//       log-sum-exps: lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s
//       (the same rescaling rule, applied across key ranges), writing bf16 O
//       and fp32 LSE.
//
// Data movement: TMA copies each page -- all key/value heads, 16 tokens -- into
// a multi-stage shared-memory ring, as 128-byte-swizzled boxes of
// [head][token][64 dims] so that each head's 16 token rows are conflict-free for
// ldmatrix.  There is no producer warp: every warp walks the CTA's page stream,
// the ring is kept S pages ahead, and the warp that releases a page's stage last
// refills it with the page S further on (its id read while the page was being
// attended).  The CTA is one warp per key/value head, so two CTAs of the
// one-byte-cache (FP8 or INT8) kernels fit an SM at 128 registers a thread.
// Each warp computes S = q K^T and O += P V for its Hq/Hkv query heads with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate; the query heads fill the first
// rows of the 16-row tile).  The decode is bound by device-memory bandwidth:
// the contraction per byte is small, and the ring keeps enough bytes in flight.
#pragma once

#include "ptx.cuh"

namespace attn07 {

constexpr int kDecPage = 16;          // tokens per page (the kernel is built for it)
constexpr int kDecMaxStages = 8;
constexpr int kDecMaxHkv = 8;
constexpr int kDecMaxCtasPerSm = 2;    // the one-byte-cache kernels run two CTAs per SM

struct DecodeParams {
    const __nv_bfloat16 *q;    // [B, Hq, d]
    const int32_t *page_table; // [B, maxp]
    const int32_t *seq_lens;   // [B]
    float *part_o;             // [B + G, Hq, d]
    float *part_lse;           // [B + G, Hq]
    __nv_bfloat16 *o;          // [B, Hq, d]
    float *lse;                // [B, Hq] or null
    const float *k_scale;      // one-byte cache: [Hkv] per-head scales of K and V; else null
    const float *v_scale;
    unsigned *status;
    int B, Hq, Hkv, d, num_pages, maxp;
    int stages;
    int window;                // the query sees the last window + 1 tokens; -1: all
    float scale_log2;
};

struct DecodeStageMeta {
    int b;        // sequence
    int lo;       // first valid token slot in this page (window start)
    int ntok;     // valid token slots end here (0 if the page id was bad)
    int first;    // first page of a segment
    int last;     // last page of a segment
};

static_assert(sizeof(DecodeStageMeta) * kDecMaxStages <= 160, "stage metadata must fit");

// Shared-memory layout (offsets from a 1024-byte-aligned base):
//   stage s:  bf16 cache: K half 0 .. K half (d/64 - 1), V half 0 .. V half (d/64 - 1),
//             each [Hkv][16][64] bf16 = Hkv * 2048 bytes;
//             one-byte cache (d = 128): K, then V, each [Hkv][16][128] bytes = Hkv * 2048
//   then full[kDecMaxStages], empty[kDecMaxStages] mbarriers, meta, release counts,
//   scalars (1 KB).
__host__ __device__ inline uint32_t dec_half_bytes(int Hkv) { return (uint32_t)Hkv * 16u * 128u; }
__host__ __device__ inline uint32_t dec_stage_bytes(int Hkv, int d, bool fp8) {
    return 2u * (fp8 ? 1u : (uint32_t)(d / 64)) * dec_half_bytes(Hkv);
}
__host__ __device__ inline uint32_t dec_ctrl_bytes() { return 1024u; }
inline size_t dec_smem_bytes(int Hkv, int d, int stages, bool fp8) {
    return 1024 /* alignment slack */ + (size_t)stages * dec_stage_bytes(Hkv, d, fp8) +
           dec_ctrl_bytes();
}

// Whether seq_lens[b] is a length the page table can hold: 0 <= len <= maxp * 16.
__device__ __forceinline__ bool dec_len_ok(const DecodeParams &p, int b) {
    const int len = p.seq_lens[b];
    return len >= 0 && (long long)len <= (long long)p.maxp * kDecPage;
}

// Cached tokens of sequence b; a length outside what the page table holds counts
// as 0 (the sequence is treated as empty and its table row is never read).
__device__ __forceinline__ int dec_len(const DecodeParams &p, int b) {
    return dec_len_ok(p, b) ? p.seq_lens[b] : 0;
}

// First token the query of sequence b attends to: len - 1 - window under a
// window, else 0.
__device__ __forceinline__ int dec_first_token(const DecodeParams &p, int b) {
    const int len = dec_len(p, b);
    return (p.window >= 0 && len - 1 - p.window > 0) ? len - 1 - p.window : 0;
}

// Pages of sequence b that hold attended tokens: logical pages
// first_token / 16 .. ceil(len / 16) - 1.
__device__ __forceinline__ int dec_pages_of(const DecodeParams &p, int b) {
    const int len = dec_len(p, b);
    return len > 0 ? (len + kDecPage - 1) / kDecPage - dec_first_token(p, b) / kDecPage : 0;
}

// The CTA whose page range [c*T/G, (c+1)*T/G) holds global page x.
__host__ __device__ __forceinline__ int dec_cta_of_page(long long x, long long T, long long G) {
    return (int)(((x + 1) * G - 1) / T);
}

// Whether CTA c's page range is non-empty.  Every CTA strictly between the ones
// holding a sequence's first and last page lies inside that sequence, so for
// those CTAs "non-empty" is the same as "wrote a partial for it".
__host__ __device__ __forceinline__ bool dec_range_nonempty(long long c, long long T, long long G) {
    return (c + 1) * T / G > c * T / G;
}

// The cache's element format: bf16, or one byte with a per-head scale (FP8 E4M3 or
// INT8, value = scale[head] * byte value).
enum : int { kCacheBf16 = 0, kCacheFp8 = 1, kCacheInt8 = 2 };

// Four signed bytes (INT8) -> their values as two f16 pairs (bytes 0, 1 and bytes
// 2, 3), exactly.  An f16 whose high byte is 0x64 (biased exponent 25, i.e. 2^10)
// has unit spacing on [1024, 2048): with the low byte u it is 1024 + u.  Flipping a
// byte's sign bit gives u = v + 128 for the signed value v, so the f16 holding
// 1024 + u, minus 1152 (0x6480), is v; every step is exact.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t x, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = x ^ 0x80808080u;
    const uint32_t a = prmt(u, 0x64646464u, 0x4140u);  // bytes 0, 1 over 0x64
    const uint32_t b = prmt(u, 0x64646464u, 0x4342u);  // bytes 2, 3 over 0x64
    const uint32_t off = 0x64806480u;                  // 1152 in both halves
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(off));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(off));
}

// Four cache bytes -> their values (exactly, as f16) in two f16 pairs: bytes 0 and 1,
// bytes 2 and 3.
template <int CACHE>
__device__ __forceinline__ void dec_byte4_to_f16x2x2(uint32_t x, uint32_t &lo, uint32_t &hi) {
    if constexpr (CACHE == kCacheFp8)
        e4m3x4_to_f16x2x2(x, lo, hi);
    else
        s8x4_to_f16x2x2(x, lo, hi);
}

// One-byte cache (FP8 E4M3 or INT8 bytes).  Each consumer lane reads the bytes of
// its MMA fragments straight from the stage (the contraction's k order and the
// output's column order are permuted so that they are contiguous 16-byte chunks),
// widens them to f16 (exact for both formats) and runs the products with f16
// operands; per-head scales multiply the scores and the output.
template <int CACHE>
__global__ void __launch_bounds__(32 * kDecMaxHkv, CACHE != kCacheBf16 ? 2 : 1)
decode_split_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
    constexpr bool BYTE = CACHE != kCacheBf16;  // a one-byte cache
    extern __shared__ uint8_t dec_smem_raw[];
    const uint32_t raw = smem_u32(dec_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = dec_smem_raw + (base - raw);

    const int S = p.stages;
    const uint32_t stage_bytes = dec_stage_bytes(p.Hkv, p.d, BYTE);
    const uint32_t half_bytes = dec_half_bytes(p.Hkv);
    const int nhalf = BYTE ? 1 : p.d / 64;  // TMA boxes per tensor and page
    const uint32_t ctrl = base + (uint32_t)S * stage_bytes;
    uint8_t *ctrl_ptr = base_ptr + (size_t)S * stage_bytes;
    // control block: full[8] @0, empty[8] @64, meta[8] @128, released[8] @288,
    // n_issued[8] @320, scalars @384
    const uint32_t full0 = ctrl, empty0 = ctrl + 64;
    DecodeStageMeta *meta = reinterpret_cast<DecodeStageMeta *>(ctrl_ptr + 128);
    int *released = reinterpret_cast<int *>(ctrl_ptr + 288);   // warps done with a stage
    int *n_issued = reinterpret_cast<int *>(ctrl_ptr + 320);   // pages issued into a stage
    volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl_ptr + 384);
    int *shared_n = reinterpret_cast<int *>(ctrl_ptr + 388);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int Hkv = p.Hkv;
    const int G = gridDim.x;
    // the merge grid may be scheduled now (it waits for this grid to finish)
    grid_dependents_launch();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, Hkv);
            released[s] = 0;
            n_issued[s] = 0;
        }
        *abort_flag = 0;
        fence_barrier_init();
    }

    // ---- the total page count T: every warp sums it (a few loads per 32 sequences),
    // so that each can find this CTA's first page below without waiting for another
    long long T = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        int np = (b0 + lane < p.B) ? dec_pages_of(p, b0 + lane) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) np += __shfl_xor_sync(0xffffffffu, np, o);
        T += np;
    }
    const long long p0 = (long long)blockIdx.x * T / G;
    const int n_iter = (int)((long long)(blockIdx.x + 1) * T / G - p0);
    (void)shared_n;

    // ---- the page stream of this CTA: pages p0 .. p0 + n_iter - 1 in sequence order.
    // Every warp keeps a cursor on it; the ring is filled S pages ahead of the pages
    // being attended, the stage of page it being refilled with page it + S by the warp
    // that releases it last, with the id and sizes its own cursor holds.
    // find the sequence holding global page p0: 32 sequences at a time, the lanes'
    // page counts summed by a prefix scan and the first lane past p0 taken
    int cb = 0;               // cursor: sequence
    long long seq_start = 0;  // global index of sequence cb's first page
    int cnp = 0;              // pages of sequence cb
    bool found = n_iter == 0;
    for (int b0 = 0; !found && b0 < p.B; b0 += 32) {
        const int np_l = (b0 + lane < p.B) ? dec_pages_of(p, b0 + lane) : 0;
        long long incl = np_l;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, seq_start + incl > p0);
        if (hit) {
            const int l = __ffs(hit) - 1;
            cb = b0 + l;
            cnp = __shfl_sync(0xffffffffu, np_l, l);
            seq_start += __shfl_sync(0xffffffffu, incl, l) - cnp;
            found = true;
        } else {
            seq_start += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    // (the page counts summed above cover page p0, so this holds unless seq_lens
    // changed under the kernel; the ring is then left unfilled and the bounded waits
    // end the launch with an error)
    if (!found && warp == 0 && lane == 0) record_status(p.status, kStatusBounds);
    int clp = (int)(p0 - seq_start);                               // cursor: page of cb
    int cfp = found && n_iter > 0 ? dec_first_token(p, cb) / kDecPage : 0;  // first logical page
    int cit = 0;                                                   // cursor: page index
    // moves the cursor to the next page of the stream (empty sequences skipped)
    auto advance = [&]() {
        ++clp;
        ++cit;
        while (cit < n_iter && clp >= cnp && cb + 1 < p.B) {
            ++cb;
            clp = 0;
            cnp = dec_pages_of(p, cb);
            cfp = dec_first_token(p, cb) / kDecPage;
        }
    };
    // the cursor's page id (read by lane 0; -1 past the stream, or off the sequence's
    // pages if seq_lens changed under the kernel)
    auto cursor_id = [&]() -> int {
        return (cit < n_iter && clp < cnp) ? p.page_table[(long long)cb * p.maxp + cfp + clp]
                                           : -1;
    };
    const uint64_t pol = policy_evict_first();
    // page `cit` of the stream (id pid) into its stage: its sizes into the stage's
    // metadata, then K and V by TMA (a page id out of range is reported and the stage
    // handed over empty)
    auto issue = [&](int pid) {
        const int s = cit % S;
        const bool last_of_seq = (clp == cnp - 1);
        const bool valid = (unsigned)pid < (unsigned)p.num_pages;
        DecodeStageMeta mt;
        mt.b = cb;
        mt.ntok = valid ? (last_of_seq ? dec_len(p, cb) - (cfp + clp) * kDecPage : kDecPage) : 0;
        mt.lo = clp == 0 ? dec_first_token(p, cb) - cfp * kDecPage : 0;
        mt.first = (cit == 0 || clp == 0) ? 1 : 0;
        mt.last = (cit == n_iter - 1 || last_of_seq) ? 1 : 0;
        meta[s] = mt;
        ++n_issued[s];
        const uint32_t dst = base + (uint32_t)s * stage_bytes;
        if (valid) {
            mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes);
            for (int hf = 0; hf < nhalf; ++hf) {
                tma_load_4d(dst + hf * half_bytes, &tmK, full0 + 8 * s, hf * 64, 0, 0, pid, pol);
                tma_load_4d(dst + (nhalf + hf) * half_bytes, &tmV, full0 + 8 * s, hf * 64, 0, 0,
                            pid, pol);
            }
        } else {
            record_status(p.status, kStatusBounds);
            mbar_arrive(full0 + 8 * s);
        }
    };
    __syncthreads();  // barriers initialised
    if (found) {
        // the first S pages: warp 0 issues them; every warp moves its cursor past them
        for (int i = 0; i < S && cit < n_iter; ++i) {
            if (warp == 0 && lane == 0) {
                if (i == 0) {
                    prefetch_tmap(&tmK);
                    prefetch_tmap(&tmV);
                }
                issue(cursor_id());
            }
            advance();
        }
    }

    {
        // ================= consumers: warp g serves kv head g
        const int g = warp;
        const int Gq = p.Hq / Hkv;             // query heads per kv head (<= 8)
        const int row = lane >> 2;             // mma row = query head within group
        const int quad = lane & 3;
        const bool row_ok = row < Gq;
        const int nk = p.d / 16;               // k-steps of S = q K^T
        const int nd = p.d / 8;                // n-tiles of O

        // A fragments of q (rows 0..7).  One-byte cache: the k-slots of each 16-dim step
        // are permuted so that a lane's K bytes are contiguous -- in half hf, k-step
        // 4 hf + j takes dims 16 (2 quad + hf) + 4 j .. + 3 for this lane's slots
        // (2 quad, 2 quad + 1, 2 quad + 8, 2 quad + 9); q uses the same permutation.
        // A half's 16-byte chunks are then the even (hf = 0) or the odd ones of a key
        // row, so the two rows that share a phase of a 16-byte shared load (tokens 2i
        // and 2i + 1, whose swizzles differ in the lowest bit) fall in distinct banks.
        uint32_t qa[8][2];
        float oacc[16][4];
        // scores are q . k * scale (* the head's key scale for a one-byte cache), log2
        // units
        const float sl2 = BYTE ? p.scale_log2 * p.k_scale[g] : p.scale_log2;
        const float vsc = BYTE ? p.v_scale[g] : 1.f;
        float m_run = -INFINITY, l_run = 0.f, q_run = 0.f;
        int cur_b = 0;

        int s = 0;          // ring position (stage, phase parity), advanced by one per page
        uint32_t par = 0u;
        for (int it = 0; found && it < n_iter;
             ++it, s = (s + 1 == S) ? 0 : s + 1, par ^= (s == 0) ? 1u : 0u) {
            // the id of page it + S, which this warp issues if it releases page it last
            // (read now, used after the page)
            const int next_id = lane == 0 ? cursor_id() : 0;
            bool ok = mbar_wait(full0 + 8 * s, par, p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const DecodeStageMeta mt = meta[s];
            if (mt.first) {
                cur_b = mt.b;
                const __nv_bfloat16 *qb = p.q + ((long long)cur_b * p.Hq + g * Gq) * p.d;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    if (ks < nk && row_ok) {
                        const uint32_t *qr = reinterpret_cast<const uint32_t *>(qb + row * p.d);
                        if constexpr (BYTE) {
                            const int d0 = 32 * quad + 16 * (ks >> 2) + 4 * (ks & 3);
                            qa[ks][0] = bf16x2_to_f16x2(qr[d0 >> 1]);
                            qa[ks][1] = bf16x2_to_f16x2(qr[(d0 + 2) >> 1]);
                        } else {
                            qa[ks][0] = qr[(ks * 16 + 2 * quad) >> 1];
                            qa[ks][1] = qr[(ks * 16 + 8 + 2 * quad) >> 1];
                        }
                    } else {
                        qa[ks][0] = 0u;
                        qa[ks][1] = 0u;
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
                m_run = -INFINITY;
                l_run = 0.f;
                q_run = 0.f;
            }
            const uint32_t kst = base + (uint32_t)s * stage_bytes;
            const uint32_t vst = kst + (uint32_t)nhalf * half_bytes;
            if (mt.ntok > 0) {
                // ---- S = q K^T over the 16 tokens (two n-tiles of 8 tokens)
                float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                if constexpr (BYTE) {
                    // token 8 nt + row: one 16-byte chunk per half holds this lane's dims;
                    // odd k-steps accumulate apart (two shorter dependency chains)
                    float sodd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const uint32_t rg = (uint32_t)(g * 16 + 8 * nt + row);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const uint4 w = lds128(kst + rg * 128u +
                                                   (uint32_t)(((2 * quad + hf) ^ (int)(rg & 7u)) * 16));
                            const uint32_t wj[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                uint32_t b0, b1;
                                dec_byte4_to_f16x2x2<CACHE>(wj[j], b0, b1);
                                mma_f16_16816((j & 1) ? sodd[nt] : sacc[nt], qa[4 * hf + j][0], 0u,
                                              qa[4 * hf + j][1], 0u, b0, b1);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) sacc[nt][e] += sodd[nt][e];
                    }
                } else {
                    const int mi = lane >> 3, i = lane & 7;
                    const int tok = (mi >> 1) * 8 + i;
                    const uint32_t r = (uint32_t)(g * 16 + tok);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        if (ks < nk) {
                            const int hf = ks >> 2;
                            const int chunk = (ks & 3) * 2 + (mi & 1);
                            const uint32_t addr = kst + hf * half_bytes + r * 128u +
                                                  (uint32_t)((chunk ^ (int)(r & 7u)) * 16);
                            uint32_t b00, b01, b10, b11;
                            ldsm_x4(addr, b00, b01, b10, b11);
                            mma_bf16_16816(sacc[0], qa[ks][0], 0u, qa[ks][1], 0u, b00, b01);
                            mma_bf16_16816(sacc[1], qa[ks][0], 0u, qa[ks][1], 0u, b10, b11);
                        }
                    }
                }
                // ---- mask, online softmax (rows = query heads, 4 lanes per row)
                float sv[4];
                sv[0] = sacc[0][0] * sl2;
                sv[1] = sacc[0][1] * sl2;
                sv[2] = sacc[1][0] * sl2;
                sv[3] = sacc[1][1] * sl2;
                if (mt.ntok < kDecPage || mt.lo > 0) {  // (a full page needs no mask)
                    const int t0 = 2 * quad;
                    if (t0 >= mt.ntok || t0 < mt.lo) sv[0] = -INFINITY;
                    if (t0 + 1 >= mt.ntok || t0 + 1 < mt.lo) sv[1] = -INFINITY;
                    if (t0 + 8 >= mt.ntok || t0 + 8 < mt.lo) sv[2] = -INFINITY;
                    if (t0 + 9 >= mt.ntok || t0 + 9 < mt.lo) sv[3] = -INFINITY;
                }
                float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                // the exponent's reference maximum moves only when the row maximum exceeds
                // it by more than 8 (log2 units): until then P <= 2^8, exact in range for
                // fp32, f16 and bf16, and O and the sums need no rescaling this page
                const bool need = mx > m_run + 8.f;
                const bool any_need = __any_sync(0xffffffffu, need);
                float alpha = 1.f;
                if (any_need && need) {
                    alpha = ex2(m_run - mx);
                    m_run = mx;
                }
                const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
                float pr[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) pr[j] = ex2(sv[j] - m_use);
                // P enters the PV product as bf16 (f16 for a one-byte cache); O is normalised
                // by the sum of the same rounded values, the log-sum-exp by the exact sum
                const uint32_t pa0 = BYTE ? pack_f16(pr[0], pr[1]) : pack_bf16(pr[0], pr[1]);
                const uint32_t pa2 = BYTE ? pack_f16(pr[2], pr[3]) : pack_bf16(pr[2], pr[3]);
                float pq = BYTE ? (f16lo(pa0) + f16hi(pa0)) + (f16lo(pa2) + f16hi(pa2))
                               : (bf16lo(pa0) + bf16hi(pa0)) + (bf16lo(pa2) + bf16hi(pa2));
                float ps = (pr[0] + pr[1]) + (pr[2] + pr[3]);
                pq += __shfl_xor_sync(0xffffffffu, pq, 1);
                ps += __shfl_xor_sync(0xffffffffu, ps, 1);
                pq += __shfl_xor_sync(0xffffffffu, pq, 2);
                ps += __shfl_xor_sync(0xffffffffu, ps, 2);
                l_run = l_run * alpha + ps;   // exact sum -> log-sum-exp
                q_run = q_run * alpha + pq;   // sum of the rounded P -> normalises O
                if (!any_need) {
                    // no row of the warp moved its reference: O stands
                } else if constexpr (BYTE) {
                    // O^T tiles: columns are query heads 2 quad and 2 quad + 1, whose
                    // factors live in lanes 8 quad and 8 quad + 4
                    const float ae = __shfl_sync(0xffffffffu, alpha, 8 * quad);
                    const float ao = __shfl_sync(0xffffffffu, alpha, 8 * quad + 4);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        oacc[j][0] *= ae;
                        oacc[j][1] *= ao;
                        oacc[j][2] *= ae;
                        oacc[j][3] *= ao;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        oacc[j][0] *= alpha;
                        oacc[j][1] *= alpha;
                    }
                }
                // ---- O += P V
                if constexpr (BYTE) {
                    // O^T += V^T P^T: M = 16 dims, N = 8 query heads, K = the 16 tokens.
                    // This lane's P fragments (tokens 2 quad, +1, +8, +9 of head `row`) are
                    // the B fragments as they stand.  M-tile mt's rows `row` and `row` + 8
                    // are dims 16 row + 2 mt and 16 row + 2 mt + 1, so the lane's V bytes
                    // are one 16-byte chunk per token; prmt pairs the bytes of two tokens.
                    const uint32_t ra = (uint32_t)(g * 16 + 2 * quad);
                    const uint4 wa = lds128(vst + ra * 128u + (uint32_t)((row ^ (int)(ra & 7u)) * 16));
                    const uint4 wb = lds128(vst + (ra + 1) * 128u +
                                            (uint32_t)((row ^ (int)((ra + 1) & 7u)) * 16));
                    const uint4 wc = lds128(vst + (ra + 8) * 128u +
                                            (uint32_t)((row ^ (int)((ra + 8) & 7u)) * 16));
                    const uint4 wd = lds128(vst + (ra + 9) * 128u +
                                            (uint32_t)((row ^ (int)((ra + 9) & 7u)) * 16));
                    const uint32_t a4[4] = {wa.x, wa.y, wa.z, wa.w}, b4[4] = {wb.x, wb.y, wb.z, wb.w};
                    const uint32_t c4[4] = {wc.x, wc.y, wc.z, wc.w}, d4[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        // m-tile 2 wi: bytes 0 (row) and 1 (row + 8); m-tile 2 wi + 1: bytes 2, 3
                        uint32_t e0, e1, e2, e3, f0, f1, f2, f3;
                        dec_byte4_to_f16x2x2<CACHE>(prmt(a4[wi], b4[wi], 0x5140u), e0, e1);
                        dec_byte4_to_f16x2x2<CACHE>(prmt(c4[wi], d4[wi], 0x5140u), e2, e3);
                        dec_byte4_to_f16x2x2<CACHE>(prmt(a4[wi], b4[wi], 0x7362u), f0, f1);
                        dec_byte4_to_f16x2x2<CACHE>(prmt(c4[wi], d4[wi], 0x7362u), f2, f3);
                        mma_f16_16816(oacc[2 * wi], e0, e1, e2, e3, pa0, pa2);
                        mma_f16_16816(oacc[2 * wi + 1], f0, f1, f2, f3, pa0, pa2);
                    }
                } else {
                    const int mi = lane >> 3, i = lane & 7;
                    const int tok = (mi & 1) * 8 + i;
                    const uint32_t r = (uint32_t)(g * 16 + tok);
#pragma unroll
                    for (int dn = 0; dn < 16; dn += 2) {
                        if (dn < nd) {
                            const int hf = dn >> 3;
                            const int chunk = (dn & 7) + (mi >> 1);
                            const uint32_t addr = vst + hf * half_bytes + r * 128u +
                                                  (uint32_t)((chunk ^ (int)(r & 7u)) * 16);
                            uint32_t v0, v1, v2, v3;
                            ldsm_x4_t(addr, v0, v1, v2, v3);
                            mma_bf16_16816(oacc[dn], pa0, 0u, pa2, 0u, v0, v1);
                            mma_bf16_16816(oacc[dn + 1], pa0, 0u, pa2, 0u, v2, v3);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                // release the stage; the last warp to do so refills it with page it + S
                // (the empty barrier's completed phase orders every warp's reads of the
                // stage before the copy that overwrites it)
                mbar_arrive(empty0 + 8 * s);
                if (atomicAdd(&released[s], 1) == Hkv - 1) {
                    released[s] = 0;
                    if (cit < n_iter && mbar_wait(empty0 + 8 * s, par, p.status, abort_flag))
                        issue(next_id);
                }
            }
            advance();
            if (mt.last) {
                // ---- partial result of this segment -> workspace slot b + cta
                const long long slot = (long long)cur_b + blockIdx.x;
                if constexpr (BYTE) {
                    // O^T: this lane holds heads 2 quad (c0, c2) and 2 quad + 1 (c1, c3)
                    // at dims 16 row + 2 mt, + 1
                    const float qe = __shfl_sync(0xffffffffu, q_run, 8 * quad);
                    const float qo = __shfl_sync(0xffffffffu, q_run, 8 * quad + 4);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int hq = 2 * quad + hh;
                        const float qr = hh ? qo : qe;
                        if (hq < Gq) {
                            const float inv = (qr > 0.f) ? vsc / qr : 0.f;
                            float *po = p.part_o + (slot * p.Hq + g * Gq + hq) * p.d + 16 * row;
#pragma unroll
                            for (int mt = 0; mt < 8; ++mt)
                                *reinterpret_cast<float2 *>(po + 2 * mt) =
                                    make_float2(oacc[mt][hh] * inv, oacc[mt][2 + hh] * inv);
                        }
                    }
                }
                if (row_ok) {
                    const int h = g * Gq + row;
                    if constexpr (!BYTE) {
                        const float inv = (q_run > 0.f) ? vsc / q_run : 0.f;
                        float *po = p.part_o + (slot * p.Hq + h) * p.d;
#pragma unroll
                        for (int dn = 0; dn < 16; ++dn) {
                            if (dn < nd) {
                                *reinterpret_cast<float2 *>(po + dn * 8 + 2 * quad) =
                                    make_float2(oacc[dn][0] * inv, oacc[dn][1] * inv);
                            }
                        }
                    }
                    if (quad == 0) {
                        p.part_lse[slot * p.Hq + h] =
                            (l_run > 0.f) ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
                    }
                }
            }
        }
    }
    __syncwarp();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        // an aborted launch lets the copies it issued land before the CTA exits
        for (int s = 0; s < S; ++s)
            if (n_issued[s] > 0)
                mbar_wait(full0 + 8 * s, (uint32_t)(n_issued[s] - 1) & 1u, p.status, nullptr);
    }
}

// One warp per (sequence b, query head h): combine the partial results of the CTAs
// that covered the sequence by their log-sum-exps, lanes splitting the partials
// (for the maximum and the weights) and then the d dimensions (for the weighted
// sum).  Grid (ceil(Hq / 8), B), 256 threads.  Launched as a programmatic
// dependent of the split kernel, so it may start while the split kernel's last CTAs
// still run: it waits for that grid's completion before reading the partials.
// A sequence whose length the page table cannot hold was treated as empty by the
// split kernel; this kernel records the error, once per sequence.
__global__ void __launch_bounds__(256)
decode_merge_kernel(const DecodeParams p, int G) {
    grid_dependency_wait();
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * 8 + warp;
    if (h >= p.Hq) return;
    if (h == 0 && lane == 0 && !dec_len_ok(p, b)) record_status(p.status, kStatusBounds);
    // start page of sequence b and total pages T
    long long before = 0, total = 0;
    for (int i = lane; i < p.B; i += 32) {
        const int np = dec_pages_of(p, i);
        total += np;
        if (i < b) before += np;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    const int np = dec_pages_of(p, b);
    const int dpl = p.d / 32;  // dimensions per lane: 2 or 4
    __nv_bfloat16 *ob = p.o + ((long long)b * p.Hq + h) * p.d + lane * dpl;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float mx = -INFINITY, wsum = 0.f;
    if (np > 0) {
        // CTAs c0..c1 cover the sequence's pages; a CTA whose range is empty (more CTAs
        // than pages) wrote nothing and is skipped
        const int c0 = dec_cta_of_page(before, total, G);
        const int c1 = dec_cta_of_page(before + np - 1, total, G);
        for (int cc = c0 + lane; cc <= c1; cc += 32)
            if (dec_range_nonempty(cc, total, G))
                mx = fmaxf(mx, p.part_lse[((long long)b + cc) * p.Hq + h]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (mx != -INFINITY) {
            for (int cb = c0; cb <= c1; cb += 32) {
                const int cc = cb + lane;
                float w = 0.f;
                if (cc <= c1 && dec_range_nonempty(cc, total, G))
                    w = ex2((p.part_lse[((long long)b + cc) * p.Hq + h] - mx) * kLog2e);
                wsum += w;
                const int n = min(32, c1 - cb + 1);
                for (int i = 0; i < n; ++i) {
                    const float wi = __shfl_sync(0xffffffffu, w, i);
                    if (wi == 0.f) continue;  // same for every lane
                    const float *po = p.part_o + (((long long)b + cb + i) * p.Hq + h) * p.d +
                                      lane * dpl;
                    if (dpl == 4) {
                        const float4 v = *reinterpret_cast<const float4 *>(po);
                        acc[0] = fmaf(wi, v.x, acc[0]);
                        acc[1] = fmaf(wi, v.y, acc[1]);
                        acc[2] = fmaf(wi, v.z, acc[2]);
                        acc[3] = fmaf(wi, v.w, acc[3]);
                    } else {
                        const float2 v = *reinterpret_cast<const float2 *>(po);
                        acc[0] = fmaf(wi, v.x, acc[0]);
                        acc[1] = fmaf(wi, v.y, acc[1]);
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (dpl == 4)
        *reinterpret_cast<uint2 *>(ob) = make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv),
                                                    pack_bf16(acc[2] * inv, acc[3] * inv));
    else
        *reinterpret_cast<uint32_t *>(ob) = pack_bf16(acc[0] * inv, acc[1] * inv);
    if (p.lse && lane == 0)
        p.lse[(long long)b * p.Hq + h] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

}  // namespace attn07
