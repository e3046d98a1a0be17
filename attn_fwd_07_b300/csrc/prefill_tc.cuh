// prefill_tc.cuh -- bf16 prefill attention on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for sm_103a.
//
// Method ("Donanıma Duyarlı Algoritma Tasarımı: FlashAttention",
// fatihsoysal.com): the attention formula of section "Transformer Mimarisi ve
// Self-Attention Mekanizması" is computed tile by tile in on-chip memory
// (section "FlashAttention'ın Temelleri"), with the online softmax of section
// "Online Softmax Prensibi" (running row maximum M and sum L), so the N x N
// score matrix never reaches device memory.  As in section "FlashAttention-2:
// Optimizasyonlar ve İyileştirmeler", work is split over blocks of query rows
// that each stream all the keys and values they need, loading the next block
// while the current one is computed.
//
// Work item: two 128-row query tiles that share one key/value head -- two query
// heads of the same group on the same rows when the group size is even, else
// two consecutive row tiles of one head.  Both tiles use every K_j and V_j tile
// loaded into shared memory, which halves the load traffic per MMA, and the
// two tiles' softmax runs while the tensor core works on the other tile
// ("ping-pong").
//
// Persistent CTAs: one CTA per SM.  CTA c starts on item c; its producer warp
// takes the next item index (heaviest first) from the launch's work counter while
// it loads the current item's last two key tiles, decodes each item once, skips
// blocks of items with nothing to compute, and hands the decoded items to the other
// roles through a small queue in shared memory.  Each role keeps its own ring
// positions and barrier phases across items, so the next item's query tiles and
// first key tiles load, and its first products run, while the previous item's
// output is still being written.
//
// Warp roles (512 threads, four warpgroups):
//   warps 0-3    softmax of tile 0, one thread per query row (TMEM lane)
//   warps 4-7    softmax of tile 1
//   warps 8-11   epilogue: O / L -> bf16 rows in device memory (32-byte stores),
//                for both tiles
//   warp 12      TMA producer: both Q tiles of an item, then K_j / V_j (128
//                keys) into two shared-memory rings (128-byte swizzle)
//   warp 13      MMA issuer (one thread), in this order for every j (PV with
//                N = d in one instruction per 16 keys: M128 N64 instructions run
//                at about 70% of the tensor core's rate, N128 at full rate):
//                   O_0 += P_0 V_j,  S_0 = Q_0 K_{j+1}^T,
//                   O_1 += P_1 V_j,  S_1 = Q_1 K_{j+1}^T
//                tcgen05.mma ops of one thread execute in issue order, so
//                S_{j+1} never overwrites P_j before O += P_j V_j has read it,
//                and a commit after S_{j+1} also covers that PV product.
//   warps 14-15  idle (they complete the fourth warpgroup)
// The softmax warpgroups raise their register count to 184 per thread; the
// epilogue warpgroup lowers its to 64 and the producer / MMA warpgroup to 80
// (2 x 184 + 64 + 80 = four times the 128 of the launch).
//
// Softmax step for tile t and key tile j (thread = row): load the S row from
// TMEM, mask (causal diagonal / window / sequence end), running maximum, P =
// 2^(S * scale * log2e - M) rounded to bf16 and written back over the S
// columns it came from (P is the A operand of the PV product, read from TMEM),
// row sums.  After a row's first key tile the maximum is first skipped: P is
// taken against the standing reference M, and only if some row's P sums past
// 2^24 on this tile is the S row reloaded and the step redone with its maximum.
// At the end of an item the softmax writes the row's LSE and hands 1 / L to the
// epilogue through shared memory.
//
// Rescaling: the row maximum used in the exponent only moves when the new
// maximum exceeds it by more than 8 (log2 units).  Until then P may reach
// 2^8, which fp32 and bf16 hold exactly in range; output and sums are always
// scaled consistently, so the result is the same exact softmax.  When it
// moves, O (in TMEM) and the sums are multiplied by 2^(M_old - M_new): the
// output rescaling that accompanies the online softmax.
//
// Tensor memory (512 columns of 128 lanes x 32 bit):
//   [0,128) S_0 (P_0 in its first 64 columns), [128,256) S_1 / P_1,
//   [256,256+d) O_0, [384,384+d) O_1
// The first PV product of an item into O_t waits until the epilogue has read
// the previous item's O_t out of TMEM.
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
    int ntiles;     // 128-row query tiles per sequence (of the longest sequence) to run
    int tile0;      // the first of them: tiles [tile0, tile0 + ntiles) of each sequence
    int head_pairs; // 1: an item takes two heads of a group on the same rows; 0: two row tiles
    int wl, wr;     // query i sees keys i - wl .. i + wr; -1: no limit on that side
                    // (causal: wl = -1, wr = 0; full: wl = wr = -1)
    float scale_log2;
    // paged keys/values (a chunk of queries against a cache): sequence s has
    // kv_lens[s] cached tokens, its chunk is the last q_len of them
    const int32_t *page_table;  // [nseq, maxp]
    const int32_t *kv_lens;     // [nseq]
    int maxp, num_pages;
    // the launch's work counters: work[0] hands out item indices in order, heaviest
    // first, one at a time to whichever CTA asks; work[1] counts the CTAs that have
    // finished, and the last one sets both back to zero for the next launch
    unsigned *work;
};

template <int D>
struct PrefillCfg {
    static constexpr int BM = 128;
    static constexpr int BN = 128;
    static constexpr int NH = D / 64;                     // 64-column halves of a row
    static constexpr uint32_t HALF = 128u * 128u;         // one [128 rows][64] bf16 half: 16 KB
    static constexpr uint32_t TILE = NH * HALF;
    static constexpr int SK = (D == 128) ? 3 : 4;         // K ring stages
    static constexpr int SV = (D == 128) ? 2 : 4;         // V ring stages
    static constexpr uint32_t OFF_Q = 0;                  // Q_0, Q_1
    static constexpr uint32_t OFF_K = 2 * TILE;
    static constexpr uint32_t OFF_V = OFF_K + SK * TILE;
    static constexpr uint32_t OFF_STATS = OFF_V + SV * TILE;  // [2][128] fp32: 1 / L per row
    // the queue of decoded work items the producer hands to the other roles, and how
    // many key tiles before the end of an item the producer claims the next one
    static constexpr int NQ = 4;
    static constexpr int CLAIM = 2;
    static constexpr uint32_t OFF_ITEMS = OFF_STATS + 2 * 128 * 4;
    // (one more slot holds the item the producer has claimed but not yet published)
    static constexpr uint32_t OFF_CTRL = OFF_ITEMS + (NQ + 1) * 80;
    static constexpr uint32_t CTRL_BYTES = 512;
    static constexpr size_t SMEM = 1024 + OFF_CTRL + CTRL_BYTES;
    // TMEM columns
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 384;
    static constexpr int THREADS = 512;
    // per-thread registers after the split: softmax warpgroups, epilogue warpgroup, the
    // producer / MMA warpgroup; and the registers the split needs in all (at most what
    // the launch reserves)
    static constexpr uint32_t REG_SOFTMAX = 184, REG_EPI = 64, REG_OTHER = 80;
    static constexpr uint32_t REG_NEED = 128 * (2 * REG_SOFTMAX + REG_EPI + REG_OTHER);
};

static_assert(PrefillCfg<128>::SMEM <= 227 * 1024, "prefill shared memory");
// four warpgroups of 128 threads share the 65536 registers the launch reserves
static_assert(128 * (2 * PrefillCfg<128>::REG_SOFTMAX + PrefillCfg<128>::REG_EPI +
                     PrefillCfg<128>::REG_OTHER) == 65536,
              "register split must add up to the launch's registers");

// barrier slots inside the control block (8 bytes each)
enum : uint32_t {
    BAR_QFULL = 0,
    BAR_QEMPTY = 1,
    BAR_KFULL = 2,    // +s, s < 4
    BAR_KEMPTY = 6,   // +s
    BAR_VFULL = 10,   // +s
    BAR_VEMPTY = 14,  // +s
    BAR_SFULL = 18,   // +t, t < 2
    BAR_PFULL = 20,   // +t
    BAR_OFULL = 22,   // +t
    BAR_OEMPTY = 24,  // +t
    BAR_STATS = 26,   // +t: 1 / L of the item's rows written
    BAR_STATSE = 28,  // +t: ... and read by the epilogue
    BAR_DRAIN = 30,
    BAR_IFULL = 31,   // +slot, slot < 4: item queue slot written
    BAR_IEMPTY = 35,  // +slot: ... and read by every consumer
    BAR_COUNT = 39
};

// One work item: the two query tiles, their rows, and the key tiles each needs.
struct PrefillItem {
    int head[2], row0[2], jlo[2], jhi[2];
    bool valid[2];
    int tok0, qlen, batch, kvlen, qoff, g, sq;
    int J0, n_kv;  // key tiles J0 .. J0 + n_kv - 1 cover both tiles (0: end of the queue)
};
static_assert(sizeof(PrefillItem) <= 80, "item queue slot");

__device__ __forceinline__ int prefill_items(const PrefillParams &p) {
    const int units = (p.head_pairs ? p.Hq / 2 : p.Hq) * p.nseq;
    const int nouter = p.head_pairs ? p.ntiles : (p.ntiles + 1) / 2;
    return nouter * units;
}

// The next item index of this launch from the work counter.  CTA c's first item is
// item c (no counter access on the way to the first loads); the counter hands out
// the items from gridDim.x on.
__device__ __forceinline__ int prefill_next_item(const PrefillParams &p) {
    return (int)gridDim.x + (int)atomicAdd(p.work, 1u);
}

// The items are numbered heaviest query tiles first, heads fastest (a key/value
// head's query heads run together and share its K/V tiles in L2): item idx is head
// unit idx % hunits of block idx / hunits, and block b is query-tile level
// nouter - 1 - b / nseq of sequence b % nseq.  Whether an item has work depends on
// its block only.

// Whether sequence sq's sizes are valid (packed tokens inside [0, total); a paged
// sequence's cache holds its queries and fits its page-table row), and the rows its
// queries take: [tok0, tok0 + qlen), keys [0, kvlen), query i at position qoff + i.
template <bool PAGED>
__device__ __forceinline__ bool prefill_seq(const PrefillParams &p, int sq, int &tok0, int &qlen,
                                            int &kvlen, int &qoff) {
    if (p.cu_seqlens) {
        tok0 = p.cu_seqlens[sq];
        const int tend = p.cu_seqlens[sq + 1];
        qlen = tend - tok0;
        if (tok0 < 0 || tend < tok0 || tend > p.total) return false;
    } else {
        tok0 = 0;
        qlen = p.N;
    }
    kvlen = qlen;
    qoff = 0;
    if constexpr (PAGED) {
        kvlen = p.kv_lens[sq];
        qoff = kvlen - qlen;
        if (qoff < 0 || kvlen > p.maxp * 16) return false;
    }
    return true;
}

// Records the bounds errors of sequence sq: sizes outside the rules above (nothing of
// the sequence is read or written), or more packed rows than the launch's tiles
// cover (only those rows are done).  Each sequence is checked by one lane of one CTA.
template <int D, bool PAGED>
__device__ __forceinline__ void prefill_check_seq(const PrefillParams &p, int sq) {
    int qlen = p.N;
    if (p.cu_seqlens) {
        const int tok0 = p.cu_seqlens[sq];
        const int tend = p.cu_seqlens[sq + 1];
        qlen = tend - tok0;
        if (tok0 < 0 || tend < tok0 || tend > p.total) {
            record_status(p.status, kStatusBounds);
            return;
        }
        if (qlen > (p.tile0 + p.ntiles) * PrefillCfg<D>::BM) record_status(p.status, kStatusBounds);
    }
    if constexpr (PAGED) {
        // (a sequence with no queries in this call is not checked against its cache)
        const int kvlen = p.kv_lens[sq];
        if (qlen > 0 && (kvlen - qlen < 0 || kvlen > p.maxp * 16))
            record_status(p.status, kStatusBounds);
    }
}

// Whether block b has work.
template <int D, bool PAGED>
__device__ __forceinline__ bool prefill_block_has_work(const PrefillParams &p, int b) {
    using C = PrefillCfg<D>;
    const int nouter = p.head_pairs ? p.ntiles : (p.ntiles + 1) / 2;
    const int outer = nouter - 1 - b / p.nseq;
    int tok0, qlen, kvlen, qoff;
    if (!prefill_seq<PAGED>(p, b % p.nseq, tok0, qlen, kvlen, qoff)) return false;
    const int row0 = (p.tile0 + (p.head_pairs ? outer : 2 * outer)) * C::BM;
    return row0 < min(qlen, (p.tile0 + p.ntiles) * C::BM);
}

// Decode item idx; returns false when it has nothing to compute.
template <int D, bool PAGED>
__device__ __forceinline__ bool prefill_item(const PrefillParams &p, int idx, PrefillItem &it) {
    using C = PrefillCfg<D>;
    const int hunits = p.head_pairs ? p.Hq / 2 : p.Hq;
    const int units = hunits * p.nseq;
    const int nouter = p.head_pairs ? p.ntiles : (p.ntiles + 1) / 2;
    const int outer = nouter - 1 - idx / units;
    const int rem = idx % units;
    const int hu = rem % hunits;
    const int sq = rem / hunits;
    int tok0, qlen, kvlen, qoff;
    if (!prefill_seq<PAGED>(p, sq, tok0, qlen, kvlen, qoff)) return false;
    const int batch = p.cu_seqlens ? 0 : sq;
    if (p.head_pairs) {
        it.head[0] = 2 * hu;
        it.head[1] = 2 * hu + 1;
        it.row0[0] = it.row0[1] = (p.tile0 + outer) * C::BM;
    } else {
        it.head[0] = it.head[1] = hu;
        it.row0[0] = (p.tile0 + 2 * outer) * C::BM;
        it.row0[1] = it.row0[0] + C::BM;
    }
    const int row_end = min(qlen, (p.tile0 + p.ntiles) * C::BM);  // rows this launch runs
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        it.valid[t] = it.row0[t] < row_end;
        const int last_row = min(it.row0[t] + C::BM, qlen) - 1;
        const int lo_key = p.wl < 0 ? 0 : max(0, qoff + it.row0[t] - p.wl);
        const int hi_key = p.wr < 0 ? kvlen - 1 : min(kvlen - 1, qoff + last_row + p.wr);
        it.jlo[t] = lo_key / C::BN;
        it.jhi[t] = hi_key / C::BN;
    }
    if (!it.valid[0] && !it.valid[1]) return false;
    it.J0 = it.valid[0] ? (it.valid[1] ? min(it.jlo[0], it.jlo[1]) : it.jlo[0]) : it.jlo[1];
    const int J1 = it.valid[0] ? (it.valid[1] ? max(it.jhi[0], it.jhi[1]) : it.jhi[0]) : it.jhi[1];
    it.n_kv = J1 - it.J0 + 1;
    it.tok0 = tok0;
    it.qlen = qlen;
    it.batch = batch;
    it.kvlen = kvlen;
    it.qoff = qoff;
    it.sq = sq;
    it.g = it.head[0] / (p.Hq / p.Hkv);
    return true;
}

// whether tile t takes part in key tile J0 + i of the item
__device__ __forceinline__ bool prefill_uses(const PrefillItem &it, int t, int i) {
    const int j = it.J0 + i;
    return it.valid[t] && j >= it.jlo[t] && j <= it.jhi[t];
}

// PAGED: keys and values come from a cache of 16-token pages through the page
// table (eight page boxes per 128-key tile, assembled into the same shared-memory
// layout), queries are a packed chunk per sequence positioned at the end of the
// sequence's cached tokens.
// PASS: 0 = the one-pass forward above.  The two-pass form of the FlashAttention-1
// section ("FlashAttention-1 (İki Geçişli Yaklaşım)"): 1 = statistics only (S
// tiles, running maximum and sum; no V, no PV product) written as LSE = M + ln L;
// 2 = output with the statistics known (P = 2^(s * scale * log2e - LSE * log2e)
// needs no running maximum and no rescaling; O = P V).
template <int D, bool PAGED, int PASS = 0>
__global__ void __launch_bounds__(512, 1)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using C = PrefillCfg<D>;
    extern __shared__ uint8_t pf_smem_raw[];

    // packed sequences: cu_seqlens must start at 0 and end at the total token count,
    // or rows are left unwritten (checked once per launch)
    if (p.cu_seqlens && blockIdx.x == 0 && threadIdx.x == 0 &&
        (p.cu_seqlens[0] != 0 || p.cu_seqlens[p.nseq] != p.total))
        record_status(p.status, kStatusBounds);

    const int n_items = prefill_items(p);

    const uint32_t raw = smem_u32(pf_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = pf_smem_raw + (base - raw);
    const uint32_t ctrl = base + C::OFF_CTRL;
    uint8_t *ctrl_ptr = base_ptr + C::OFF_CTRL;
    float *stats = reinterpret_cast<float *>(base_ptr + C::OFF_STATS);  // [2][128]
    PrefillItem *items = reinterpret_cast<PrefillItem *>(base_ptr + C::OFF_ITEMS);
    auto bar = [&](uint32_t i) { return ctrl + 8u * i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(ctrl_ptr + 8 * BAR_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl_ptr + 8 * BAR_COUNT + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 384) {
        mbar_init(bar(BAR_QFULL), 1);
        mbar_init(bar(BAR_QEMPTY), 1);
        for (int s = 0; s < C::SK; ++s) {
            mbar_init(bar(BAR_KFULL + s), 1);
            mbar_init(bar(BAR_KEMPTY + s), 1);
        }
        for (int s = 0; s < C::SV; ++s) {
            mbar_init(bar(BAR_VFULL + s), 1);
            mbar_init(bar(BAR_VEMPTY + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(BAR_SFULL + t), 1);
            mbar_init(bar(BAR_PFULL + t), 4);
            mbar_init(bar(BAR_OFULL + t), 1);
            mbar_init(bar(BAR_OEMPTY + t), 4);
            mbar_init(bar(BAR_STATS + t), 4);
            mbar_init(bar(BAR_STATSE + t), 4);
        }
        mbar_init(bar(BAR_DRAIN), 1);
        for (int q = 0; q < C::NQ; ++q) {
            mbar_init(bar(BAR_IFULL + q), 1);
            // every consumer of the queue: the MMA thread, 8 softmax and 4 epilogue warps
            mbar_init(bar(BAR_IEMPTY + q), 13);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 13) {
        tmem_alloc(ctrl + 8 * BAR_COUNT, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // (each role lowers or raises its warpgroup's registers first thing, so that the
    // register limit of its code is the new count)
    if (warp >= 12) {
    setmaxnreg_dec<C::REG_OTHER>();
    if (warp == 12) {
        // ============================ TMA producer
        // every packed or paged sequence's sizes are checked once per launch, the
        // sequences spread over the CTAs' producer warps
        if (p.cu_seqlens != nullptr || PAGED)
            for (int sq = (int)blockIdx.x * 32 + lane; sq < p.nseq; sq += (int)gridDim.x * 32)
                prefill_check_seq<D, PAGED>(p, sq);
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            int kvc = 0;                     // key tiles loaded so far (ring position)
            int nq = 0;                      // items whose query tiles were loaded
            int npub = 0;                    // queue entries published (the end mark included)
            int issued_k = 0, issued_v = 0;  // ring positions issued
            bool ok = true;
            // the next item with work, decoded: indices come from the launch's counter,
            // heaviest first; the ones with nothing to compute are skipped here, once
            // An item without work belongs to a block without work (a query-tile level
            // past its sequence's end, or a sequence whose sizes are invalid): the blocks
            // after it are checked here, up to a valid one, and the counter is moved past
            // the ones between (none of their items has work), so that no CTA claims
            // them one at a time.
            const int hunits = p.head_pairs ? p.Hq / 2 : p.Hq;
            const int n_blocks = n_items / hunits;
            auto fetch = [&](PrefillItem &dst, bool first) -> bool {
                int idx = first ? (int)blockIdx.x : prefill_next_item(p);
                for (;;) {
                    if (idx >= n_items) return false;
                    if (prefill_item<D, PAGED>(p, idx, dst)) return true;
                    int b = idx / hunits + 1;
                    for (int k = 0; k < 64 && b < n_blocks && !prefill_block_has_work<D, PAGED>(p, b);
                         ++k)
                        ++b;
                    const long long target = (long long)b * hunits - (long long)gridDim.x;
                    if (target > 0) atomicMax(p.work, (unsigned)target);
                    idx = prefill_next_item(p);
                }
            };
            PrefillItem it;
            bool have = fetch(it, true);
            for (;;) {
                // hand the item (or the end of the queue) to the other roles
                const int slot = npub % C::NQ;
                if (!mbar_wait(bar(BAR_IEMPTY + slot), ((uint32_t)(npub / C::NQ) & 1u) ^ 1u,
                               p.status, abort_flag)) {
                    ok = false;
                    break;
                }
                if (have)
                    items[slot] = it;
                else
                    items[slot].n_kv = 0;
                mbar_arrive(bar(BAR_IFULL + slot));
                ++npub;
                if (!have) break;
                // both query tiles, once the previous item's QK products are done with theirs
                if (!mbar_wait(bar(BAR_QEMPTY), ((uint32_t)nq & 1u) ^ 1u, p.status, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(BAR_QFULL), (uint32_t)(it.valid[0] + it.valid[1]) * C::TILE);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!it.valid[t]) continue;
#pragma unroll
                    for (int hf = 0; hf < C::NH; ++hf)
                        tma_load_4d(base + C::OFF_Q + t * C::TILE + hf * C::HALF, &tmQ,
                                    bar(BAR_QFULL), hf * 64, it.head[t], it.tok0 + it.row0[t],
                                    it.batch, pol_q);
                }
                ++nq;
                // the next item is claimed when this one's last CLAIM key tiles are being
                // loaded: late enough that the end of the launch evens out, early enough
                // that its query tiles are in L2 when they are needed
                PrefillItem &nx = items[C::NQ];  // (kept in shared memory, off the registers)
                bool have_nx = false;
                const int j_claim = max(0, it.n_kv - C::CLAIM);
                const int npg = (it.kvlen + 15) / 16;  // pages holding this sequence's keys
                // PAGED: page ids of key tile J0 + j (eight 16-token pages), read one tile
                // ahead so the loads overlap the waits; -1 past the sequence
                int ids_next[8];
                auto read_ids = [&](int j) {
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) {
                        const int pg = (it.J0 + j) * 8 + q8;
                        ids_next[q8] = (j < it.n_kv && pg < npg)
                                           ? p.page_table[(long long)it.sq * p.maxp + pg] : -1;
                    }
                };
                if constexpr (PAGED) read_ids(0);
                for (int j = 0; j < it.n_kv; ++j) {
                    const int kv = kvc + j;
                    const int kvrow = it.tok0 + (it.J0 + j) * C::BN;
                    // a page past the sequence, or a page id out of range (reported), is
                    // loaded from an out-of-range page coordinate: the copy fills zeros
                    int pcoord[8];
                    if constexpr (PAGED) {
#pragma unroll
                        for (int q8 = 0; q8 < 8; ++q8) {
                            const int pg = (it.J0 + j) * 8 + q8;
                            int pid = ids_next[q8];
                            if (pg >= npg) {
                                pid = p.num_pages;
                            } else if ((unsigned)pid >= (unsigned)p.num_pages) {
                                record_status(p.status, kStatusBounds);
                                pid = p.num_pages;
                            }
                            pcoord[q8] = pid;
                        }
                        read_ids(j + 1);
                    }
                    const int sk = kv % C::SK;
                    if (!mbar_wait(bar(BAR_KEMPTY + sk), ((uint32_t)(kv / C::SK) & 1u) ^ 1u,
                                   p.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(BAR_KFULL + sk), C::TILE);
#pragma unroll
                    for (int hf = 0; hf < C::NH; ++hf) {
                        const uint32_t dst = base + C::OFF_K + sk * C::TILE + hf * C::HALF;
                        if constexpr (PAGED) {
#pragma unroll
                            for (int q8 = 0; q8 < 8; ++q8)
                                tma_load_4d(dst + q8 * 2048u, &tmK, bar(BAR_KFULL + sk), hf * 64,
                                            0, it.g, pcoord[q8], pol_kv);
                        } else {
                            tma_load_4d(dst, &tmK, bar(BAR_KFULL + sk), hf * 64, it.g, kvrow,
                                        it.batch, pol_kv);
                        }
                    }
                    issued_k = kv + 1;
                    if (j == j_claim) {
                        have_nx = fetch(nx, false);
                        if (have_nx) {
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                if (!nx.valid[t]) continue;
#pragma unroll
                                for (int hf = 0; hf < C::NH; ++hf)
                                    tma_prefetch_4d(&tmQ, hf * 64, nx.head[t],
                                                    nx.tok0 + nx.row0[t], nx.batch);
                            }
                        }
                    }
                    if constexpr (PASS == 1) continue;  // the statistics need no values
                    const int sv = kv % C::SV;
                    if (!mbar_wait(bar(BAR_VEMPTY + sv), ((uint32_t)(kv / C::SV) & 1u) ^ 1u,
                                   p.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(BAR_VFULL + sv), C::TILE);
#pragma unroll
                    for (int hf = 0; hf < C::NH; ++hf) {
                        const uint32_t dst = base + C::OFF_V + sv * C::TILE + hf * C::HALF;
                        if constexpr (PAGED) {
#pragma unroll
                            for (int q8 = 0; q8 < 8; ++q8)
                                tma_load_4d(dst + q8 * 2048u, &tmV, bar(BAR_VFULL + sv), hf * 64,
                                            0, it.g, pcoord[q8], pol_kv);
                        } else {
                            tma_load_4d(dst, &tmV, bar(BAR_VFULL + sv), hf * 64, it.g, kvrow,
                                        it.batch, pol_kv);
                        }
                    }
                    issued_v = kv + 1;
                }
                kvc += it.n_kv;
                if (!ok) break;
                it = nx;
                have = have_nx;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                for (int kv = max(0, issued_k - C::SK); kv < issued_k; ++kv)
                    mbar_wait(bar(BAR_KFULL + kv % C::SK), (uint32_t)(kv / C::SK) & 1u, p.status,
                              nullptr);
                for (int kv = max(0, issued_v - C::SV); kv < issued_v; ++kv)
                    mbar_wait(bar(BAR_VFULL + kv % C::SV), (uint32_t)(kv / C::SV) & 1u, p.status,
                              nullptr);
                if (nq > 0)
                    mbar_wait(bar(BAR_QFULL), (uint32_t)(nq - 1) & 1u, p.status, nullptr);
            }
        }
    } else if (warp == 13) {
        // ============================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
            // PV: V is MN-major; its two 64-dim halves (128-byte swizzle atoms) lie 16 KB
            // apart, which the descriptor's leading offset describes
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
            // descriptors of the two query tiles (fixed) and of ring stage 0's K and V; a
            // stage's descriptors are stage 0's advanced by the stage offset
            const SmemDesc qd0 = smem_desc_parts(base + C::OFF_Q, 1024, 1024);
            const SmemDesc qd1 = smem_desc_parts(base + C::OFF_Q + C::TILE, 1024, 1024);
            const SmemDesc kd0 = smem_desc_parts(base + C::OFF_K, 1024, 1024);
            const SmemDesc vd0 = smem_desc_parts(base + C::OFF_V, C::HALF, 1024);
            // S_t = Q_t K^T (K in ring stage st) into S buffer t
            auto issue_qk = [&](int t, int st) {
                const SmemDesc qd = t ? qd1 : qd0;
                const SmemDesc kd{kd0.lo + (uint32_t)st * (C::TILE >> 4), kd0.hi};
                const uint32_t dcol = tmem + (t ? C::COL_S1 : C::COL_S0);
                // each of the D/16 steps advances the start addresses by a constant (32
                // bytes within a 64-dim half, 16 KB between the halves)
                tc_mma_ss_off<0, 0>(dcol, qd, kd, idesc_qk, 0u);
                tc_mma_ss_off<32, 32>(dcol, qd, kd, idesc_qk, 1u);
                tc_mma_ss_off<64, 64>(dcol, qd, kd, idesc_qk, 1u);
                tc_mma_ss_off<96, 96>(dcol, qd, kd, idesc_qk, 1u);
                if constexpr (D == 128) {
                    tc_mma_ss_off<C::HALF, C::HALF>(dcol, qd, kd, idesc_qk, 1u);
                    tc_mma_ss_off<C::HALF + 32, C::HALF + 32>(dcol, qd, kd, idesc_qk, 1u);
                    tc_mma_ss_off<C::HALF + 64, C::HALF + 64>(dcol, qd, kd, idesc_qk, 1u);
                    tc_mma_ss_off<C::HALF + 96, C::HALF + 96>(dcol, qd, kd, idesc_qk, 1u);
                }
                tc_commit(bar(BAR_SFULL + t));
            };
            // O_t += P_t V (V in ring stage st): P_t (bf16, 128 x 128) from the S_t columns
            auto issue_pv = [&](int t, int st, uint32_t acc) {
                const SmemDesc vd{vd0.lo + (uint32_t)st * (C::TILE >> 4), vd0.hi};
                const uint32_t pcol = tmem + (t ? C::COL_S1 : C::COL_S0);
                const uint32_t ocol = tmem + (t ? C::COL_O1 : C::COL_O0);
                tc_mma_ts_off<0>(ocol, pcol, vd, idesc_pv, acc);
                tc_mma_ts_off<2048>(ocol, pcol + 8, vd, idesc_pv, 1u);
                tc_mma_ts_off<4096>(ocol, pcol + 16, vd, idesc_pv, 1u);
                tc_mma_ts_off<6144>(ocol, pcol + 24, vd, idesc_pv, 1u);
                tc_mma_ts_off<8192>(ocol, pcol + 32, vd, idesc_pv, 1u);
                tc_mma_ts_off<10240>(ocol, pcol + 40, vd, idesc_pv, 1u);
                tc_mma_ts_off<12288>(ocol, pcol + 48, vd, idesc_pv, 1u);
                tc_mma_ts_off<14336>(ocol, pcol + 56, vd, idesc_pv, 1u);
            };
            // ring positions are kept as (stage, phase parity) and advanced one at a time:
            // no division on the issuing thread's path
            int ks = 0, vs = 0;          // K / V stages of the current key tile
            uint32_t kph = 0, vph = 0;   // ... and the parities of their phases
            int nq = 0;                  // items whose query tiles were used
            int pc0 = 0, pc1 = 0;        // P hand-offs consumed per tile
            int oc0 = 0, oc1 = 0;        // items per tile whose O was produced
            bool ok = true;
            for (int ci = 0; ok; ++ci) {
                // the next item from the producer's queue (an end mark closes it)
                const int slot = ci % C::NQ;
                if (!mbar_wait(bar(BAR_IFULL + slot), (uint32_t)(ci / C::NQ) & 1u, p.status,
                               abort_flag)) {
                    ok = false;
                    break;
                }
                const PrefillItem it = items[slot];
                mbar_arrive(bar(BAR_IEMPTY + slot));
                if (it.n_kv == 0) break;
                // steps [f_t, l_t] of the item use tile t (none for an invalid tile)
                const int f0 = it.valid[0] ? it.jlo[0] - it.J0 : 1 << 30;
                const int l0 = it.valid[0] ? it.jhi[0] - it.J0 : -1;
                const int f1 = it.valid[1] ? it.jlo[1] - it.J0 : 1 << 30;
                const int l1 = it.valid[1] ? it.jhi[1] - it.J0 : -1;
                const int n_kv = it.n_kv;
                ok = mbar_wait(bar(BAR_QFULL), (uint32_t)nq & 1u, p.status, abort_flag) &&
                     mbar_wait(bar(BAR_KFULL + ks), kph, p.status, abort_flag);
                if (!ok) break;
                ++nq;
                tc_fence_after();
                if (f0 == 0) issue_qk(0, ks);
                if (f1 == 0) issue_qk(1, ks);
                if (n_kv == 1) tc_commit(bar(BAR_QEMPTY));  // the item's last QK product
                tc_commit(bar(BAR_KEMPTY + ks));
                for (int j = 0; j < n_kv; ++j) {
                    const int ks1 = ks + 1 == C::SK ? 0 : ks + 1;
                    const uint32_t kph1 = ks1 == 0 ? kph ^ 1u : kph;
                    const bool more = j + 1 < n_kv;
                    // the value tile of this step and the key tile of the next are waited for
                    // first: they are normally in place, and checking them while the softmax
                    // still works keeps the checks off the path from P to the next product
                    // (every key tile of the item is used by at least one query tile)
                    if (PASS != 1 && !mbar_wait(bar(BAR_VFULL + vs), vph, p.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (more && !mbar_wait(bar(BAR_KFULL + ks1), kph1, p.status, abort_flag)) {
                        ok = false;
                        break;
                    }
                    // tile 0, then tile 1: O_t += P_t V_j, S_t = Q_t K_{j+1}^T
                    if (j >= f0 && j <= l0) {
                        // (statistics pass: PFULL says the S tile has been read)
                        if (!mbar_wait(bar(BAR_PFULL + 0), (uint32_t)pc0 & 1u, p.status,
                                       abort_flag)) {
                            ok = false;
                            break;
                        }
                        ++pc0;
                        if constexpr (PASS != 1) {
                            // the item's first product into O_0 waits until the epilogue has
                            // read the previous item's O_0
                            if (j == f0 && !mbar_wait(bar(BAR_OEMPTY + 0),
                                                      ((uint32_t)oc0 & 1u) ^ 1u, p.status,
                                                      abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_pv(0, vs, j == f0 ? 0u : 1u);
                            if (j == l0) tc_commit(bar(BAR_OFULL + 0));
                        }
                    }
                    if (j + 1 >= f0 && j + 1 <= l0) issue_qk(0, ks1);
                    if (j >= f1 && j <= l1) {
                        if (!mbar_wait(bar(BAR_PFULL + 1), (uint32_t)pc1 & 1u, p.status,
                                       abort_flag)) {
                            ok = false;
                            break;
                        }
                        ++pc1;
                        if constexpr (PASS != 1) {
                            if (j == f1 && !mbar_wait(bar(BAR_OEMPTY + 1),
                                                      ((uint32_t)oc1 & 1u) ^ 1u, p.status,
                                                      abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_pv(1, vs, j == f1 ? 0u : 1u);
                            if (j == l1) tc_commit(bar(BAR_OFULL + 1));
                        }
                    }
                    if (j + 1 >= f1 && j + 1 <= l1) issue_qk(1, ks1);
                    if (j + 2 == n_kv) tc_commit(bar(BAR_QEMPTY));  // the item's last QK
                    if (PASS != 1) tc_commit(bar(BAR_VEMPTY + vs));
                    if (more) tc_commit(bar(BAR_KEMPTY + ks1));
                    if (++vs == C::SV) {
                        vs = 0;
                        vph ^= 1u;
                    }
                    ks = ks1;
                    kph = kph1;
                }
                if (!ok) break;
                if (it.valid[0]) ++oc0;
                if (it.valid[1]) ++oc1;
            }
            // all issued MMAs complete before TMEM is released
            tc_commit(bar(BAR_DRAIN));
            mbar_wait(bar(BAR_DRAIN), 0u, p.status, nullptr);
        }
    }
    } else if (warp < 8) {
        // ============================ softmax: warpgroup t, thread = query row
        setmaxnreg_inc<C::REG_SOFTMAX>();
        const int t = warp >> 2;
        const int r = threadIdx.x & 127;           // row in tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t scol = tmem + lane_base + (t ? C::COL_S1 : C::COL_S0);
        const uint32_t ocol = tmem + lane_base + (t ? C::COL_O1 : C::COL_O0);
        const float sl2 = p.scale_log2;
        int sc = 0;   // S tiles consumed (SFULL phases)
        int oc = 0;   // items of this tile (STATS / STATSE phases)
        bool ok = true;
        for (int ci = 0; ok; ++ci) {
            // the next item from the producer's queue (an end mark closes it)
            const int slot = ci % C::NQ;
            ok = mbar_wait(bar(BAR_IFULL + slot), (uint32_t)(ci / C::NQ) & 1u, p.status, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            const PrefillItem it = items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_IEMPTY + slot));
            if (it.n_kv == 0) break;
            if (!it.valid[t]) continue;
            const int j_first = it.jlo[t];
            const int n_mine = it.jhi[t] - j_first + 1;
            const int qpos = it.row0[t] + r;  // position within the sequence
            // allowed keys of this row: [klo, khi]
            const int klo = p.wl < 0 ? 0 : it.qoff + qpos - p.wl;
            const int khi = p.wr < 0 ? it.kvlen - 1 : min(it.kvlen - 1, it.qoff + qpos + p.wr);
            float m_ref = -INFINITY;                   // log2 units, scaled
            float l = 0.f;                             // sum of P (fp32) -> LSE
            float lr = 0.f;                            // sum of bf16-rounded P -> normalises O
            const long long lse_idx = p.cu_seqlens
                                          ? (long long)it.head[t] * p.total + it.tok0 + qpos
                                          : ((long long)it.batch * p.Hq + it.head[t]) * p.N + qpos;
            if constexpr (PASS == 2) {
                // the row's statistics from the first pass: P = 2^(s * sl2 - LSE * log2e)
                const float lse_row = qpos < it.qlen ? p.lse[lse_idx] : 0.f;
                m_ref = lse_row * kLog2e;
            }
            for (int j = 0; j < n_mine; ++j) {
                ok = mbar_wait(bar(BAR_SFULL + t), (uint32_t)sc & 1u, p.status, abort_flag);
                ++sc;
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[128];
                float *s = reinterpret_cast<float *>(sr);
                const int kv0 = (j_first + j) * C::BN;
                const bool masked = kv0 < klo || kv0 + C::BN - 1 > khi;
                // keys outside [klo, khi] of columns [c0, c0 + 64) masked
                auto mask_half = [&](int c0) {
                    if (masked) {
#pragma unroll
                        for (int c = c0; c < c0 + 64; ++c)
                            if (kv0 + c < klo || kv0 + c > khi) s[c] = -INFINITY;
                    }
                };
                // the S row from TMEM, masked
                auto load_s = [&]() {
                    tmem_ld32(scol + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                    tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                    tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
                    tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
                    tc_wait_ld();
                    mask_half(0);
                    mask_half(64);
                };
                // one-pass fast path (below): after a row's first key tile
                const bool fast = PASS == 0 && __all_sync(0xffffffffu, j > 0 && m_ref != -INFINITY);
                if (!fast) load_s();
                if constexpr (PASS == 1) {
                    // the S tile is in registers: the next one may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_PFULL + t));
                }
                bool p_done = false;
                if constexpr (PASS == 1) {
                    // Statistics pass, fast path: while the reference stands only the sum of P
                    // is needed (same bound as below).  The S row stays in registers (no P is
                    // stored), so a tile whose sum passes 2^24 goes on to the maximum below.
                    if (__all_sync(0xffffffffu, j > 0 && m_ref != -INFINITY)) {
                        float fe[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int c = 0; c < 128; c += 2) {
                            float t0, t1;
                            ffma2(t0, t1, s[c], s[c + 1], sl2, sl2, -m_ref, -m_ref);
                            const int a = (c >> 1) & 1;
                            fadd2(fe[2 * a], fe[2 * a + 1], ex2(t0), ex2(t1));
                        }
                        const float lt = (fe[0] + fe[1]) + (fe[2] + fe[3]);
                        if (__all_sync(0xffffffffu, lt <= 16777216.f)) {
                            l += lt;
                            p_done = true;
                        }
                    }
                }
                if constexpr (PASS == 0) {
                    // Fast path: try P against the current reference maximum first.  If no
                    // row's sum of P over this tile exceeds 2^24, no element exceeds the
                    // reference by more than 24 (log2 units): P, the sums and O stay far
                    // inside the fp32/bf16 range (relative precision does not depend on the
                    // scale), so the reference stands and the row maximum is never needed.
                    // The S row arrives in two halves: the second half's load is in flight
                    // while the first half's P is computed and stored, and each 32 keys' P
                    // goes to TMEM as soon as it is packed (over S columns already read).
                    // Otherwise the S row is still in registers: the path with the maximum
                    // below recomputes P over the same columns, moving the reference when
                    // it is exceeded by more than 8.
                    if (fast) {
                        tmem_ld32(scol + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                        tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                        tc_wait_ld();
                        tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
                        tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
                        mask_half(0);
                        float fe[4] = {0.f, 0.f, 0.f, 0.f};
                        float fq[2] = {0.f, 0.f};
#pragma unroll
                        for (int cb = 0; cb < 128; cb += 32) {
                            if (cb == 64) {
                                tc_wait_ld();
                                mask_half(64);
                            }
                            uint32_t pk[16];
#pragma unroll
                            for (int c = cb; c < cb + 32; c += 2) {
                                float t0, t1;
                                ffma2(t0, t1, s[c], s[c + 1], sl2, sl2, -m_ref, -m_ref);
                                const float p0 = ex2(t0);
                                const float p1 = ex2(t1);
                                const int a = (c >> 1) & 1;
                                fadd2(fe[2 * a], fe[2 * a + 1], p0, p1);
                                const uint32_t pp = pack_bf16(p0, p1);
                                add_bf16x2_to(fq[a], pp);
                                pk[(c - cb) >> 1] = pp;
                            }
                            tmem_st16(scol + (cb >> 1), pk);
                        }
                        const float lt = (fe[0] + fe[1]) + (fe[2] + fe[3]);
                        if (__all_sync(0xffffffffu, lt <= 16777216.f)) {
                            l += lt;
                            lr += fq[0] + fq[1];
                            p_done = true;
                        }
                    }
                }
                // row maximum: eight independent 3-input max chains (the output pass of the
                // two-pass form knows the row's statistics and skips this)
                if (!p_done) {
                if constexpr (PASS != 2) {
                float mxa[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mxa[i] = fmax3(s[i], s[i + 8], s[i + 16]);
#pragma unroll
                for (int c = 24; c + 16 <= 120; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) mxa[i] = fmax3(mxa[i], s[c + i], s[c + 8 + i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mxa[i] = fmaxf(mxa[i], s[120 + i]);
                const float mx = fmax3(fmax3(mxa[0], mxa[1], mxa[2]),
                                       fmax3(mxa[3], mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool need = m_new > m_ref + 8.0f;
                if (j == 0) {
                    m_ref = m_new;
                } else if (__any_sync(0xffffffffu, need)) {
                    // O_t holds P_{j-1} V_{j-1} complete: the commit that signalled S_j
                    // covers every MMA issued before it
                    const float alpha = need ? ex2(m_ref - m_new) : 1.0f;
                    if (need) {
                        l *= alpha;
                        lr *= alpha;
                        m_ref = m_new;
                    }
#pragma unroll 1
                    for (int c = 0; c < (PASS == 1 ? 0 : D); c += 16) {
                        uint32_t orr[16];
                        tmem_ld16(ocol + c, orr);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st16(ocol + c, orr);
                    }
                }
                }  // PASS != 2
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                // P = 2^(s*scale*log2e - M); the exact row sum feeds the log-sum-exp, and the
                // row sum of the bf16-rounded P (the values the PV product uses) normalises O,
                // so O / L stays an exact convex combination of V rows.  P goes over the first
                // 64 columns of the S buffer it came from, 32 values (16 columns) at a time,
                // so the S registers of a chunk are free once it is stored.
                float le[4] = {0.f, 0.f, 0.f, 0.f};
                float lq[2] = {0.f, 0.f};
#pragma unroll
                for (int cb = 0; cb < 128; cb += 32) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = cb; c < cb + 32; c += 2) {
                        float t0, t1;
                        ffma2(t0, t1, s[c], s[c + 1], sl2, sl2, -m_use, -m_use);
                        const float p0 = ex2(t0);
                        const float p1 = ex2(t1);
                        const int a = (c >> 1) & 1;
                        fadd2(le[2 * a], le[2 * a + 1], p0, p1);
                        if constexpr (PASS != 1) {
                            const uint32_t pp = pack_bf16(p0, p1);
                            add_bf16x2_to(lq[a], pp);
                            pk[(c - cb) >> 1] = pp;
                        }
                    }
                    if constexpr (PASS != 1) tmem_st16(scol + (cb >> 1), pk);
                }
                l += (le[0] + le[1]) + (le[2] + le[3]);
                lr += lq[0] + lq[1];
                }  // !p_done
                if constexpr (PASS != 1) {
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_PFULL + t));
                }
            }
            if (!ok) break;
            // ---- end of the item: LSE (the output pass takes it as input), and 1 / L
            //      for the epilogue once it has read the previous item's
            if (PASS != 2 && qpos < it.qlen && p.lse)
                p.lse[lse_idx] = (l > 0.f) ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
            if constexpr (PASS != 1) {
                ok = mbar_wait(bar(BAR_STATSE + t), ((uint32_t)oc & 1u) ^ 1u, p.status, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                stats[t * 128 + r] = (lr > 0.f) ? 1.f / lr : 0.f;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_STATS + t));
            }
            ++oc;
        }
    } else {
        // ============================ epilogue: thread = query row of both tiles
        setmaxnreg_dec<C::REG_EPI>();
        {
            const int r = threadIdx.x & 127;       // row in tile = TMEM lane
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            const bool o32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
            int oc[2] = {0, 0};
            bool ok = true;
            for (int ci = 0; ok; ++ci) {
                // the next item from the producer's queue (an end mark closes it)
                const int slot = ci % C::NQ;
                ok = mbar_wait(bar(BAR_IFULL + slot), (uint32_t)(ci / C::NQ) & 1u, p.status,
                               abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const PrefillItem it = items[slot];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(BAR_IEMPTY + slot));
                if (it.n_kv == 0) break;
                // (the statistics pass writes no output)
#pragma unroll 1
                for (int t = 0; t < 2 && PASS != 1; ++t) {
                    if (!it.valid[t]) continue;
                    ok = mbar_wait(bar(BAR_STATS + t), (uint32_t)oc[t] & 1u, p.status, abort_flag);
                    const float inv = stats[t * 128 + r];
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(bar(BAR_STATSE + t));
                    ok = ok && mbar_wait(bar(BAR_OFULL + t), (uint32_t)oc[t] & 1u, p.status,
                                         abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ocol = tmem + lane_base + (t ? C::COL_O1 : C::COL_O0);
                    const int qpos = it.row0[t] + r;
                    const bool row_ok = qpos < it.qlen;
                    const long long tok = (long long)it.tok0 + qpos;
                    __nv_bfloat16 *orow =
                        p.o + ((p.cu_seqlens ? tok : (long long)it.batch * p.N + qpos) * p.Hq +
                               it.head[t]) * D;
                    // 32 columns per TMEM wait; each 16 columns (32 bytes of the row) go out
                    // in one 32-byte store when O is 32-byte aligned (rows are D * 2 bytes)
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t orr[2][16];
                        tmem_ld16(ocol + c, orr[0]);
                        tmem_ld16(ocol + c + 16, orr[1]);
                        tc_wait_ld();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t pkd[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                pkd[e] = pack_bf16(__uint_as_float(orr[h][2 * e]) * inv,
                                                   __uint_as_float(orr[h][2 * e + 1]) * inv);
                            if (row_ok) {
                                if (o32) {
                                    stg256(orow + c + 16 * h, pkd);
                                } else {
                                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c + 16 * h);
                                    dst[0] = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
                                    dst[1] = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
                                }
                            }
                        }
                    }
                    // O_t is out of TMEM: the next item's first product may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(BAR_OEMPTY + t));
                    ++oc[t];
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // every role of this CTA is done with the work counter; the last CTA to get here
    // sets the launch's counters back to zero
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.work + 1, 1u) == gridDim.x - 1) {
            __threadfence();
            p.work[0] = 0u;
            p.work[1] = 0u;
        }
    }
}

}  // namespace attn07
