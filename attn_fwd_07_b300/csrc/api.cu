// api.cu -- the C ABI of libattn07.so (declared in include/attn07.h): argument
// validation, tensor-map construction and kernel launches.  No entry point
// allocates, frees or synchronises device memory (attn_get_device_status
// synchronises its stream by design).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <math.h>
#include <mutex>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "attn07.h"
#include "attn07_testing.h"
#include "decode.cuh"
#include "prefill_simt.cuh"
#include "prefill_tc.cuh"
#include "selftest.cuh"

using namespace attn07;

// Device status word shared by every kernel of the library (per device).
__device__ unsigned int g_attn_status;

// Work counters of the tensor-core prefill, two per slot (next item, CTAs done).  A
// launch takes the next slot in turn; it leaves its counters at zero when its last CTA
// ends, so a slot is ready for reuse (a replayed graph reuses its launches' slots).
// Launches in flight at the same time, on other streams, use other slots, up to 1024.
constexpr int kWorkSlots = 1024;
__device__ unsigned g_prefill_work[2 * kWorkSlots];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    unsigned *status = nullptr;
    unsigned *work = nullptr;  // g_prefill_work on this device
};

// prefill launches in this process, for the choice of work-counter slot
std::atomic<unsigned> g_prefill_launches{0};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// The last CUDA failure seen by an entry point on this host thread (reported by
// attn_last_cuda_error).
thread_local char g_last_cuda_error[160] = "no CUDA error recorded";

attn_status_t cuda_fail(cudaError_t e) {
    (void)cudaGetLastError();
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
}

attn_status_t driver_fail(CUresult r, const char *what) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s failed with CUresult %d", what,
             (int)r);
    return ATTN_ERR_CUDA;
}

// status of the launches just enqueued
attn_status_t launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// The tensor-core prefill's warpgroups trade registers with setmaxnreg; the counts they
// ask for must fit in what the launch reserves per thread, or a raise would wait for
// ever.  Checked per instantiation against the compiled register count.
template <int D, bool PAGED, int PASS>
cudaError_t prefill_regs_fit() {
    using C = PrefillCfg<D>;
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, prefill_tc_kernel<D, PAGED, PASS>);
    if (e != cudaSuccess) return e;
    const long long have = (long long)a.numRegs * C::THREADS;
    const long long need = (long long)C::REG_NEED;
    return have >= need ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Shared-memory size attribute of every instantiation of the tensor-core prefill, and the
// register check above.
template <int D>
cudaError_t prefill_attrs() {
    const int smem = (int)PrefillCfg<D>::SMEM;
    cudaError_t e;
    if ((e = prefill_regs_fit<D, false, 0>()) != cudaSuccess ||
        (e = prefill_regs_fit<D, true, 0>()) != cudaSuccess ||
        (e = prefill_regs_fit<D, false, 1>()) != cudaSuccess ||
        (e = prefill_regs_fit<D, false, 2>()) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(prefill_tc_kernel<D, false, 0>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(prefill_tc_kernel<D, true, 0>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(prefill_tc_kernel<D, false, 1>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(prefill_tc_kernel<D, false, 2>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Per-device one-time set-up: SM count, status word address, kernel attributes.
attn_status_t device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        if ((e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        void *sym = nullptr;
        if ((e = cudaGetSymbolAddress(&sym, g_attn_status)) != cudaSuccess) return cuda_fail(e);
        st.status = static_cast<unsigned *>(sym);
        if ((e = cudaGetSymbolAddress(&sym, g_prefill_work)) != cudaSuccess) return cuda_fail(e);
        st.work = static_cast<unsigned *>(sym);
        if ((e = cudaFuncSetAttribute(prefill_simt_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)prefill_simt_smem_bytes(kSimtMaxD))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(prefill_simt_rows_kernel<4>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)prefill_simt_rows_smem_bytes(4, kSimtMaxD))) != cudaSuccess ||
            (e = cudaFuncSetAttribute(prefill_simt_rows_kernel<2>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)prefill_simt_rows_smem_bytes(2, kSimtMaxD))) != cudaSuccess)
            return cuda_fail(e);
        if ((e = prefill_attrs<128>()) != cudaSuccess || (e = prefill_attrs<64>()) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaFuncSetAttribute(decode_split_kernel<kCacheFp8>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      227 * 1024)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(decode_split_kernel<kCacheInt8>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      227 * 1024)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(decode_split_kernel<kCacheBf16>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      227 * 1024)) != cudaSuccess)
            return cuda_fail(e);
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cuda_fail(e);
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        st.ready = true;
    }
    *out = &st;
    return ATTN_OK;
}

// bf16 tensor map, 128-byte swizzle, box inner extent 64 elements.
attn_status_t make_map(CUtensorMap *m, const void *ptr, int rank, const cuuint64_t *dims,
                       const cuuint64_t *strides_bytes, const cuuint32_t *box,
                       CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, dtype, (cuuint32_t)rank,
                          const_cast<void *>(ptr), dims, strides_bytes, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : driver_fail(r, "cuTensorMapEncodeTiled");
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int D>
void launch_prefill_variant(unsigned grid, const PrefillParams &p, const CUtensorMap &mq,
                            const CUtensorMap &mk, const CUtensorMap &mv, bool paged, int pass,
                            cudaStream_t stream) {
    using C = PrefillCfg<D>;
    if (paged)
        prefill_tc_kernel<D, true, 0><<<grid, C::THREADS, C::SMEM, stream>>>(p, mq, mk, mv);
    else if (pass == 1)
        prefill_tc_kernel<D, false, 1><<<grid, C::THREADS, C::SMEM, stream>>>(p, mq, mk, mv);
    else if (pass == 2)
        prefill_tc_kernel<D, false, 2><<<grid, C::THREADS, C::SMEM, stream>>>(p, mq, mk, mv);
    else
        prefill_tc_kernel<D, false, 0><<<grid, C::THREADS, C::SMEM, stream>>>(p, mq, mk, mv);
}

// Keys and values held in a cache of 16-token pages (chunked prefill).
struct PagedKV {
    const int32_t *page_table;  // [nseq, maxp]
    const int32_t *kv_lens;     // [nseq]
    int maxp, num_pages;
};

// Launch the tensor-core prefill on a [tokens, heads, d] layout with `nseq`
// sequences along the outermost axis (dense) or one packed axis (varlen,
// cu_seqlens non-null).  With `paged`, q is a packed chunk per sequence and k, v
// are caches [num_pages, 16, Hkv, d] read through the page table.
attn_status_t launch_prefill_tc(const void *q, const void *k, const void *v, void *o, float *lse,
                                const int32_t *cu_seqlens, int nseq, int N_or_total,
                                int ntiles, int Hq, int Hkv, int d, int wl, int wr,
                                float scale, cudaStream_t stream,
                                const PagedKV *paged = nullptr, int pass = 0, int tile0 = 0) {
    DeviceState *st = nullptr;
    attn_status_t s = device_state(&st);
    if (s != ATTN_OK) return s;
    const bool varlen = cu_seqlens != nullptr;
    // dims innermost first: d, heads, tokens, batch
    const cuuint64_t nb = varlen ? 1 : (cuuint64_t)nseq;
    const cuuint64_t dq[4] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)N_or_total, nb};
    const cuuint64_t dk[4] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)N_or_total, nb};
    const cuuint64_t sq[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hq * d * 2,
                              (cuuint64_t)N_or_total * Hq * d * 2};
    const cuuint64_t sk[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2,
                              (cuuint64_t)N_or_total * Hkv * d * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    CUtensorMap mq, mk, mv;
    if ((s = make_map(&mq, q, 4, dq, sq, box)) != ATTN_OK) return s;
    if (paged) {
        // cache as (dim, token-in-page, head, page); one box = one page of one head
        const cuuint64_t dc[4] = {(cuuint64_t)d, 16, (cuuint64_t)Hkv,
                                  (cuuint64_t)paged->num_pages};
        const cuuint64_t sc[3] = {(cuuint64_t)Hkv * d * 2, (cuuint64_t)d * 2,
                                  (cuuint64_t)16 * Hkv * d * 2};
        const cuuint32_t bc[4] = {64, 16, 1, 1};
        if ((s = make_map(&mk, k, 4, dc, sc, bc)) != ATTN_OK) return s;
        if ((s = make_map(&mv, v, 4, dc, sc, bc)) != ATTN_OK) return s;
    } else {
        if ((s = make_map(&mk, k, 4, dk, sk, box)) != ATTN_OK) return s;
        if ((s = make_map(&mv, v, 4, dk, sk, box)) != ATTN_OK) return s;
    }
    PrefillParams p;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.cu_seqlens = cu_seqlens;
    p.status = st->status;
    p.N = varlen ? 0 : N_or_total;
    p.nseq = nseq;
    p.total = varlen ? N_or_total : 0;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.ntiles = ntiles;
    p.tile0 = tile0;
    // a CTA takes two query heads of one group on the same rows when the group size is
    // even, else two consecutive row tiles of one head
    p.head_pairs = ((Hq / Hkv) % 2 == 0) ? 1 : 0;
    p.wl = wl < 0 ? -1 : wl;
    p.wr = wr < 0 ? -1 : wr;
    p.scale_log2 = scale * kLog2e;
    p.page_table = paged ? paged->page_table : nullptr;
    p.kv_lens = paged ? paged->kv_lens : nullptr;
    p.maxp = paged ? paged->maxp : 0;
    p.num_pages = paged ? paged->num_pages : 0;
    p.work = st->work + 2 * (g_prefill_launches++ % kWorkSlots);
    // work items (pairs of query tiles); persistent CTAs, one per SM, walk them
    const long long items = p.head_pairs ? (long long)ntiles * (Hq / 2) * nseq
                                         : (long long)((ntiles + 1) / 2) * Hq * nseq;
    if (items > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    if (items == 0) return ATTN_OK;
    const unsigned gx = (unsigned)std::min<long long>(items, st->sms);
    if (d == 128)
        launch_prefill_variant<128>(gx, p, mq, mk, mv, paged != nullptr, pass, stream);
    else
        launch_prefill_variant<64>(gx, p, mq, mk, mv, paged != nullptr, pass, stream);
    return launch_status();
}

}  // namespace

extern "C" {

const char *attn_version(void) { return "attn07 0.1.0 sm_103a"; }

const char *attn_last_cuda_error(void) { return g_last_cuda_error; }

const char *attn_status_string(attn_status_t s) {
    switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_DEVICE_BOUNDS: return "device found an index out of range";
    }
    return "unknown status";
}

attn_status_t attn_get_device_status(attn_stream_t stream) {
    DeviceState *st = nullptr;
    attn_status_t s = device_state(&st);
    if (s != ATTN_OK) return s;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned v = 0;
    e = cudaMemcpy(&v, st->status, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        const unsigned zero = 0;
        e = cudaMemcpy(st->status, &zero, sizeof(unsigned), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return (attn_status_t)v;
}

attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int Hq, int Hkv, int N, int d, int causal, float scale,
                       attn_stream_t stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if ((long long)B * N * Hq * d > (1LL << 40)) return ATTN_ERR_UNSUPPORTED;
    const int ntiles = (N + 127) / 128;
    return launch_prefill_tc(q, k, v, o, lse, nullptr, B, N, ntiles, Hq, Hkv, d, -1,
                             causal ? 0 : -1, scale, reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int Hq, int Hkv, int N, int d, int window_left,
                              int window_right, float scale, attn_stream_t stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if ((long long)B * N * Hq * d > (1LL << 40)) return ATTN_ERR_UNSUPPORTED;
    const int ntiles = (N + 127) / 128;
    return launch_prefill_tc(q, k, v, o, lse, nullptr, B, N, ntiles, Hq, Hkv, d, window_left,
                             window_right, scale, reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                              int max_seqlen, int Hq, int Hkv, int d, int causal, float scale,
                              attn_stream_t stream) {
    if (!q || !k || !v || !o || !cu_seqlens) return ATTN_ERR_INVALID_ARG;
    if (num_seqs <= 0 || total_tokens < 0 || max_seqlen < 0 || Hq <= 0 || Hkv <= 0 ||
        Hq % Hkv != 0 || d <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (total_tokens == 0 || max_seqlen == 0) return ATTN_OK;
    const int ntiles = (max_seqlen + 127) / 128;
    return launch_prefill_tc(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, ntiles, Hq, Hkv,
                             d, -1, causal ? 0 : -1, scale, reinterpret_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_two_pass(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                                attn_stream_t stream) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if ((long long)B * N * Hq * d > (1LL << 40)) return ATTN_ERR_UNSUPPORTED;
    const int ntiles = (N + 127) / 128;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    attn_status_t s = launch_prefill_tc(q, k, v, o, lse, nullptr, B, N, ntiles, Hq, Hkv, d, -1,
                                        causal ? 0 : -1, scale, cs, nullptr, 1);
    if (s != ATTN_OK) return s;
    return launch_prefill_tc(q, k, v, o, lse, nullptr, B, N, ntiles, Hq, Hkv, d, -1,
                             causal ? 0 : -1, scale, cs, nullptr, 2);
}

attn_status_t attn_fwd_chunked_paged(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *page_table, const int32_t *seq_lens,
                                     const int32_t *cu_seqlens_q, void *o, float *lse,
                                     int num_seqs, int total_q, int max_qlen, int Hq, int Hkv,
                                     int d, int page_size, int num_pages, int max_pages_per_seq,
                                     int causal, float scale, attn_stream_t stream) {
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !cu_seqlens_q || !o)
        return ATTN_ERR_INVALID_ARG;
    if (num_seqs <= 0 || total_q < 0 || max_qlen < 0 || Hq <= 0 || Hkv <= 0 ||
        Hq % Hkv != 0 || d <= 0 || page_size <= 0 || num_pages <= 0 || max_pages_per_seq <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
        return ATTN_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if (total_q == 0 || max_qlen == 0) return ATTN_OK;
    const int ntiles = (max_qlen + 127) / 128;
    const PagedKV pk{page_table, seq_lens, max_pages_per_seq, num_pages};
    return launch_prefill_tc(q, k_cache, v_cache, o, lse, cu_seqlens_q, num_seqs, total_q,
                             ntiles, Hq, Hkv, d, -1, causal ? 0 : -1, scale,
                             reinterpret_cast<cudaStream_t>(stream), &pk);
}

namespace {

// fp32 prefill with `rows` query rows per CTA: 16 (prefill_simt_kernel), 4 or 2
// (prefill_simt_rows_kernel<4>, <2>); 0 lets the launch size decide.  With C CTAs of
// 16 rows: 2-row CTAs when 8 C <= #SM (one per SM at most), 4-row CTAs when
// 2 C <= #SM (one or two per SM), else 16-row CTAs (each K/V tile loaded into shared
// memory then serves 16 rows).  Smaller tiles put a short launch on more SMs.
attn_status_t fwd_f32_impl(const float *q, const float *k, const float *v, float *o, float *lse,
                           int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                           int rows, attn_stream_t stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
    if (rows != 0 && rows != kSimtBM && rows != 4 && rows != 2) return ATTN_ERR_INVALID_ARG;
    if (d > kSimtMaxD || d % 16 != 0) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
    DeviceState *st = nullptr;
    attn_status_t s = device_state(&st);
    if (s != ATTN_OK) return s;
    SimtParams p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.cu_seqlens = nullptr;
    p.N = N;
    p.total = 0;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    if (rows == 0) {
        const long long ctas16 = (long long)((N + kSimtBM - 1) / kSimtBM) * Hq * B;
        rows = 8 * ctas16 <= st->sms ? 2 : 2 * ctas16 <= st->sms ? 4 : kSimtBM;
    }
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 2) {
        dim3 grid((N + 1) / 2, Hq, B);
        prefill_simt_rows_kernel<2><<<grid, kSimtThreads, prefill_simt_rows_smem_bytes(2, d), cs>>>(p);
    } else if (rows == 4) {
        dim3 grid((N + 3) / 4, Hq, B);
        prefill_simt_rows_kernel<4><<<grid, kSimtThreads, prefill_simt_rows_smem_bytes(4, d), cs>>>(p);
    } else {
        dim3 grid((N + kSimtBM - 1) / kSimtBM, Hq, B);
        prefill_simt_kernel<<<grid, kSimtThreads, prefill_simt_smem_bytes(d), cs>>>(p);
    }
    return launch_status();
}

}  // namespace

attn_status_t attn_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                           int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                           attn_stream_t stream) {
    return fwd_f32_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, 0, stream);
}

attn_status_t attn_testing_fwd_f32_rows(const float *q, const float *k, const float *v, float *o,
                                        float *lse, int B, int Hq, int Hkv, int N, int d,
                                        int causal, float scale, int rows,
                                        attn_stream_t stream) {
    if (rows != kSimtBM && rows != 4 && rows != 2) return ATTN_ERR_INVALID_ARG;
    return fwd_f32_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, rows, stream);
}

size_t attn_decode_workspace_size(int B, int Hq, int d, int max_pages_per_seq, int page_size) {
    if (B <= 0 || Hq <= 0 || d <= 0 || max_pages_per_seq <= 0 || page_size <= 0) return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != ATTN_OK) return 0;
    // one slot per sequence plus one per CTA of the split kernel (up to two per SM)
    const size_t slots = (size_t)B + (size_t)kDecMaxCtasPerSm * st->sms;
    const size_t bytes_o = slots * Hq * d * sizeof(float);
    const size_t bytes_l = slots * Hq * sizeof(float);
    return ((bytes_o + 255) & ~(size_t)255) + bytes_l;
}

}  // extern "C"

namespace {

// The paged decode behind attn_decode_paged (window = -1), attn_decode_paged_window
// (the query sees the last window + 1 tokens), attn_decode_paged_fp8 and
// attn_decode_paged_int8 (cache = kCacheFp8 / kCacheInt8: the cache holds one byte per
// element, k_scale and v_scale its per-head scales).
attn_status_t decode_paged_impl(const void *q, const void *k_cache, const void *v_cache,
                                const float *k_scale, const float *v_scale, int cache,
                                const int32_t *page_table, const int32_t *seq_lens, void *o,
                                float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                int num_pages, int max_pages_per_seq, int window, float scale,
                                void *workspace, size_t workspace_bytes, attn_stream_t stream,
                                int ctas = 0) {
    const bool byte = cache != kCacheBf16;
    if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !o || !workspace)
        return ATTN_ERR_INVALID_ARG;
    if (byte && (!k_scale || !v_scale)) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page_size <= 0 ||
        num_pages <= 0 || max_pages_per_seq <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
        !aligned16(workspace))
        return ATTN_ERR_INVALID_ARG;
    if (page_size != kDecPage || (d != 64 && d != 128) || Hkv > kDecMaxHkv || Hq / Hkv > 8)
        return ATTN_ERR_UNSUPPORTED;
    if (byte && d != 128) return ATTN_ERR_UNSUPPORTED;
    DeviceState *st = nullptr;
    attn_status_t s = device_state(&st);
    if (s != ATTN_OK) return s;
    const size_t need = attn_decode_workspace_size(B, Hq, d, max_pages_per_seq, page_size);
    if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
    const size_t stage = dec_stage_bytes(Hkv, d, byte);
    // one-byte pages are half the bytes and twice the conversion work per byte: two
    // CTAs per SM (sixteen consumer warps) with half the ring each hide more of the
    // consumers' latency; the bf16 kernel keeps one CTA per SM and the deeper ring
    const int ctas_per_sm = byte ? 2 : 1;
    int stages = (int)(((byte ? 108 : 220) * 1024 - 2048) / stage);
    if (stages > kDecMaxStages) stages = kDecMaxStages;
    if (stages < 2) return ATTN_ERR_UNSUPPORTED;
    // cache as a 4-D tensor: (dim, token-in-page, head, page) so that one box
    // lands in shared memory as [head][token][128-byte row]: 64 bf16 dims per box,
    // or all 128 one-byte dims
    const cuuint64_t esz = byte ? 1 : 2;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)page_size, (cuuint64_t)Hkv,
                                (cuuint64_t)num_pages};
    const cuuint64_t strides[3] = {(cuuint64_t)Hkv * d * esz, (cuuint64_t)d * esz,
                                   (cuuint64_t)page_size * Hkv * d * esz};
    const cuuint32_t box[4] = {byte ? 128u : 64u, (cuuint32_t)page_size, (cuuint32_t)Hkv, 1};
    const CUtensorMapDataType dt = byte ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap mk, mv;
    if ((s = make_map(&mk, k_cache, 4, dims, strides, box, dt)) != ATTN_OK) return s;
    if ((s = make_map(&mv, v_cache, 4, dims, strides, box, dt)) != ATTN_OK) return s;

    const size_t slots = (size_t)B + (size_t)kDecMaxCtasPerSm * st->sms;
    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.part_o = static_cast<float *>(workspace);
    p.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                           ((slots * Hq * d * sizeof(float) + 255) & ~(size_t)255));
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.status = st->status;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.num_pages = num_pages;
    p.maxp = max_pages_per_seq;
    p.stages = stages;
    p.window = window < 0 ? -1 : window;
    p.scale_log2 = scale * kLog2e;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // the workspace has a slot per CTA for up to kDecMaxCtasPerSm CTAs per SM
    if (ctas < 0 || ctas > kDecMaxCtasPerSm * st->sms) return ATTN_ERR_UNSUPPORTED;
    const int G = ctas > 0 ? ctas : st->sms * ctas_per_sm;
    const size_t smem = dec_smem_bytes(Hkv, d, stages, byte);
    if (cache == kCacheFp8)
        decode_split_kernel<kCacheFp8><<<G, 32 * Hkv, smem, cs>>>(p, mk, mv);
    else if (cache == kCacheInt8)
        decode_split_kernel<kCacheInt8><<<G, 32 * Hkv, smem, cs>>>(p, mk, mv);
    else
        decode_split_kernel<kCacheBf16><<<G, 32 * Hkv, smem, cs>>>(p, mk, mv);
    if ((s = launch_status()) != ATTN_OK) return s;
    // the merge as a programmatic dependent of the split kernel: it is scheduled while
    // the split kernel's last CTAs run and waits on the device for their results, which
    // takes the launch gap between the two kernels off the step
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((Hq + 7) / 8), (unsigned)B, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = cs;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_merge_kernel, p, G);
    if (e != cudaSuccess) return cuda_fail(e);
    return launch_status();
}

}  // namespace

extern "C" {

attn_status_t attn_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *page_table, const int32_t *seq_lens, void *o,
                                float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                int num_pages, int max_pages_per_seq, float scale,
                                void *workspace, size_t workspace_bytes, attn_stream_t stream) {
    return decode_paged_impl(q, k_cache, v_cache, nullptr, nullptr, kCacheBf16, page_table,
                             seq_lens, o, lse,
                             B, Hq, Hkv, d,
                             page_size, num_pages, max_pages_per_seq, -1, scale, workspace,
                             workspace_bytes, stream);
}

attn_status_t attn_decode_paged_fp8(const void *q, const void *k_cache, const void *v_cache,
                                    const float *k_scale, const float *v_scale,
                                    const int32_t *page_table, const int32_t *seq_lens, void *o,
                                    float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                    int num_pages, int max_pages_per_seq, float scale,
                                    void *workspace, size_t workspace_bytes,
                                    attn_stream_t stream) {
    if (!k_scale || !v_scale) return ATTN_ERR_INVALID_ARG;
    return decode_paged_impl(q, k_cache, v_cache, k_scale, v_scale, kCacheFp8, page_table,
                             seq_lens, o, lse, B, Hq, Hkv, d, page_size, num_pages,
                             max_pages_per_seq, -1, scale, workspace, workspace_bytes, stream);
}

attn_status_t attn_decode_paged_int8(const void *q, const void *k_cache, const void *v_cache,
                                     const float *k_scale, const float *v_scale,
                                     const int32_t *page_table, const int32_t *seq_lens, void *o,
                                     float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                     int num_pages, int max_pages_per_seq, float scale,
                                     void *workspace, size_t workspace_bytes,
                                     attn_stream_t stream) {
    if (!k_scale || !v_scale) return ATTN_ERR_INVALID_ARG;
    return decode_paged_impl(q, k_cache, v_cache, k_scale, v_scale, kCacheInt8, page_table,
                             seq_lens, o, lse, B, Hq, Hkv, d, page_size, num_pages,
                             max_pages_per_seq, -1, scale, workspace, workspace_bytes, stream);
}

attn_status_t attn_decode_paged_window(const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *page_table, const int32_t *seq_lens,
                                       void *o, float *lse, int B, int Hq, int Hkv, int d,
                                       int page_size, int num_pages, int max_pages_per_seq,
                                       int window, float scale, void *workspace,
                                       size_t workspace_bytes, attn_stream_t stream) {
    if (window < -1) return ATTN_ERR_INVALID_ARG;
    return decode_paged_impl(q, k_cache, v_cache, nullptr, nullptr, kCacheBf16, page_table,
                             seq_lens, o, lse,
                             B, Hq, Hkv, d,
                             page_size, num_pages, max_pages_per_seq, window, scale, workspace,
                             workspace_bytes, stream);
}

// ---------------------------------------------------------------- test hook
// attn_decode_paged with the split kernel's CTA count chosen by the caller (declared in
// attn07_testing.h, not part of the interface): the merged result must not depend on how
// the pages are cut into CTA ranges, which tests check at counts the length mix of a
// workload would not produce by itself.
attn_status_t attn_testing_decode_paged_ctas(const void *q, const void *k_cache,
                                             const void *v_cache, const int32_t *page_table,
                                             const int32_t *seq_lens, void *o, float *lse, int B,
                                             int Hq, int Hkv, int d, int page_size, int num_pages,
                                             int max_pages_per_seq, float scale, void *workspace,
                                             size_t workspace_bytes, int ctas,
                                             attn_stream_t stream) {
    if (ctas <= 0) return ATTN_ERR_INVALID_ARG;
    return decode_paged_impl(q, k_cache, v_cache, nullptr, nullptr, kCacheBf16, page_table,
                             seq_lens, o, lse,
                             B, Hq, Hkv, d, page_size, num_pages, max_pages_per_seq, -1, scale,
                             workspace, workspace_bytes, stream, ctas);
}

// ---------------------------------------------------------------- no-allocation decode
// Scratch for attn_decode_paged_noalloc: a fixed device array that every GPU
// loading this library holds until exit.  Host code only ever sees a host-side
// stand-in for its name; the device address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];
}  // namespace

attn_status_t attn_decode_paged_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *page_table, const int32_t *seq_lens,
                                        void *o, float *lse, int B, int Hq, int Hkv, int d,
                                        int page_size, int num_pages, int max_pages_per_seq,
                                        float scale, attn_stream_t stream) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || page_size <= 0 || max_pages_per_seq <= 0)
        return ATTN_ERR_INVALID_ARG;
    // the device's set-up first, so that its own status (an unusable device, a device
    // index past the library's table) is what the caller sees
    DeviceState *st = nullptr;
    attn_status_t s = device_state(&st);
    if (s != ATTN_OK) return s;
    const size_t need = attn_decode_workspace_size(B, Hq, d, max_pages_per_seq, page_size);
    if (need > (size_t)ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            // once per device, with that device current
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr) return cuda_fail(e);
            g_noalloc_ptr[dev] = ptr;
        }
        scratch = g_noalloc_ptr[dev];
    }
    return attn_decode_paged(q, k_cache, v_cache, page_table, seq_lens, o, lse, B, Hq, Hkv, d,
                             page_size, num_pages, max_pages_per_seq, scale, scratch,
                             (size_t)ATTN_NOALLOC_SCRATCH_BYTES, stream);
}

// ---------------------------------------------------------------- wait-bound self-test
// Result words of selftest_wait_timeout_kernel (a fixed device array: the check needs
// no allocation and runs on whatever device is current).
static __device__ unsigned long long g_selftest_out[4];

attn_status_t attn_selftest_wait_timeout(unsigned long long *elapsed_ns, attn_stream_t stream) {
    DeviceState *st = nullptr;
    attn_status_t s = device_state(&st);
    if (s != ATTN_OK) return s;
    void *dout = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&dout, g_selftest_out);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    selftest_wait_timeout_kernel<<<1, 64, 0, cs>>>(st->status,
                                                   static_cast<unsigned long long *>(dout));
    if ((s = launch_status()) != ATTN_OK) return s;
    unsigned long long h[4];
    if ((e = cudaMemcpyFromSymbolAsync(h, g_selftest_out, sizeof(h), 0, cudaMemcpyDeviceToHost,
                                       cs)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaStreamSynchronize(cs)) != cudaSuccess) return cuda_fail(e);
    if (elapsed_ns) {
        elapsed_ns[0] = h[1];
        elapsed_ns[1] = h[3];
    }
    // as designed: neither wait succeeded; warp 0 ran to the bound, warp 1 left on the
    // abort flag before its own bound (kSelftestStaggerNs + kWaitLimitNs after the start)
    const bool as_designed = h[0] == 0 && h[2] == 0 && h[1] >= kWaitLimitNs &&
                             h[3] < kSelftestStaggerNs + kWaitLimitNs;
    if (!as_designed) {
        snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                 "wait self-test: results %llu %llu, %llu ns and %llu ns", h[0], h[2], h[1], h[3]);
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

// ---------------------------------------------------------------- prefill from host memory
// attn_fwd_host: the work is cut into G groups of consecutive key/value heads (with their
// query heads).  Group c's Q/K/V slices are copied into one of NB device buffer sets on
// the copy-in stream, attention runs on the caller's stream, and the O/LSE slices go back
// on the copy-out stream; events order the three, so the copy in of group c + 1, the
// compute of group c and the copy out of group c - 1 overlap (a host-to-device copy,
// a kernel and a device-to-host copy use different engines).
namespace {

constexpr int kHostMaxGroups = 16;
constexpr int kHostSets = 2;

struct HostStaging {
    void *buf = nullptr;
    size_t bytes = 0;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t e_in[kHostMaxGroups], e_comp[kHostMaxGroups], e_out[kHostMaxGroups];
    bool ready = false;
};
std::mutex g_host_mu;
HostStaging g_host[kMaxDevices];

attn_status_t host_staging_init(HostStaging &h) {
    if (h.ready) return ATTN_OK;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&h.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&h.s_out, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e);
    for (int c = 0; c < kHostMaxGroups; ++c) {
        if ((e = cudaEventCreateWithFlags(&h.e_in[c], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&h.e_comp[c], cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&h.e_out[c], cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e);
    }
    h.ready = true;
    return ATTN_OK;
}

void host_staging_release(HostStaging &h) {
    if (!h.ready) return;
    cudaStreamSynchronize(h.s_in);
    cudaStreamSynchronize(h.s_out);
    if (h.buf) cudaFree(h.buf);
    h.buf = nullptr;
    h.bytes = 0;
    for (int c = 0; c < kHostMaxGroups; ++c) {
        cudaEventDestroy(h.e_in[c]);
        cudaEventDestroy(h.e_comp[c]);
        cudaEventDestroy(h.e_out[c]);
    }
    cudaStreamDestroy(h.s_in);
    cudaStreamDestroy(h.s_out);
    h.ready = false;
}

inline size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// `height` rows of `width` bytes, `spitch` / `dpitch` bytes apart: one plain copy when the
// rows are contiguous on both sides (or there is one row, where a pitch would only have
// to satisfy the 2-D copy's pitch limit for nothing), else a 2-D copy.
cudaError_t copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                      size_t height, cudaMemcpyKind kind, cudaStream_t stream) {
    if (height == 1 || (dpitch == width && spitch == width))
        return cudaMemcpyAsync(dst, src, width * height, kind, stream);
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, stream);
}

// Number of key/value head groups: a divisor of Hkv, at most 4 (each group then moves
// at least a quarter of the tensors per copy call), at least 1.
int host_groups(int Hkv) {
    for (int g = 4; g > 1; --g)
        if (Hkv % g == 0) return g;
    return 1;
}

}  // namespace

attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                            attn_stream_t stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if ((long long)B * N * Hq * d > (1LL << 40)) return ATTN_ERR_UNSUPPORTED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;

    std::lock_guard<std::mutex> lock(g_host_mu);
    HostStaging &h = g_host[dev];
    attn_status_t st = host_staging_init(h);
    if (st != ATTN_OK) return st;
    cudaStream_t sc = reinterpret_cast<cudaStream_t>(stream);
    auto reserve = [&](size_t bytes) -> attn_status_t {
        if (h.bytes >= bytes) return ATTN_OK;
        cudaError_t e2;
        if (h.buf) {
            if ((e2 = cudaFree(h.buf)) != cudaSuccess) return cuda_fail(e2);
            h.buf = nullptr;
            h.bytes = 0;
        }
        if ((e2 = cudaMalloc(&h.buf, bytes)) != cudaSuccess) return cuda_fail(e2);
        h.bytes = bytes;
        return ATTN_OK;
    };
    const char *hq_src = static_cast<const char *>(q);
    const char *hk_src = static_cast<const char *>(k);
    const char *hv_src = static_cast<const char *>(v);
    char *ho = static_cast<char *>(o);
    const size_t rows = (size_t)B * N;
    // the copies wait for work the caller queued on its stream before this call
    if ((e = cudaEventRecord(h.e_out[0], sc)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaStreamWaitEvent(h.s_in, h.e_out[0], 0)) != cudaSuccess) return cuda_fail(e);

    if (causal) {
        // Causal: query rows [n0, n1) need keys [0, n1) only, so the work is cut along
        // the sequence.  Chunk c's rows of Q, K and V (contiguous per sequence) are
        // copied in order; its query tiles run once chunks 0..c are in place; its rows
        // of O and LSE go back while later chunks are copied in and computed.
        const size_t tq = (size_t)Hq * d * 2, tkv = (size_t)Hkv * d * 2;  // bytes per token
        const size_t q_bytes = round256(rows * tq), kv_bytes = round256(rows * tkv);
        const size_t lse_bytes = lse ? round256(rows * Hq * 4) : 0;
        if ((st = reserve(2 * q_bytes + 2 * kv_bytes + lse_bytes)) != ATTN_OK) return st;
        char *dq = static_cast<char *>(h.buf), *dout = dq + q_bytes, *dk = dout + q_bytes;
        char *dv = dk + kv_bytes;
        float *dlse = lse ? reinterpret_cast<float *>(dv + kv_bytes) : nullptr;
        const int ntiles = (N + 127) / 128;
        // pieces of whole 256-row pairs of tiles, about sixteen of them: the last piece's
        // compute and copy out are all that is left once the copies in are done
        const int tiles_per = std::max(2, ((ntiles + 15) / 16 + 1) & ~1);
        const int C = (ntiles + tiles_per - 1) / tiles_per;
        for (int c = 0; c < C && st == ATTN_OK; ++c) {
            const int t0 = c * tiles_per, t1 = std::min(ntiles, t0 + tiles_per);
            const size_t n0 = (size_t)t0 * 128, n1 = std::min((size_t)N, (size_t)t1 * 128);
            const size_t nr = n1 - n0;
            if ((e = copy_rows(dq + n0 * tq, (size_t)N * tq, hq_src + n0 * tq, (size_t)N * tq,
                                       nr * tq, B, cudaMemcpyHostToDevice, h.s_in)) != cudaSuccess ||
                (e = copy_rows(dk + n0 * tkv, (size_t)N * tkv, hk_src + n0 * tkv,
                                       (size_t)N * tkv, nr * tkv, B, cudaMemcpyHostToDevice,
                                       h.s_in)) != cudaSuccess ||
                (e = copy_rows(dv + n0 * tkv, (size_t)N * tkv, hv_src + n0 * tkv,
                                       (size_t)N * tkv, nr * tkv, B, cudaMemcpyHostToDevice,
                                       h.s_in)) != cudaSuccess ||
                (e = cudaEventRecord(h.e_in[c], h.s_in)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(sc, h.e_in[c], 0)) != cudaSuccess) {
                st = cuda_fail(e);
                break;
            }
            st = launch_prefill_tc(dq, dk, dv, dout, dlse, nullptr, B, N, t1 - t0, Hq, Hkv, d, -1,
                                   0, scale, sc, nullptr, 0, t0);
            if (st != ATTN_OK) break;
            if ((e = cudaEventRecord(h.e_comp[c], sc)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(h.s_out, h.e_comp[c], 0)) != cudaSuccess ||
                (e = copy_rows(ho + n0 * tq, (size_t)N * tq, dout + n0 * tq, (size_t)N * tq,
                                       nr * tq, B, cudaMemcpyDeviceToHost, h.s_out)) != cudaSuccess ||
                (lse && (e = copy_rows(lse + n0, (size_t)N * 4, dlse + n0, (size_t)N * 4,
                                               nr * 4, (size_t)B * Hq, cudaMemcpyDeviceToHost,
                                               h.s_out)) != cudaSuccess))
                st = cuda_fail(e);
        }
    } else {
        // Full attention: every row needs every key, so the work is cut by groups of
        // key/value heads (with their query heads) over two device buffer sets.
        const int G = host_groups(Hkv);
        const int hk = Hkv / G, hq = Hq / G;
        const size_t row_q = (size_t)hq * d * 2, row_kv = (size_t)hk * d * 2;  // per token
        const size_t q_bytes = round256(rows * row_q), kv_bytes = round256(rows * row_kv);
        const size_t lse_bytes = lse ? round256((size_t)B * hq * N * 4) : 0;
        const size_t set_bytes = 2 * q_bytes + 2 * kv_bytes + lse_bytes;  // Q, O, K, V, LSE
        if ((st = reserve(kHostSets * set_bytes)) != ATTN_OK) return st;
        for (int c = 0; c < G && st == ATTN_OK; ++c) {
            char *set = static_cast<char *>(h.buf) + (size_t)(c % kHostSets) * set_bytes;
            char *dq = set, *dout = set + q_bytes, *dk = set + 2 * q_bytes;
            char *dv = dk + kv_bytes;
            float *dlse = lse ? reinterpret_cast<float *>(dv + kv_bytes) : nullptr;
            // copy in: the set's inputs are free once the compute of group c - NB is done
            if (c >= kHostSets &&
                (e = cudaStreamWaitEvent(h.s_in, h.e_comp[c - kHostSets], 0)) != cudaSuccess)
                st = cuda_fail(e);
            if (st == ATTN_OK &&
                ((e = copy_rows(dq, row_q, hq_src + (size_t)c * row_q, (size_t)Hq * d * 2,
                                        row_q, rows, cudaMemcpyHostToDevice, h.s_in)) != cudaSuccess ||
                 (e = copy_rows(dk, row_kv, hk_src + (size_t)c * row_kv, (size_t)Hkv * d * 2,
                                        row_kv, rows, cudaMemcpyHostToDevice, h.s_in)) != cudaSuccess ||
                 (e = copy_rows(dv, row_kv, hv_src + (size_t)c * row_kv, (size_t)Hkv * d * 2,
                                        row_kv, rows, cudaMemcpyHostToDevice, h.s_in)) != cudaSuccess ||
                 (e = cudaEventRecord(h.e_in[c], h.s_in)) != cudaSuccess))
                st = cuda_fail(e);
            // compute: after its inputs, and once the copy out of group c - NB freed O / LSE
            if (st == ATTN_OK && (e = cudaStreamWaitEvent(sc, h.e_in[c], 0)) != cudaSuccess)
                st = cuda_fail(e);
            if (st == ATTN_OK && c >= kHostSets &&
                (e = cudaStreamWaitEvent(sc, h.e_out[c - kHostSets], 0)) != cudaSuccess)
                st = cuda_fail(e);
            if (st == ATTN_OK)
                st = attn_fwd(dq, dk, dv, dout, dlse, B, hq, hk, N, d, 0, scale, stream);
            if (st == ATTN_OK && (e = cudaEventRecord(h.e_comp[c], sc)) != cudaSuccess)
                st = cuda_fail(e);
            // copy out: O rows into the group's head slice, LSE [B, Hq, N] rows of this group
            if (st == ATTN_OK &&
                ((e = cudaStreamWaitEvent(h.s_out, h.e_comp[c], 0)) != cudaSuccess ||
                 (e = copy_rows(ho + (size_t)c * row_q, (size_t)Hq * d * 2, dout, row_q,
                                        row_q, rows, cudaMemcpyDeviceToHost, h.s_out)) != cudaSuccess ||
                 (lse && (e = copy_rows(lse + (size_t)c * hq * N, (size_t)Hq * N * 4, dlse,
                                                (size_t)hq * N * 4, (size_t)hq * N * 4, (size_t)B,
                                                cudaMemcpyDeviceToHost, h.s_out)) != cudaSuccess) ||
                 (e = cudaEventRecord(h.e_out[c], h.s_out)) != cudaSuccess))
                st = cuda_fail(e);
        }
    }
    // o and lse are complete (or the call failed) when both copy streams and the compute
    // stream have drained; nothing of this call is left in flight
    cudaError_t e1 = cudaStreamSynchronize(h.s_in);
    cudaError_t e2 = cudaStreamSynchronize(sc);
    cudaError_t e3 = cudaStreamSynchronize(h.s_out);
    if (st == ATTN_OK && e1 != cudaSuccess) st = cuda_fail(e1);
    if (st == ATTN_OK && e2 != cudaSuccess) st = cuda_fail(e2);
    if (st == ATTN_OK && e3 != cudaSuccess) st = cuda_fail(e3);
    return st;
}

attn_status_t attn_release_host_staging(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_host_mu);
    host_staging_release(g_host[dev]);
    return ATTN_OK;
}

}  // extern "C"
