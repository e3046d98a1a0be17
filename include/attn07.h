/*
 * attn07.h -- C ABI of the B300 (sm_103a) exact-attention library libattn07.so.
 *
 * Operation.  Exact scaled-dot-product attention, O = softmax(Q K^T * scale) V,
 * as stated in "Donanıma Duyarlı Algoritma Tasarımı: FlashAttention"
 * (fatihsoysal.com), section "Transformer Mimarisi ve Self-Attention
 * Mekanizması" (the attention formula; Q, K, V are (sequence, dimension)
 * matrices; the softmax is taken over each row of Q K^T).  The result is the
 * exact one, not an approximation (yapayzekasozluk.tr "attention" tag page,
 * entry "Flash Attention"), computed tile by tile on chip with the online
 * softmax of the same fatihsoysal.com page, section "Online Softmax
 * Prensibi", so that the N x N score matrix never reaches device memory.
 *
 * For query head h the key/value head is h / (Hq / Hkv): groups of Hq/Hkv
 * consecutive query heads share one key/value head (grouped-query attention,
 * yapayzekasozluk.tr "attention" tag page, entry "KV Cache").
 *
 * Log-sum-exp output.  Where an `lse` pointer is accepted, row r receives
 * LSE_r = ln sum_j exp(s_rj) over the row's allowed keys, s_rj = scale * q_r . k_j
 * (natural log, of the scaled scores), in fp32.  A row with no allowed key gets
 * O = 0 and LSE = -inf.  `lse` may be NULL when it is not wanted.
 *
 * Causal masking.  With causal != 0, query i of a sequence sees keys j <= i
 * (queries and keys of a sequence share positions).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, owned by the caller; the
 *     library allocates, frees and synchronises nothing.  Two exceptions by
 *     design: attn_get_device_status synchronises `stream`, and attn_fwd_host
 *     (HOST pointers) keeps a device staging area and returns when its outputs
 *     are written.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and runs asynchronously; the return value reports argument
 *     validation and launch errors only.  Calls may run concurrently on
 *     different streams.  The tensor-core prefill takes its work items from a
 *     counter in a library-owned device array of 1024 slots, one per launch in
 *     turn, which each launch leaves at zero when it ends: a launch must end
 *     before the 1024th prefill launch after it in the same process starts.
 *   - Invalid arguments return ATTN_ERR_INVALID_ARG and launch nothing;
 *     sizes outside what the kernels implement return ATTN_ERR_UNSUPPORTED and
 *     launch nothing.  Launch failures return ATTN_ERR_CUDA.
 *   - `scale` must be finite and > 0 (1/sqrt(d) in the usual case); any other
 *     value returns ATTN_ERR_INVALID_ARG.
 *   - Errors found on the device never fault the device: the kernel records
 *     them in a device status word, skips the access, and
 *     attn_get_device_status() reports them.  They are: a page id out of
 *     range, a sequence length outside what the page table can hold, a
 *     cu_seqlens vector that breaks its rules (ATTN_ERR_DEVICE_BOUNDS), and a
 *     pipeline wait that ran past its bound (ATTN_ERR_TIMEOUT).
 *   - Entry points are thread-safe and re-entrant.
 *   - bf16 means IEEE bfloat16 (1-8-7) stored in 2 bytes, round-to-nearest-even
 *     on output.
 */
#ifndef ATTN07_H
#define ATTN07_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, Hq % Hkv != 0, ... */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head dim, page size, ...) */
    ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
    ATTN_ERR_TIMEOUT = 4,      /* a device-side pipeline wait ran past its bound */
    ATTN_ERR_DEVICE_BOUNDS = 5 /* the device found an index or length out of range */
} attn_status_t;

/*
 * attn_fwd -- batched prefill attention, bf16 in, bf16 out.
 * Source: the attention formula (fatihsoysal.com page, section "Transformer
 * Mimarisi ve Self-Attention Mekanizması") computed with the tiling and online
 * softmax of sections "FlashAttention'ın Temelleri" and "Online Softmax
 * Prensibi", work split over query-row tiles as in section
 * "FlashAttention-2: Optimizasyonlar ve İyileştirmeler".
 *   q   [B, N, Hq,  d] bf16, contiguous (token-major, then head, then dim)
 *   k,v [B, N, Hkv, d] bf16, contiguous
 *   o   [B, N, Hq,  d] bf16, written
 *   lse [B, Hq, N]     fp32, written, or NULL
 *   B >= 1, N >= 1, Hq >= 1, Hkv >= 1, Hq % Hkv == 0.
 *   d must be 64 or 128 (else ATTN_ERR_UNSUPPORTED).  scale is typically
 *   1/sqrt(d).  Pointers must be 16-byte aligned.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                       attn_stream_t stream);

/*
 * attn_fwd_host -- attn_fwd with every tensor in HOST memory: q, k, v are read
 * from the host, o and lse are written to the host, and the call returns when
 * they hold the result (or an error).  Same layouts, sizes, values and errors
 * as attn_fwd, except that the pointers need no alignment and are host
 * pointers (page-locked memory lets the copies run asynchronously; pageable
 * memory works, with the copies serialised by the driver).
 * How: inputs are copied to the device on a library stream, attention runs on
 * `stream`, results are copied back on a second library stream, in pieces
 * ordered by events so that copy in, compute and copy out overlap.  Causal:
 * the pieces are runs of about a sixteenth of the sequence (whole 256-row
 * query tile pairs); rows [n0, n1) need keys [0, n1) only, so a piece's query tiles
 * run as soon as its own rows and the earlier ones are on the device.  Full
 * attention: the pieces are up to four groups of key/value heads (a divisor of
 * Hkv) with their query heads, over two device buffer sets.  Either way every
 * row's result is bitwise the one attn_fwd gives on the whole tensors (a row's
 * arithmetic depends on neither the other rows' tiles nor the other heads).
 * Device memory: a staging area per device (the whole tensors for a causal
 * call; two groups' slices for full attention), allocated on first use, grown
 * when a larger call needs it, and kept for the next call;
 * attn_release_host_staging frees it.
 * Calls on one device are serialised by a lock.  Work the caller queued on
 * `stream` before the call completes before the copies start.
 */
attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                            attn_stream_t stream);

/* Frees the current device's attn_fwd_host staging area and its streams and
 * events (after the copies in flight, if any, have finished).  Returns ATTN_OK,
 * or ATTN_ERR_CUDA if the current device cannot be read. */
attn_status_t attn_release_host_staging(void);

/*
 * attn_fwd_window -- attn_fwd with local ("sliding window") attention: query i
 * of a sequence sees only keys j with  i - window_left <= j <= i + window_right
 * (yapayzekasozluk.tr "attention" tag page, entry "Sliding Window Attention":
 * each token attends to the tokens within a window around its own position,
 * w/2 on either side in the page's form, so the work grows as N * w instead of
 * N^2).  window_left / window_right >= 0 bound that side; -1 leaves it
 * unbounded: (-1, 0) is causal attention, (-1, -1) full attention, (w/2, w/2)
 * the page's symmetric window.  Every row sees at least its own key.  Key tiles
 * wholly outside a row block's window are skipped.  Layouts, sizes and errors
 * as attn_fwd; window values below -1 return ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int Hq, int Hkv, int N, int d, int window_left,
                              int window_right, float scale, attn_stream_t stream);

/*
 * attn_fwd_two_pass -- attn_fwd computed in the two-pass order that
 * "Donanıma Duyarlı Algoritma Tasarımı: FlashAttention" (fatihsoysal.com)
 * describes in section "FlashAttention-1 (İki Geçişli Yaklaşım)": a first pass
 * over all key tiles computes only each row's maximum M and sum L (no values,
 * no output), a second pass recomputes Q K^T, normalises with M and L and
 * accumulates O, with no running rescaling.  Same result as attn_fwd up to
 * rounding; it repeats the Q K^T work (about 1.5x the tensor work of attn_fwd)
 * and is kept as an independent evaluation order.  The statistics travel
 * between the passes in `lse` (LSE = M + ln L), which is therefore required:
 * lse == NULL returns ATTN_ERR_INVALID_ARG.  Arguments otherwise as attn_fwd.
 */
attn_status_t attn_fwd_two_pass(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                                attn_stream_t stream);

/*
 * attn_fwd_chunked_paged -- a chunk of new queries per sequence against that
 * sequence's paged key/value cache: chunked prefill, and prefill after a reused
 * (cached) prompt prefix (yapayzekasozluk.tr "attention" tag page, entry "KV
 * Cache": earlier tokens' keys and values, including a shared prefix, are kept
 * in fixed-size pages and new tokens attend to them).  The same tensor-core
 * kernel as attn_fwd, with each 128-key tile gathered from eight pages.
 *   q            [total_q, Hq, d] bf16: sequence s's chunk is rows
 *                cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1
 *   k_cache,
 *   v_cache      [num_pages, page_size, Hkv, d] bf16, page_table int32
 *                [num_seqs, max_pages_per_seq] (as attn_decode_paged)
 *   seq_lens     int32 [num_seqs], DEVICE: cached tokens of sequence s, the chunk's
 *                own tokens included -- the caller appends the chunk's keys and
 *                values before the call; chunk query i sits at position
 *                seq_lens[s] - q_len + i.  Needs q_len <= seq_lens[s] <=
 *                max_pages_per_seq * page_size; a sequence that breaks this is
 *                skipped and ATTN_ERR_DEVICE_BOUNDS recorded.
 *   cu_seqlens_q int32 [num_seqs + 1], DEVICE, with the rules and device checks
 *                of attn_fwd_varlen's cu_seqlens (over total_q tokens); max_qlen
 *                a host-side bound on every q_len, checked as max_seqlen is.
 *   o            [total_q, Hq, d] bf16;  lse [Hq, total_q] fp32 or NULL.
 *   causal != 0: query i sees positions <= its own; else all cached tokens.
 *   A page id out of range is recorded as ATTN_ERR_DEVICE_BOUNDS and its tokens
 *   are read as zero keys and values (never from outside the cache).
 *   Supported: page_size == 16, d in {64, 128}.
 */
attn_status_t attn_fwd_chunked_paged(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *page_table, const int32_t *seq_lens,
                                     const int32_t *cu_seqlens_q, void *o, float *lse,
                                     int num_seqs, int total_q, int max_qlen, int Hq, int Hkv,
                                     int d, int page_size, int num_pages, int max_pages_per_seq,
                                     int causal, float scale, attn_stream_t stream);

/*
 * attn_fwd_f32 -- the same operation with fp32 q, k, v and o: the attention
 * formula of the fatihsoysal.com page, section "Transformer Mimarisi ve
 * Self-Attention Mekanizması", in its plain form where Q, K and V are each a
 * (sequence length, dimension) matrix of real numbers, computed tile by tile
 * with the online softmax of section "Online Softmax Prensibi".  Arithmetic is
 * fp32 throughout, on the CUDA cores (no reduced-precision tensor-core path).
 * Same layouts and rules as attn_fwd, except the head dimension:
 * 16 <= d <= 128 and d % 16 == 0 (else ATTN_ERR_UNSUPPORTED).  B <= 65535 and
 * Hq <= 65535.
 */
attn_status_t attn_fwd_f32(const float *q, const float *k, const float *v, float *o,
                           float *lse, int B, int Hq, int Hkv, int N, int d, int causal,
                           float scale, attn_stream_t stream);

/*
 * attn_fwd_varlen -- prefill over a batch of requests of different lengths
 * (yapayzekasozluk.tr "attention" tag page, entry "KV Cache": batched inference
 * serves requests of different lengths together), packed along the token axis
 * with no padding.  Each sequence is an independent problem of the attention
 * formula (fatihsoysal.com page, section "Transformer Mimarisi ve
 * Self-Attention Mekanizması"), computed as in attn_fwd.
 *   q   [total_tokens, Hq,  d] bf16      k,v [total_tokens, Hkv, d] bf16
 *   o   [total_tokens, Hq,  d] bf16      lse [Hq, total_tokens] fp32 or NULL
 *   cu_seqlens  int32 [num_seqs + 1], DEVICE pointer: sequence s owns tokens
 *               cu_seqlens[s] .. cu_seqlens[s+1]-1; cu_seqlens[0] = 0,
 *               non-decreasing, cu_seqlens[num_seqs] = total_tokens.
 *   max_seqlen  host-side upper bound on every sequence length (sizes the
 *               launch).
 *   Zero-length sequences are allowed.  d must be 64 or 128.
 *   Checked on the device, each recording ATTN_ERR_DEVICE_BOUNDS: a sequence
 *   whose tokens leave [0, total_tokens) or whose length is negative is skipped
 *   (nothing of it is read or written); a sequence longer than the launch's
 *   query tiles (ceil(max_seqlen / 128) tiles of 128 rows) has only the rows
 *   of those tiles written; cu_seqlens[0] != 0 or cu_seqlens[num_seqs] !=
 *   total_tokens leaves the rows outside the sequences unwritten.
 */
attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                              int max_seqlen, int Hq, int Hkv, int d, int causal, float scale,
                              attn_stream_t stream);

/*
 * attn_decode_paged -- one new query token per sequence attending to that
 * sequence's cached keys and values held in fixed-size pages
 * (yapayzekasozluk.tr "attention" tag page, entry "KV Cache": cached keys and
 * values, grouped query heads, a cache kept in fixed-size pages).  The query
 * sees every cached token (no mask).  The key range of each sequence is split
 * over the GPU, each piece is attended with the online softmax, and the pieces
 * are combined by their log-sum-exps (the rescaling rule of section "Online
 * Softmax Prensibi" of the fatihsoysal.com page).
 *   q           [B, Hq, d] bf16
 *   k_cache,
 *   v_cache     [num_pages, page_size, Hkv, d] bf16
 *   page_table  int32 [B, max_pages_per_seq]: entry p of sequence b is the
 *               physical page holding its tokens p*page_size .. p*page_size+page_size-1;
 *               only the first ceil(seq_lens[b]/page_size) entries are read.
 *   seq_lens    int32 [B]: cached tokens per sequence, 0 <= seq_lens[b] <=
 *               max_pages_per_seq * page_size.  DEVICE pointer (read on the device).
 *               A sequence outside that range is treated as empty (its page
 *               table row is not read; O = 0, LSE = -inf) and
 *               ATTN_ERR_DEVICE_BOUNDS is recorded.
 *   o           [B, Hq, d] bf16, written;  lse [B, Hq] fp32 or NULL.
 *   workspace   device scratch of at least attn_decode_workspace_size(...) bytes,
 *               16-byte aligned, owned by the caller; its contents on entry do
 *               not matter and are overwritten.
 *   Supported: page_size == 16, d in {64, 128}, Hq/Hkv <= 8, Hkv <= 8 (one
 *   consumer warp per key/value head); other sizes return ATTN_ERR_UNSUPPORTED.
 *   A page id outside [0, num_pages) is not read: its tokens are treated as
 *   masked and ATTN_ERR_DEVICE_BOUNDS is recorded for attn_get_device_status.
 *   A sequence with seq_lens[b] == 0 gets O = 0, LSE = -inf.
 */
attn_status_t attn_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *page_table, const int32_t *seq_lens, void *o,
                                float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                int num_pages, int max_pages_per_seq, float scale,
                                void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_paged_fp8 -- attn_decode_paged against a cache held in 8-bit
 * floating point (yapayzekasozluk.tr "attention" tag page, entry "KV Cache":
 * keeping the cache in INT8/FP8 cuts its memory 2-4x at a small cost in
 * quality).  The decode is bound by reading the cache, so halving its bytes
 * roughly halves the time of a step.
 *   k_cache,
 *   v_cache     [num_pages, page_size, Hkv, d] uint8: FP8 E4M3 ("E4M3FN": bias 7,
 *               no infinities, 0x7f/0xff NaN) bytes
 *   k_scale,
 *   v_scale     float32 [Hkv], DEVICE pointers: element c of head g of a cached key
 *               (value) stands for k_scale[g] * e4m3 (v_scale[g] * e4m3)
 *   q, o, lse, page_table, seq_lens, workspace and their rules as attn_decode_paged.
 *   Inside the kernel the cache is widened to f16 (exactly) and q is rounded to
 *   f16 (exact for |q| below 65504; larger values are not supported); scores and
 *   sums are fp32.  Supported: d == 128, page_size == 16, Hkv <= 8, Hq/Hkv <= 8.
 */
attn_status_t attn_decode_paged_fp8(const void *q, const void *k_cache, const void *v_cache,
                                    const float *k_scale, const float *v_scale,
                                    const int32_t *page_table, const int32_t *seq_lens, void *o,
                                    float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                    int num_pages, int max_pages_per_seq, float scale,
                                    void *workspace, size_t workspace_bytes,
                                    attn_stream_t stream);

/*
 * attn_decode_paged_int8 -- attn_decode_paged against a cache held as 8-bit
 * integers (the same "KV Cache" entry of the yapayzekasozluk.tr "attention" tag
 * page: INT8 or FP8 storage of the cache, 2-4x less memory).  The decode reads
 * half the bytes of a bf16 cache, like the FP8 form.
 *   k_cache,
 *   v_cache     [num_pages, page_size, Hkv, d] int8 (two's complement bytes,
 *               -128 .. 127)
 *   k_scale,
 *   v_scale     float32 [Hkv], DEVICE pointers: element c of head g of a cached key
 *               (value) stands for k_scale[g] * int8 (v_scale[g] * int8)
 *   q, o, lse, page_table, seq_lens, workspace and their rules as attn_decode_paged.
 *   Inside the kernel the cache is widened to f16 (exactly: every int8 is an f16)
 *   and q is rounded to f16 (exact for |q| below 65504; larger values are not
 *   supported); scores and sums are fp32.  Null k_scale or v_scale returns
 *   ATTN_ERR_INVALID_ARG.  Supported: d == 128, page_size == 16, Hkv <= 8,
 *   Hq/Hkv <= 8.
 */
attn_status_t attn_decode_paged_int8(const void *q, const void *k_cache, const void *v_cache,
                                     const float *k_scale, const float *v_scale,
                                     const int32_t *page_table, const int32_t *seq_lens, void *o,
                                     float *lse, int B, int Hq, int Hkv, int d, int page_size,
                                     int num_pages, int max_pages_per_seq, float scale,
                                     void *workspace, size_t workspace_bytes,
                                     attn_stream_t stream);

/*
 * attn_decode_paged_window -- attn_decode_paged where the new query attends only
 * to the last window + 1 cached tokens of its sequence (positions
 * seq_lens[b] - 1 - window .. seq_lens[b] - 1): the decode side of local
 * attention (yapayzekasozluk.tr "attention" tag page, entry "Sliding Window
 * Attention": each token attends to a fixed window of neighbours, so per-token
 * cost and the cache a step reads stay constant as the sequence grows).  Only
 * the pages holding those tokens are read; the page table may still list the
 * older pages.  window = -1 attends to every cached token (attn_decode_paged);
 * window < -1 returns ATTN_ERR_INVALID_ARG.  Everything else as
 * attn_decode_paged, including the workspace size.
 */
attn_status_t attn_decode_paged_window(const void *q, const void *k_cache, const void *v_cache,
                                       const int32_t *page_table, const int32_t *seq_lens,
                                       void *o, float *lse, int B, int Hq, int Hkv, int d,
                                       int page_size, int num_pages, int max_pages_per_seq,
                                       int window, float scale, void *workspace,
                                       size_t workspace_bytes, attn_stream_t stream);

/*
 * Bytes of workspace attn_decode_paged (and attn_decode_paged_window,
 * attn_decode_paged_fp8) needs for these sizes on the current device: the
 * partial outputs and log-sum-exps of the split key ranges (fp32).  0 on
 * invalid sizes or when the device cannot be queried.  It depends only on B,
 * Hq, d and the GPU's SM count, never on the sequence lengths.
 */
size_t attn_decode_workspace_size(int B, int Hq, int d, int max_pages_per_seq, int page_size);

/* Static, human-readable text for a status code. */
const char *attn_status_string(attn_status_t s);

/*
 * Synchronises `stream`, then reads and clears the device status word shared
 * by all kernels of this library on the current device.  Returns ATTN_OK if no
 * kernel recorded an error since the last call, else the first recorded error
 * (ATTN_ERR_TIMEOUT or ATTN_ERR_DEVICE_BOUNDS), or ATTN_ERR_CUDA if the
 * synchronisation itself failed.
 */
attn_status_t attn_get_device_status(attn_stream_t stream);

/*
 * attn_selftest_wait_timeout -- checks on the device that a pipeline wait whose
 * arrival never comes ends in an error the host can read, not in a hang or a
 * fault.  Every wait of the attention kernels goes through the same bounded
 * wait: after 2 s it records a timeout in the device status word, raises its
 * CTA's abort flag so that the CTA's other waits end too, and lets the kernel
 * return.  This runs one CTA of two waiting warps on barriers nothing arrives
 * on.  Warp 0 waits first and runs to the bound.  Warp 1 starts its wait 0.5 s
 * later and must leave on the abort flag before its own bound.  The call takes
 * about 2 s and synchronises `stream`.
 *   elapsed_ns  host array of 2, or NULL: nanoseconds from the kernel's start
 *               to the end of warp 0's and warp 1's waits.
 * Returns ATTN_OK when both waits ended as described (the status word then
 * holds the timeout: attn_get_device_status returns ATTN_ERR_TIMEOUT once, and
 * the device stays usable), ATTN_ERR_CUDA otherwise (attn_last_cuda_error says
 * what was seen).
 */
attn_status_t attn_selftest_wait_timeout(unsigned long long *elapsed_ns, attn_stream_t stream);

/*
 * attn_decode_paged_noalloc -- attn_decode_paged for callers that cannot
 * allocate device memory: a host that hands the library only its input and
 * output buffers (a plugin interface with no workspace to lend), or a serving
 * process that reserved all device memory up front and may not call cudaMalloc
 * while requests run.  No counterpart on the attention pages: it exists only so
 * those callers can run the paged decode.
 *   Same arguments, layouts and results as attn_decode_paged, without the
 *   workspace.  The scratch it needs lives in a fixed device array compiled
 *   into the library (ATTN_NOALLOC_SCRATCH_BYTES, 8 MiB, held on every GPU that
 *   loads the library until the process exits); sizes whose scratch
 *   (attn_decode_workspace_size) exceeds it return ATTN_ERR_UNSUPPORTED and
 *   launch nothing.  It allocates and frees nothing.
 *   The first call on each device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.  Every call uses the same array: calls whose work overlaps on the
 *   GPU (different streams, or different host threads on one device) race on it
 *   and must be ordered by the caller.  No part of the array needs to start at
 *   zero; each call overwrites what it reads.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
attn_status_t attn_decode_paged_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *page_table, const int32_t *seq_lens,
                                        void *o, float *lse, int B, int Hq, int Hkv, int d,
                                        int page_size, int num_pages, int max_pages_per_seq,
                                        float scale, attn_stream_t stream);

/*
 * Text of the last CUDA runtime or driver failure that made an entry point
 * return ATTN_ERR_CUDA on the calling host thread (error name and message), or
 * "no CUDA error recorded".  The pointer stays valid until the thread's next
 * failing call; the text is not cleared by successful calls.
 */
const char *attn_last_cuda_error(void);

/* Library version, e.g. "attn07 0.1.0 sm_103a". */
const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN07_H */
