/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact scaled-dot-product
 * attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline of the benchmark load this file's library.  The CUDA library never
 * links, includes or calls it, and it shares no code with the CUDA library.
 *
 * What it computes (the definition, written out):
 *   "Donanıma Duyarlı Algoritma Tasarımı: FlashAttention" (fatihsoysal.com),
 *   section "Transformer Mimarisi ve Self-Attention Mekanizması":
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *   Q, K, V are (sequence length, dimension) matrices, Q K^T is the
 *   (sequence, sequence) compatibility matrix, softmax turns each ROW of it
 *   into a probability distribution, and that distribution weights the rows
 *   of V.  The max shift softmax(x) = softmax(x - max x) used below is the
 *   identity the same page states in section "FlashAttention'ın Temelleri".
 *
 *   The scale is passed in by the caller (1/sqrt(d_k) in every workload).
 *   Per query row i of batch b and query head h, with kv head
 *   g = h / (Hq / Hkv) (grouped-query attention: contiguous groups of query
 *   heads share one key/value head -- yapayzekasozluk.tr "attention" tag
 *   page, entry "KV Cache"):
 *       s_j   = scale * sum_c Q[b,i,h,c] * K[b,j,g,c]      for allowed j
 *       m     = max_j s_j
 *       P_j   = exp(s_j - m) / sum_j' exp(s_j' - m)
 *       O_c   = sum_j P_j * V[b,j,g,c]
 *       LSE   = m + ln sum_j exp(s_j - m)
 *   allowed j: all keys; or, when causal, keys j <= i.  A row with no allowed
 *   key (an empty sequence) has O = 0 and LSE = -inf.
 *
 * All arithmetic is fp64.  Inputs arrive as fp32 arrays; every bf16 value is
 * exactly representable in fp32, so the oracle sees exactly the values the
 * GPU sees.  Rows are independent by definition and are spread over OpenMP
 * threads; no blocking, fusion or reordering is done inside a row: the whole
 * score row is materialised, then normalised, then multiplied with V.
 *
 * Layouts (all row-major, contiguous):
 *   dense   q [B, N, Hq, d], k/v [B, N, Hkv, d], o [B, N, Hq, d], lse [B, Hq, N]
 *   varlen  q [T, Hq, d],   k/v [T, Hkv, d],   o [T, Hq, d],   lse [Hq, T]
 *   decode  q [B, Hq, d], caches [P, page_size, Hkv, d], page_table [B, maxp],
 *           seq_lens [B], o [B, Hq, d], lse [B, Hq]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One output row of the definition above.  qrow: d values; krows/vrows:
 * pointers to the n allowed key/value rows, each d values, row r at
 * krow(r).  The key rows are addressed through a callback-free stride table
 * so the same routine serves dense, varlen and paged layouts. */
static void attention_row(const float *qrow, const float *const *krows,
                          const float *const *vrows, int64_t n, int d,
                          double scale, double *s /* n scratch */,
                          double *orow, double *lse)
{
    if (n == 0) {
        for (int c = 0; c < d; ++c) orow[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* the score row s_j = scale * q . k_j */
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += (double)qrow[c] * (double)krows[j][c];
        s[j] = scale * acc;
    }
    /* max shift, then the row's normaliser */
    double m = s[0];
    for (int64_t j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* P_j = exp(s_j - m) / l, then O = P V */
    for (int64_t j = 0; j < n; ++j) s[j] /= l;
    for (int c = 0; c < d; ++c) orow[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double p = s[j];
        const float *vr = vrows[j];
        for (int c = 0; c < d; ++c) orow[c] += p * (double)vr[c];
    }
    *lse = m + log(l);
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of OpenMP threads the library would use for nthreads <= 0. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Dense (batched) attention for a list of rows.  rows holds nrows triples
 * (b, h, i); row r's output goes to o_rows[r*d .. r*d+d) and lse_rows[r].
 * Passing every (b, h, i) gives the full result; passing a sample gives the
 * same values for just those rows (used to check large problems row by row).
 * Nq query rows attend over Nk keys; causal masking keeps key j iff j <= i
 * (queries and keys share position 0).  Returns 0, or -1 on bad arguments.
 */
int oracle_attn_rows(const float *q, const float *k, const float *v,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d,
                     int causal, double scale,
                     const int32_t *rows, int64_t nrows,
                     double *o_rows, double *lse_rows, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 || d <= 0)
        return -1;
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
    int bad = 0;
#pragma omp parallel num_threads(nt) reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        const float **kr = (const float **)malloc(sizeof(float *) * (size_t)(Nk > 0 ? Nk : 1));
        const float **vr = (const float **)malloc(sizeof(float *) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Nq) {
                bad = 1;
                continue;
            }
            const int g = h / group;
            int64_t n = Nk;
            if (causal && (int64_t)i + 1 < n) n = (int64_t)i + 1;
            for (int64_t j = 0; j < n; ++j) {
                kr[j] = k + (((int64_t)b * Nk + j) * Hkv + g) * d;
                vr[j] = v + (((int64_t)b * Nk + j) * Hkv + g) * d;
            }
            const float *qr = q + (((int64_t)b * Nq + i) * Hq + h) * d;
            attention_row(qr, kr, vr, n, d, scale, s, o_rows + r * d, lse_rows + r);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * Full dense attention: o [B, N, Hq, d] (fp64) and lse [B, Hq, N] (fp64).
 */
int oracle_attn_fwd(const float *q, const float *k, const float *v,
                    double *o, double *lse,
                    int B, int Hq, int Hkv, int N, int d,
                    int causal, double scale, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || N < 0 || d <= 0) return -1;
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
#pragma omp parallel num_threads(nt)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        const float **kr = (const float **)malloc(sizeof(float *) * (size_t)(N > 0 ? N : 1));
        const float **vr = (const float **)malloc(sizeof(float *) * (size_t)(N > 0 ? N : 1));
        const int64_t total = (int64_t)B * Hq * N;
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < total; ++r) {
            const int b = (int)(r / ((int64_t)Hq * N));
            const int h = (int)((r / N) % Hq);
            const int i = (int)(r % N);
            const int g = h / group;
            const int64_t n = causal ? (int64_t)i + 1 : N;
            for (int64_t j = 0; j < n; ++j) {
                kr[j] = k + (((int64_t)b * N + j) * Hkv + g) * d;
                vr[j] = v + (((int64_t)b * N + j) * Hkv + g) * d;
            }
            const float *qr = q + (((int64_t)b * N + i) * Hq + h) * d;
            double *orow = o + (((int64_t)b * N + i) * Hq + h) * d;
            attention_row(qr, kr, vr, n, d, scale, s, orow, lse + ((int64_t)b * Hq + h) * N + i);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return 0;
}

/*
 * Local ("sliding window") attention, yapayzekasozluk.tr "attention" tag
 * page, entry "Sliding Window Attention": each token attends only to the
 * tokens within a window around its own position instead of the whole
 * sequence (the page's form: w/2 to the left and w/2 to the right).  Written
 * with separate left and right extents: query i of a sequence of n tokens
 * sees keys j with
 *       i - wl <= j <= i + wr     and 0 <= j < n,
 * where wl < 0 (or wr < 0) means no limit on that side; wl < 0, wr = 0 is
 * causal attention and wl < 0, wr < 0 is full attention.  Same layouts and
 * row list as oracle_attn_rows (queries and keys of the same length N).
 */
int oracle_attn_window_rows(const float *q, const float *k, const float *v,
                            int B, int Hq, int Hkv, int N, int d, int wl, int wr,
                            double scale, const int32_t *rows, int64_t nrows,
                            double *o_rows, double *lse_rows, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || N < 0 || d <= 0) return -1;
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
    int bad = 0;
#pragma omp parallel num_threads(nt) reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        const float **kr = (const float **)malloc(sizeof(float *) * (size_t)(N > 0 ? N : 1));
        const float **vr = (const float **)malloc(sizeof(float *) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= N) {
                bad = 1;
                continue;
            }
            const int g = h / group;
            /* the allowed keys form one contiguous range [lo, hi] */
            int64_t lo = 0, hi = (int64_t)N - 1;
            if (wl >= 0 && (int64_t)i - wl > lo) lo = (int64_t)i - wl;
            if (wr >= 0 && (int64_t)i + wr < hi) hi = (int64_t)i + wr;
            const int64_t n = hi >= lo ? hi - lo + 1 : 0;
            for (int64_t j = 0; j < n; ++j) {
                kr[j] = k + (((int64_t)b * N + lo + j) * Hkv + g) * d;
                vr[j] = v + (((int64_t)b * N + lo + j) * Hkv + g) * d;
            }
            const float *qr = q + (((int64_t)b * N + i) * Hq + h) * d;
            attention_row(qr, kr, vr, n, d, scale, s, o_rows + r * d, lse_rows + r);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * Variable-length packed attention.  Sequence s owns tokens
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of the packed arrays; each sequence is
 * its own independent attention problem (its queries see only its keys).
 * o [T, Hq, d], lse [Hq, T].
 */
int oracle_attn_varlen(const float *q, const float *k, const float *v,
                       double *o, double *lse, const int32_t *cu_seqlens,
                       int num_seqs, int total, int Hq, int Hkv, int d,
                       int causal, double scale, int nthreads)
{
    if (num_seqs < 0 || total < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0)
        return -1;
    if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != total) return -1;
    int64_t maxlen = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int64_t len = (int64_t)cu_seqlens[s + 1] - cu_seqlens[s];
        if (len < 0) return -1;
        if (len > maxlen) maxlen = len;
    }
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
#pragma omp parallel num_threads(nt)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **kr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **vr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < (int64_t)total * Hq; ++r) {
            const int t = (int)(r / Hq);
            const int h = (int)(r % Hq);
            /* find the sequence that owns token t */
            int sq = 0;
            while (cu_seqlens[sq + 1] <= t) ++sq;
            const int64_t start = cu_seqlens[sq];
            const int64_t i = t - start;
            const int64_t len = (int64_t)cu_seqlens[sq + 1] - start;
            const int g = h / group;
            const int64_t n = causal ? i + 1 : len;
            for (int64_t j = 0; j < n; ++j) {
                kr[j] = k + ((start + j) * Hkv + g) * d;
                vr[j] = v + ((start + j) * Hkv + g) * d;
            }
            attention_row(q + ((int64_t)t * Hq + h) * d, kr, vr, n, d, scale, s,
                          o + ((int64_t)t * Hq + h) * d, lse + (int64_t)h * total + t);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return 0;
}

/*
 * Decode against a paged key/value cache (yapayzekasozluk.tr "attention" tag
 * page, entry "KV Cache": the keys and values of earlier tokens are kept and
 * the new token attends to all of them; the cache is held in fixed-size
 * pages).  Sequence b has seq_lens[b] cached tokens; logical token t lives in
 * physical page page_table[b * maxp + t / page_size], slot t % page_size.
 * The single new query of sequence b sees every cached token (no mask).
 * Only the sequences listed in seqs (nseq entries) are computed; their rows
 * go to o_rows[(r*Hq + h)*d ..] and lse_rows[r*Hq + h].
 * Returns 0, or -1 if a page id is out of range or an argument is bad.
 */
int oracle_decode_paged_rows(const float *q, const float *k_cache, const float *v_cache,
                             const int32_t *page_table, const int32_t *seq_lens,
                             int B, int Hq, int Hkv, int d, int page_size,
                             int num_pages, int maxp, double scale,
                             const int32_t *seqs, int nseq,
                             double *o_rows, double *lse_rows, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page_size <= 0)
        return -1;
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
    int64_t maxlen = 0;
    for (int r = 0; r < nseq; ++r) {
        const int b = seqs[r];
        if (b < 0 || b >= B) return -1;
        const int64_t len = seq_lens[b];
        if (len < 0 || len > (int64_t)maxp * page_size) return -1;
        for (int64_t p = 0; p < (len + page_size - 1) / page_size; ++p) {
            const int32_t pid = page_table[(int64_t)b * maxp + p];
            if (pid < 0 || pid >= num_pages) return -1;
        }
        if (len > maxlen) maxlen = len;
    }
#pragma omp parallel num_threads(nt)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **kr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **vr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t rr = 0; rr < (int64_t)nseq * Hq; ++rr) {
            const int r = (int)(rr / Hq);
            const int h = (int)(rr % Hq);
            const int b = seqs[r];
            const int g = h / group;
            const int64_t len = seq_lens[b];
            for (int64_t t = 0; t < len; ++t) {
                const int64_t page = page_table[(int64_t)b * maxp + t / page_size];
                const int64_t off = ((page * page_size + t % page_size) * Hkv + g) * d;
                kr[t] = k_cache + off;
                vr[t] = v_cache + off;
            }
            attention_row(q + ((int64_t)b * Hq + h) * d, kr, vr, len, d, scale, s,
                          o_rows + rr * d, lse_rows + rr);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return 0;
}

/*
 * Decode with a sliding window (yapayzekasozluk.tr "attention" tag page,
 * entry "Sliding Window Attention"): the new query of sequence b, at position
 * seq_lens[b] - 1, sees only the cached tokens within `window` positions
 * before it, i.e. logical tokens max(0, len - 1 - window) .. len - 1; window
 * < 0 means every cached token (then this equals oracle_decode_paged_rows).
 * Page lookup, layouts and the row list as oracle_decode_paged_rows.
 */
int oracle_decode_paged_window_rows(const float *q, const float *k_cache, const float *v_cache,
                                    const int32_t *page_table, const int32_t *seq_lens,
                                    int B, int Hq, int Hkv, int d, int page_size,
                                    int num_pages, int maxp, int window, double scale,
                                    const int32_t *seqs, int nseq,
                                    double *o_rows, double *lse_rows, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page_size <= 0)
        return -1;
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
    int64_t maxlen = 0;
    for (int r = 0; r < nseq; ++r) {
        const int b = seqs[r];
        if (b < 0 || b >= B) return -1;
        const int64_t len = seq_lens[b];
        if (len < 0 || len > (int64_t)maxp * page_size) return -1;
        const int64_t first = (window >= 0 && len - 1 - window > 0) ? len - 1 - window : 0;
        for (int64_t p = first / page_size; p < (len + page_size - 1) / page_size; ++p) {
            const int32_t pid = page_table[(int64_t)b * maxp + p];
            if (pid < 0 || pid >= num_pages) return -1;
        }
        if (len > maxlen) maxlen = len;
    }
#pragma omp parallel num_threads(nt)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **kr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **vr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t rr = 0; rr < (int64_t)nseq * Hq; ++rr) {
            const int r = (int)(rr / Hq);
            const int h = (int)(rr % Hq);
            const int b = seqs[r];
            const int g = h / group;
            const int64_t len = seq_lens[b];
            const int64_t first = (window >= 0 && len - 1 - window > 0) ? len - 1 - window : 0;
            for (int64_t t = first; t < len; ++t) {
                const int64_t page = page_table[(int64_t)b * maxp + t / page_size];
                const int64_t off = ((page * page_size + t % page_size) * Hkv + g) * d;
                kr[t - first] = k_cache + off;
                vr[t - first] = v_cache + off;
            }
            attention_row(q + ((int64_t)b * Hq + h) * d, kr, vr, len - first, d, scale, s,
                          o_rows + rr * d, lse_rows + rr);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return 0;
}

/*
 * A chunk of new queries against a paged cache (prefix caching / chunked
 * prefill; yapayzekasozluk.tr "attention" tag page, entry "KV Cache": the keys
 * and values of earlier tokens, and of a reused prompt prefix, are kept and
 * the new tokens attend to them).  Sequence s has seq_lens[s] cached tokens,
 * the last q_len of which are the chunk's own tokens (the caller appended
 * them to the cache before the call); its queries are rows cu_q[s] ..
 * cu_q[s+1]-1 of q, query i sitting at position seq_lens[s] - q_len + i.
 * Causal: query i sees the cached tokens at positions <= its own; otherwise
 * all seq_lens[s] of them.  Page lookup as oracle_decode_paged_rows.
 * q [Tq, Hq, d]; rows lists (token t of q, head h) pairs; o_rows [n, d],
 * lse_rows [n].  Returns 0, or -1 on a bad argument or page id.
 */
int oracle_chunk_paged_rows(const float *q, const float *k_cache, const float *v_cache,
                            const int32_t *page_table, const int32_t *seq_lens,
                            const int32_t *cu_q, int num_seqs, int total_q, int Hq, int Hkv,
                            int d, int page_size, int num_pages, int maxp, int causal,
                            double scale, const int32_t *rows, int64_t nrows,
                            double *o_rows, double *lse_rows, int nthreads)
{
    if (num_seqs < 0 || total_q < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 ||
        page_size <= 0)
        return -1;
    if (cu_q[0] != 0 || cu_q[num_seqs] != total_q) return -1;
    int64_t maxlen = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int64_t qlen = (int64_t)cu_q[s + 1] - cu_q[s];
        const int64_t len = seq_lens[s];
        if (qlen < 0 || len < qlen || len > (int64_t)maxp * page_size) return -1;
        for (int64_t p = 0; p < (len + page_size - 1) / page_size; ++p) {
            const int32_t pid = page_table[(int64_t)s * maxp + p];
            if (pid < 0 || pid >= num_pages) return -1;
        }
        if (len > maxlen) maxlen = len;
    }
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
    int bad = 0;
#pragma omp parallel num_threads(nt) reduction(| : bad)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **kr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
        const float **vr = (const float **)malloc(sizeof(float *) * (size_t)(maxlen > 0 ? maxlen : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            const int t = rows[2 * r], h = rows[2 * r + 1];
            if (t < 0 || t >= total_q || h < 0 || h >= Hq) {
                bad = 1;
                continue;
            }
            int sq = 0;
            while (cu_q[sq + 1] <= t) ++sq;
            const int64_t qlen = (int64_t)cu_q[sq + 1] - cu_q[sq];
            const int64_t len = seq_lens[sq];
            const int64_t pos = len - qlen + (t - cu_q[sq]);
            const int64_t n = causal ? pos + 1 : len;
            const int g = h / group;
            for (int64_t j = 0; j < n; ++j) {
                const int64_t page = page_table[(int64_t)sq * maxp + j / page_size];
                const int64_t off = ((page * page_size + j % page_size) * Hkv + g) * d;
                kr[j] = k_cache + off;
                vr[j] = v_cache + off;
            }
            attention_row(q + ((int64_t)t * Hq + h) * d, kr, vr, n, d, scale, s,
                          o_rows + r * d, lse_rows + r);
        }
        free(s);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * The value of one FP8 E4M3 byte (OCP 8-bit floating point, "E4M3FN": 1 sign
 * bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities; exponent
 * and mantissa all ones is NaN):
 *     e = 0:   (-1)^s * (m / 8) * 2^(1 - 7)        (subnormal, includes zero)
 *     e > 0:   (-1)^s * (1 + m / 8) * 2^(e - 7)
 */
double oracle_e4m3_value(uint8_t x)
{
    const int sgn = x >> 7, e = (x >> 3) & 15, m = x & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m / 8.0, 1 - 7) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -mag : mag;
}

/*
 * Decode against a paged cache held as one byte per element (yapayzekasozluk.tr
 * "attention" tag page, entry "KV Cache": the cache may be kept in INT8/FP8 to
 * cut its memory 2-4x).  Cached key (value) element c of head g stands for
 * k_scale[g] * value(byte) (v_scale[g] * value(byte)), value() being the byte
 * format's rule; the query attends to those dequantised values exactly as in
 * oracle_decode_paged_rows.  The bytes are dequantised here in fp64, row by
 * row, into scratch rows.
 */
static int decode_paged_bytes_rows(double (*value)(uint8_t), const float *q,
                                   const uint8_t *k_cache, const uint8_t *v_cache,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *page_table, const int32_t *seq_lens,
                                   int B, int Hq, int Hkv, int d, int page_size,
                                   int num_pages, int maxp, double scale,
                                   const int32_t *seqs, int nseq,
                                   double *o_rows, double *lse_rows, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page_size <= 0)
        return -1;
    const int group = Hq / Hkv;
    const int nt = set_threads(nthreads);
    int64_t maxlen = 0;
    for (int r = 0; r < nseq; ++r) {
        const int b = seqs[r];
        if (b < 0 || b >= B) return -1;
        const int64_t len = seq_lens[b];
        if (len < 0 || len > (int64_t)maxp * page_size) return -1;
        for (int64_t p = 0; p < (len + page_size - 1) / page_size; ++p) {
            const int32_t pid = page_table[(int64_t)b * maxp + p];
            if (pid < 0 || pid >= num_pages) return -1;
        }
        if (len > maxlen) maxlen = len;
    }
    const int64_t cap = maxlen > 0 ? maxlen : 1;
#pragma omp parallel num_threads(nt)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)cap);
        /* dequantised key/value rows in fp64 (scale * value is not always a float,
         * so the definition is written out again below on double rows instead of
         * going through attention_row, which reads float rows) */
        double *kd = (double *)malloc(sizeof(double) * (size_t)cap * d);
        double *vd = (double *)malloc(sizeof(double) * (size_t)cap * d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t rr = 0; rr < (int64_t)nseq * Hq; ++rr) {
            const int r = (int)(rr / Hq);
            const int h = (int)(rr % Hq);
            const int b = seqs[r];
            const int g = h / group;
            const int64_t len = seq_lens[b];
            double *orow = o_rows + rr * d;
            if (len == 0) {
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                lse_rows[rr] = -INFINITY;
                continue;
            }
            for (int64_t t = 0; t < len; ++t) {
                const int64_t page = page_table[(int64_t)b * maxp + t / page_size];
                const int64_t off = ((page * page_size + t % page_size) * Hkv + g) * d;
                for (int c = 0; c < d; ++c) {
                    kd[t * d + c] = (double)k_scale[g] * value(k_cache[off + c]);
                    vd[t * d + c] = (double)v_scale[g] * value(v_cache[off + c]);
                }
            }
            /* the definition, as in attention_row, on the dequantised rows */
            const float *qr = q + ((int64_t)b * Hq + h) * d;
            for (int64_t t = 0; t < len; ++t) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += (double)qr[c] * kd[t * d + c];
                s[t] = scale * acc;
            }
            double m = s[0];
            for (int64_t t = 1; t < len; ++t)
                if (s[t] > m) m = s[t];
            double l = 0.0;
            for (int64_t t = 0; t < len; ++t) {
                s[t] = exp(s[t] - m);
                l += s[t];
            }
            for (int c = 0; c < d; ++c) orow[c] = 0.0;
            for (int64_t t = 0; t < len; ++t) {
                const double pw = s[t] / l;
                for (int c = 0; c < d; ++c) orow[c] += pw * vd[t * d + c];
            }
            lse_rows[rr] = m + log(l);
        }
        free(s);
        free(kd);
        free(vd);
    }
    return 0;
}

/* The FP8 E4M3 cache: value(byte) = e4m3(byte) (oracle_e4m3_value above). */
int oracle_decode_paged_fp8_rows(const float *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                 const float *k_scale, const float *v_scale,
                                 const int32_t *page_table, const int32_t *seq_lens,
                                 int B, int Hq, int Hkv, int d, int page_size,
                                 int num_pages, int maxp, double scale,
                                 const int32_t *seqs, int nseq,
                                 double *o_rows, double *lse_rows, int nthreads)
{
    return decode_paged_bytes_rows(oracle_e4m3_value, q, k_cache, v_cache, k_scale, v_scale,
                                   page_table, seq_lens, B, Hq, Hkv, d, page_size, num_pages,
                                   maxp, scale, seqs, nseq, o_rows, lse_rows, nthreads);
}

/* The value of one INT8 byte: the byte read as a two's complement integer,
 * -128 .. 127. */
double oracle_int8_value(uint8_t x)
{
    return x < 128 ? (double)x : (double)x - 256.0;
}

/* The INT8 cache: value(byte) = int8(byte). */
int oracle_decode_paged_int8_rows(const float *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                  const float *k_scale, const float *v_scale,
                                  const int32_t *page_table, const int32_t *seq_lens,
                                  int B, int Hq, int Hkv, int d, int page_size,
                                  int num_pages, int maxp, double scale,
                                  const int32_t *seqs, int nseq,
                                  double *o_rows, double *lse_rows, int nthreads)
{
    return decode_paged_bytes_rows(oracle_int8_value, q, k_cache, v_cache, k_scale, v_scale,
                                   page_table, seq_lens, B, Hq, Hkv, d, page_size, num_pages,
                                   maxp, scale, seqs, nseq, o_rows, lse_rows, nthreads);
}

/*
 * The pages' online softmax statistics, in their order ("Donanıma Duyarlı
 * Algoritma Tasarımı: FlashAttention", section "Online Softmax Prensibi",
 * steps 1-5).  The row x[0..n) is consumed in blocks of `block` values.  For
 * each block the local maximum m_new and the local sum l_new of
 * exp(x - m_new) are formed; then
 *     M_new = max(M_old, m_new)
 *     L_old = L_old * exp(M_old - M_new)
 *     l_new = l_new * exp(m_new - M_new)
 *     L_new = L_old + l_new
 * The first block starts from M = -inf, L = 0.  On return *M is max_j x_j and
 * *L is sum_j exp(x_j - M).  This is not used to produce the oracle's
 * attention outputs; the tests use it to check that the recurrence reaches
 * the direct maximum and sum.
 */
void oracle_online_softmax_stats(const double *x, int64_t n, int64_t block,
                                 double *M, double *L)
{
    double Mg = -INFINITY, Lg = 0.0;
    if (block <= 0) block = n > 0 ? n : 1;
    for (int64_t start = 0; start < n; start += block) {
        const int64_t end = start + block < n ? start + block : n;
        double m_new = x[start];
        for (int64_t j = start + 1; j < end; ++j)
            if (x[j] > m_new) m_new = x[j];
        double l_new = 0.0;
        for (int64_t j = start; j < end; ++j) l_new += exp(x[j] - m_new);
        const double M_new = Mg > m_new ? Mg : m_new;
        const double L_old = (Lg == 0.0) ? 0.0 : Lg * exp(Mg - M_new);
        l_new = l_new * exp(m_new - M_new);
        Lg = L_old + l_new;
        Mg = M_new;
    }
    *M = Mg;
    *L = Lg;
}

/*
 * Combining the results of attention over disjoint key subsets, by the same
 * rescaling rule as the online softmax above: each part s carries its own
 * normalised output o_s (d values) and log-sum-exp lse_s over its keys.  The
 * combined log-sum-exp is ln sum_s exp(lse_s), and the combined output is
 * sum_s exp(lse_s - lse) * o_s.  Parts with lse_s = -inf (no keys) contribute
 * nothing.  Used by the tests to check that splitting the keys and combining
 * reproduces attention over all keys.
 */
void oracle_merge_parts(const double *o_parts, const double *lse_parts, int nparts,
                        int d, double *o, double *lse)
{
    double m = -INFINITY;
    for (int s = 0; s < nparts; ++s)
        if (lse_parts[s] > m) m = lse_parts[s];
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int s = 0; s < nparts; ++s) l += exp(lse_parts[s] - m);
    const double out_lse = m + log(l);
    for (int s = 0; s < nparts; ++s) {
        if (lse_parts[s] == -INFINITY) continue;
        const double w = exp(lse_parts[s] - out_lse);
        for (int c = 0; c < d; ++c) o[c] += w * o_parts[(int64_t)s * d + c];
    }
    *lse = out_lse;
}
