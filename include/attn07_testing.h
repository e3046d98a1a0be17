/*
 * attn07_testing.h -- test hooks exported by libattn07.so.  They are not part of
 * the library's interface (include/attn07.h): they exist so that the tests can
 * drive a kernel into configurations its normal launch does not choose.
 */
#ifndef ATTN07_TESTING_H
#define ATTN07_TESTING_H

#include "attn07.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_decode_paged with the split kernel run on `ctas` CTAs (1 <= ctas <= twice
 * the GPU's SM count) instead of the library's choice.  The pages of all
 * sequences are cut into `ctas` equal contiguous ranges, each attended on its
 * own, and each sequence's pieces are merged by their log-sum-exps (the
 * rescaling rule of the fatihsoysal.com page, section "Online Softmax
 * Prensibi", applied to whole key ranges), so the result must match
 * attn_decode_paged's up to rounding whatever the count.  Arguments, layouts,
 * workspace and errors as attn_decode_paged; ctas <= 0 returns
 * ATTN_ERR_INVALID_ARG, more than twice the SM count ATTN_ERR_UNSUPPORTED.
 */
attn_status_t attn_testing_decode_paged_ctas(const void *q, const void *k_cache,
                                             const void *v_cache, const int32_t *page_table,
                                             const int32_t *seq_lens, void *o, float *lse, int B,
                                             int Hq, int Hkv, int d, int page_size, int num_pages,
                                             int max_pages_per_seq, float scale, void *workspace,
                                             size_t workspace_bytes, int ctas,
                                             attn_stream_t stream);

/*
 * attn_fwd_f32 with a fixed tile height: `rows` = 16 (16 query rows per CTA,
 * 16 threads per row), 4 (4 rows per CTA, 64 threads per row) or 2 (2 rows per
 * CTA, 128 threads per row) instead of the library's choice by launch size.  Both compute the same attention formula
 * (the fatihsoysal.com page, section "Transformer Mimarisi ve Self-Attention
 * Mekanizması") with the online softmax of section "Online Softmax Prensibi",
 * in fp32; their results differ only by the order of fp32 additions.
 * Arguments, layouts and errors as attn_fwd_f32; any other `rows` returns
 * ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_testing_fwd_f32_rows(const float *q, const float *k, const float *v, float *o,
                                        float *lse, int B, int Hq, int Hkv, int N, int d,
                                        int causal, float scale, int rows,
                                        attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN07_TESTING_H */
