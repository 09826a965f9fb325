/*
 * mla_indexer.h — C ABI of the sparse-attention indexer (libmla_decode.so):
 * token scores over a request's cached index keys, then the top-k lists the
 * sparse decode (mla_decode with topk_idx) consumes.
 *
 * The operation ("The 31-Millisecond Smoking Gun", the DeepSeek-V4-Flash
 * architecture paragraph and "Potential mistake: Overlooking the indexer":
 * sparse token selection scores every cached token each decode step, a
 * [requests, positions, 64] tensor, and attention runs over the selected
 * ones).  The pages give the shape, not the formula; the reading used here
 * is the published DSA indexer form, 64 index heads of 128 dims:
 *
 *     I[b, t, j] = sum_h w[b, t, h] * ReLU(q_I[b, t, h, :] . k_I[row(b, j), :])
 *
 * for the visible positions j of query token t (j < len_b; with
 * MLA_FLAG_CAUSAL, j <= len_b - s_q + t), with index keys cached per token in
 * 64-token pages reached through the same block table as the latent cache
 * (row(b, j) = block_table[b * bt_stride + j / 64] * 64 + j % 64).  Top-k: the
 * k visible positions with the largest score, ties to the smaller position,
 * listed in increasing position order and padded with -1.
 *
 * Conventions: as for mla_decode.h (device pointers, asynchronous on
 * `stream`, no allocation, no host synchronisation, graph-capturable).
 * `status` is a device int the kernels set (from 0, atomically) to
 * MLA_ERR_TIMEOUT if a bounded wait runs out or MLA_ERR_BAD_TABLE if a
 * length exceeds `max_len`; never cleared by the calls.  mla_workspace_status
 * reads it.
 */
#ifndef MLA_INDEXER_H_
#define MLA_INDEXER_H_

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

enum { MLA_IDX_HEADS = 64, MLA_IDX_DIM = 128 };

/* Scores of every visible position.
 *   q_idx        bf16 [batch, s_q, 64, 128], contiguous, 16-B aligned
 *   w_idx        fp32 [batch, s_q, 64], contiguous
 *   k_idx_cache  bf16 [num_pages, 64, 128] index keys, contiguous, 16-B aligned
 *   block_table, bt_stride, cache_lens, batch, s_q: as for mla_decode
 *                (s_q 1 .. MLA_MAX_SQ)
 *   flags        0 or MLA_FLAG_CAUSAL
 *   max_len      an upper bound of every cache_lens[b] (<= 64 * bt_stride);
 *                a longer length is clamped to it and flagged in *status
 *   scores       fp32; the row of (b, t) at scores + (b * s_q + t) *
 *                scores_stride; entries 0 .. visible - 1 are written, the
 *                rest of the row is left untouched
 *   scores_stride  >= max_len, multiple of 4
 */
int mla_indexer_scores(const void* q_idx, const float* w_idx, const void* k_idx_cache, int64_t num_pages,
                       const int32_t* block_table, int64_t bt_stride, const int32_t* cache_lens, int batch,
                       int s_q, unsigned flags, int max_len, float* scores, int64_t scores_stride, int* status,
                       mla_stream_t stream);

/* Top-k of each (b, t) score row over its visible positions.
 *   scores, scores_stride, cache_lens, batch, s_q, flags, max_len: as above
 *   topk         1 .. 65536
 *   max_len      at most 2,064,384 (MLA_ERR_UNSUPPORTED beyond)
 *   out_idx      int32 [batch, s_q, topk]: increasing positions, then -1
 */
int mla_topk(const float* scores, int64_t scores_stride, const int32_t* cache_lens, int batch, int s_q,
             unsigned flags, int max_len, int topk, int32_t* out_idx, int* status, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_INDEXER_H_ */
