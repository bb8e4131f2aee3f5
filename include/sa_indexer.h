/*
 * sparse_attn for GB300 (sm_103a): the C ABI of the indexer's selection step.
 *
 * The conventions of sparse_attn.h apply (device pointers into caller-owned memory, `stream` a
 * cudaStream_t as void*, arguments checked before anything is enqueued, no allocation).
 */
#ifndef SA_INDEXER_H
#define SA_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#include "sparse_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SA_SCORE_F32 = 0,   /* score is f32 */
    SA_SCORE_BF16 = 1   /* score is bf16 (IEEE bfloat16 bit patterns) */
} sa_score_format;

/* Most compressed positions one call can select from (a row's keys are held in shared memory). */
#define SA_INDEXER_MAX_POSITIONS 49152

/*
 * The indexer's selection of the compressed idx.
 *
 * Source: "DeepSeek V4.1" attention page, Indexer.forward (the steps after the index scores are
 * formed: the visibility mask of a prefill, topk, the sort into position order, and the
 * unreachable -> -1 / offset rule).
 *
 * For every sequence bi < b and query si < s, over the n_comp compressed positions of its score
 * row (n_comp must equal (start_pos + s) / ratio, the positions the page's index_k holds):
 *   visible = (si + 1) / ratio at a prefill (start_pos == 0): position t >= visible scores -inf;
 *             n_comp at a decode step (no mask)
 *   k       = min(index_topk, n_comp)
 *   the k highest-scoring positions, sorted ascending; each written as t + offset when
 *   t < visible, else -1 (so a query that sees fewer than k positions gets a -1 tail).
 * Equal scores are picked lowest position first (the page's topk leaves their order open);
 * -0 and +0 are equal.  NaN scores are not supported.
 *
 * Arguments
 *   score         [b][s][n_comp], f32 or bf16 (score_format), dense
 *   idx           int32, row (bi, si) at idx + bi * batch_stride + si * ld, k entries written;
 *                 ld >= k, so the k columns can sit after the window columns of a wider idx
 *                 tensor; batch_stride >= (s - 1) * ld + k when b > 1; must not overlap score
 *   offset        added to every visible pick (the page's offset: the rows before the
 *                 compressed ones in kv); 0 <= offset and offset + n_comp <= 2^31 - 1
 * Returns SA_ERR_UNSUPPORTED for a chunked prefill (start_pos > 0 and s > 1, which the page
 * does not describe) and for n_comp > SA_INDEXER_MAX_POSITIONS; SA_ERR_INVALID_ARG for a bad
 * argument.  b * s == 0 or k == 0 is a no-op.  The caller computes k to size idx.
 */
sa_status sa_indexer_topk(const void* score, int score_format, int64_t b, int64_t s,
                          int64_t n_comp, int64_t start_pos, int ratio, int index_topk,
                          int32_t offset, int32_t* idx, int64_t ld, int64_t batch_stride,
                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SA_INDEXER_H */
