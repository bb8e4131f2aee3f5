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
 * Source: "DeepSeek V4.1" source-layer attention page (indexer view), Indexer.forward (the steps after the index scores are
 * formed: the visibility mask of a prefill, the level-two candidate mask of a layer that uses
 * another layer's candidate blocks, topk, the sort into position order, and the
 * unreachable -> -1 / offset rule).
 *
 * For every sequence bi < b and query si < s, over the n_comp compressed positions of its score
 * row (n_comp must equal (start_pos + s) / ratio, the positions the page's index_k holds):
 *   visible = (si + 1) / ratio at a prefill (start_pos == 0): position t >= visible scores -inf;
 *             n_comp at a decode step (no mask)
 *   candidates (optional): a position whose candidates byte is 0 scores -inf too
 *   k       = min(index_topk, n_comp)
 *   the k highest-scoring positions, sorted ascending; each written as t + offset when
 *   t < visible, else -1 (so a query that sees fewer than k positions gets a -1 tail).
 * Equal scores are picked lowest position first (the page's topk leaves their order open);
 * -0 and +0 are equal.  NaN scores are not supported.
 *
 * Arguments
 *   score         [b][s][n_comp], f32 or bf16 (score_format), dense
 *   candidates    NULL, or uint8 [b][s][n_comp] (nonzero = inside a candidate block, e.g. the
 *                 mask sa_candidate_blocks writes)
 *   idx           int32, row (bi, si) at idx + bi * batch_stride + si * ld, k entries written;
 *                 ld >= k, so the k columns can sit after the window columns of a wider idx
 *                 tensor; batch_stride >= (s - 1) * ld + k when b > 1; must not overlap score
 *   offset        added to every visible pick (the page's offset: the rows before the
 *                 compressed ones in kv); 0 <= offset and offset + n_comp <= 2^31 - 1
 * Returns SA_ERR_UNSUPPORTED for a chunked prefill (start_pos > 0 and s > 1, which the page
 * does not describe) and for n_comp > SA_INDEXER_MAX_POSITIONS; SA_ERR_INVALID_ARG for a bad
 * argument.  b * s == 0 or k == 0 is a no-op.  The caller computes k to size idx.
 */
sa_status sa_indexer_topk(const void* score, int score_format, const uint8_t* candidates,
                          int64_t b, int64_t s, int64_t n_comp, int64_t start_pos, int ratio,
                          int index_topk, int32_t offset, int32_t* idx, int64_t ld,
                          int64_t batch_stride, void* stream);

/*
 * Level one of the two-level top-k: the candidate blocks.
 *
 * Source: "DeepSeek V4.1" source-layer attention page (indexer view), select_candidate_blocks (and Indexer.forward, which
 * calls it on the masked index scores of the candidate-source layer with its compress_lens).
 *
 * For every sequence bi and query si, with visible as for sa_indexer_topk (positions at or past
 * it count as -inf, as the page's caller has masked them) and nb = ceil(n_comp / block_size):
 *   block j's score = the highest logit among positions j * block_size .. + block_size - 1
 *                     (-inf when none is visible, and past the row's end)
 *   the block holding position visible - 1 scores +inf (none when visible == 0)
 *   the min(topk_blocks, nb) highest-scoring blocks are picked, equal scores lowest block first;
 *   a pick that scores -inf is dropped
 *   mask[bi][si][t] = 1 when t's block was kept, else 0.
 *
 * Arguments
 *   logits        [b][s][n_comp], f32 or bf16 (score_format), dense; n_comp = (start_pos + s) /
 *                 ratio as for sa_indexer_topk
 *   mask          uint8 [b][s][n_comp], written; must not overlap logits
 * Returns SA_ERR_UNSUPPORTED for a chunked prefill and for more than SA_INDEXER_MAX_POSITIONS
 * blocks; SA_ERR_INVALID_ARG for a bad argument (block_size < 1, topk_blocks < 0, ...).
 * b * s == 0 is a no-op; topk_blocks == 0 zeroes the mask.  NaN logits are not supported.
 */
sa_status sa_candidate_blocks(const void* logits, int score_format, int64_t b, int64_t s,
                              int64_t n_comp, int64_t start_pos, int ratio, int topk_blocks,
                              int block_size, uint8_t* mask, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SA_INDEXER_H */
