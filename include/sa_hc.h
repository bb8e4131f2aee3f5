/*
 * sparse_attn for GB300 (sm_103a): the C ABI of the Hyper-Connections split (hc_split_sinkhorn).
 *
 * The conventions of sparse_attn.h apply (device pointers into caller-owned memory, `stream` a
 * cudaStream_t as void*, arguments checked before anything is enqueued, no allocation).
 */
#ifndef SA_HC_H
#define SA_HC_H

#include <stddef.h>
#include <stdint.h>

#include "sparse_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * hc_split_sinkhorn.
 *
 * Source: "DeepSeek V4.1" attention-write page (decode), hc_split_sinkhorn and its kernel (the block's mixes
 * split into pre / post weights and a Sinkhorn-normalised comb matrix); the model config on the
 * "DeepSeek V4.1" first-layer attention update page (hc_mult 4, hc_sinkhorn_iters 20, hc_eps 1e-6).
 *
 * For every token i < n, with a_j = mixes[i][j] * hc_scale[.] + hc_base[j] in f32:
 *   pre[i][j]  = sigmoid(a_j) + eps              (hc_scale[0], j < hc)
 *   post[i][j] = 2 sigmoid(a_{hc + j})           (hc_scale[1])
 *   comb[i]    = the hc x hc matrix a_{2 hc + j hc + k} (row j, column k; hc_scale[2]): each row
 *                replaced by its softmax plus eps, each column divided by (its sum + eps), then
 *                sinkhorn_iters - 1 rounds of dividing each row, then each column, by its sum + eps.
 * Everything in f32, as on the page (expf, IEEE reciprocals; a normalisation multiplies by the
 * reciprocal of its sum where the page divides, one rounding apart).
 *
 * Arguments
 *   mixes      f32 [n][(2 + hc) * hc], 16-byte aligned
 *   hc_scale   f32 [3];  hc_base f32 [(2 + hc) * hc]
 *   pre, post  f32 [n][hc], written;  comb f32 [n][hc][hc], written; no output may overlap an
 *              input or another output
 * Supported: hc = 4 (the model's hc_mult), sinkhorn_iters >= 1, n <= (2^31 - 1) * 256.  Otherwise
 * SA_ERR_UNSUPPORTED (hc) or SA_ERR_INVALID_ARG.  n == 0 is a no-op.
 */
sa_status sa_hc_split_sinkhorn(const float* mixes, int64_t n, int hc, const float* hc_scale,
                               const float* hc_base, int sinkhorn_iters, float eps, float* pre,
                               float* post, float* comb, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SA_HC_H */
