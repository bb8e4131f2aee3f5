/*
 * sparse_attn for GB300 (sm_103a): the C ABI.
 *
 * DeepSeek V4.1's index-gathered latent attention with an attention sink, plus the two input
 * helpers on the same path (the window index table and the fp8 block quantiser).  Every entry
 * point takes plain pointers and sizes; no framework types cross this boundary.
 *
 * Conventions for every call
 *   - Tensor pointers are DEVICE pointers into caller-owned memory, row-major, densely packed
 *     unless a stride argument says otherwise, 16-byte aligned.  The library allocates no device
 *     memory and keeps no state between calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Work is
 *     enqueued on it and the call returns without synchronising, except where noted.
 *   - Arguments are checked before anything is enqueued: a bad argument returns an error and
 *     launches nothing.  Kernels never trap; data errors they detect are recorded in the
 *     workspace status word (see sa_read_status).
 *   - bf16 tensors hold IEEE bfloat16 bit patterns (uint16); e4m3 is the OCP "fn" fp8 variant
 *     (no infinities, largest finite 448); e8m0 is an unsigned power-of-two exponent, 2^(e-127).
 */
#ifndef SPARSE_ATTN_H
#define SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SA_OK = 0,
    SA_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size, misalignment */
    SA_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement (see each call) */
    SA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    SA_ERR_INDEX = 4,        /* a kernel saw an index outside [-1, rows) (sa_read_status) */
    SA_ERR_WORKSPACE = 5,    /* workspace missing or smaller than the size query returned */
    SA_ERR_TIMEOUT = 6       /* a kernel's bounded wait gave up (sa_read_status); its output is
                                not valid */
} sa_status;

typedef enum {
    SA_KV_BF16 = 0,          /* kv is bf16 [b][rows][d] */
    SA_KV_FP8_E4M3 = 1       /* kv is e4m3 [b][rows][d] + kv_scale e8m0 [b][rows][d/32] */
} sa_kv_format;

/* Which kernel family computes sparse_attn (sa_sparse_attn_family). */
typedef enum {
    SA_FAMILY_AUTO = 0,      /* what sa_sparse_attn uses: tcgen05 for head_dim 512, else mma.sync */
    SA_FAMILY_TCGEN05 = 1,   /* the tcgen05 / TMEM kernels; head_dim 512 only */
    SA_FAMILY_MMA_SYNC = 2   /* the warp-level mma.sync kernels; every supported head_dim */
} sa_kernel_family;

/* Status word block at the start of every workspace, in bytes. */
#define SA_STATUS_BYTES 256

/*
 * sparse_attn.
 *
 * Source: "Module attn" API page (spark_model, deepseek_v41_ref/attn), Functions: sparse_attn
 * and the precision paragraph; "DeepSeek V4.1" attention page, Attention.forward (the call
 * sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale), one kv tensor serving as keys and
 * values) and Attention.__init__ (attn_sink: one f32 per local head; softmax_scale =
 * head_dim ** -0.5).
 *
 * For every sequence bi < b, query token si < s and head hh < h:
 *   J    = the entries of idx[bi][si][0..topk) that are not -1 (repeats count repeatedly)
 *   l_j  = softmax_scale * sum_k q[bi][si][hh][k] * kv[bi][j][k]        (f32 accumulate)
 *   o    = sum_j e^(l_j) kv[bi][j][:] / (e^(sink[hh]) + sum_j e^(l_j))   (sink: denominator only)
 *   o[bi][si][hh][:] = bf16 round-to-nearest-even of o;  o = 0 when J is empty.
 *
 * Arguments
 *   q          bf16 [b][s][h][d]
 *   kv         bf16 [b][rows][d] (SA_KV_BF16) or e4m3 [b][rows][d] (SA_KV_FP8_E4M3)
 *   kv_scale   e8m0 [b][rows][d/32] for SA_KV_FP8_E4M3 (block 32 along d), NULL for bf16.
 *              An fp8 row j decodes to e4m3(kv[j][k]) * 2^(kv_scale[j][k/32] - 127), exactly
 *              the bf16 values the act_quant round trip produces.
 *   sink       f32 [h] (may be -inf)
 *   idx        int32 [b][s][topk], each entry in [-1, rows).  An entry outside that range is
 *              treated as -1 and sets SA_ERR_INDEX in the workspace status word.
 *   softmax_scale  f32 multiplier of the dot products
 *   o          bf16 [b][s][h][d], written; must not overlap any input
 *   workspace  device scratch of at least sa_sparse_attn_workspace_size(...) bytes, aligned to
 *              256 bytes; its first SA_STATUS_BYTES hold the status word, which the caller zeroes
 *              once (e.g. cudaMemsetAsync) and which the library only ever ORs into.  The rest is
 *              overwritten by every call; calls sharing one workspace must be stream-ordered.
 * Supported: d a multiple of 64 in [64, 512]; 1 <= h <= 128; b, s, rows >= 0; topk >= 0;
 *   b*s*h < 2^31; rows * d < 2^31 * 16.  Otherwise SA_ERR_UNSUPPORTED.  b*s == 0 is a no-op.
 */
sa_status sa_sparse_attn(const void* q, const void* kv, const uint8_t* kv_scale, int kv_format,
                         const float* sink, const int32_t* idx, float softmax_scale,
                         int64_t b, int64_t s, int h, int d, int64_t rows, int topk,
                         void* o, void* workspace, size_t workspace_bytes, void* stream);

/*
 * sa_sparse_attn computed by a chosen kernel family (sa_kernel_family), e.g. to compare the two
 * families on the same inputs.  Same source, arguments, result and workspace size as
 * sa_sparse_attn; SA_FAMILY_AUTO is exactly sa_sparse_attn.  SA_FAMILY_TCGEN05 with a head_dim
 * other than 512 returns SA_ERR_UNSUPPORTED; any other family value SA_ERR_INVALID_ARG.
 */
sa_status sa_sparse_attn_family(const void* q, const void* kv, const uint8_t* kv_scale,
                                int kv_format, const float* sink, const int32_t* idx,
                                float softmax_scale, int64_t b, int64_t s, int h, int d,
                                int64_t rows, int topk, void* o, void* workspace,
                                size_t workspace_bytes, int family, void* stream);

/*
 * sparse_attn with the inverse rotary embedding of the output fused in.
 *
 * Source: "DeepSeek V4.1" attention page, Attention.forward (after sparse_attn, the last
 * rope_dim dims of o are rotated back with apply_rotary_emb(..., inverse=True)) and
 * apply_rotary_emb (pairs of dims as complex numbers, times the position's rotation or its
 * conjugate); Attention.__init__ (rope_head_dim = 64 of head_dim 512).
 *
 * Computes what sa_sparse_attn computes, then, for every sequence bi, token si and head hh,
 * with p = start_pos + si and k < rope_dim / 2, the pair (a, b) = o[.., d - rope_dim + 2k],
 * o[.., d - rope_dim + 2k + 1] becomes
 *   (a c + b s,  b c - a s),   (c, s) = rot[p][k][0], rot[p][k][1]
 * (a + i b times c - i s).  The rotation is applied to the f32 result before its one rounding
 * to bf16; the two-step form (o rounded to bf16, rotated, rounded again) differs from it by at
 * most about one bf16 unit of o.
 *
 * Arguments as sa_sparse_attn (same workspace size), plus
 *   rot        f32 [npos][rope_dim / 2][2] (cos, sin) per position, 8-byte aligned; must not
 *              overlap o
 *   npos       positions in rot; start_pos + s <= npos
 *   rope_dim   even, 2 <= rope_dim <= d
 *   start_pos  position of token 0 of every sequence (the prefill's 0, a decode step's length)
 * Supported: d = 512 (the tcgen05 kernel family, which fuses the rotation into its epilogue);
 * other head dims return SA_ERR_UNSUPPORTED.
 */
sa_status sa_sparse_attn_rope(const void* q, const void* kv, const uint8_t* kv_scale,
                              int kv_format, const float* sink, const int32_t* idx,
                              float softmax_scale, int64_t b, int64_t s, int h, int d,
                              int64_t rows, int topk, void* o, void* workspace,
                              size_t workspace_bytes, const float* rot, int64_t npos, int rope_dim,
                              int64_t start_pos, void* stream);

/* Workspace bytes sa_sparse_attn needs for this shape (always >= SA_STATUS_BYTES), enough for
 * either kernel family and any GPU: a pure function of the arguments.  Returns 0 for an
 * unsupported shape. */
size_t sa_sparse_attn_workspace_size(int64_t b, int64_t s, int h, int d, int64_t rows, int topk,
                                     int kv_format);

/* Size of the library's own scratch array used by sa_sparse_attn_static_scratch (64 MiB). */
#define SA_STATIC_SCRATCH_BYTES (64u << 20)

/*
 * sparse_attn without a caller workspace.  The source pages have no counterpart to this call: it
 * exists for callers that cannot allocate device memory -- a plugin inside a host runtime that
 * owns every device allocation and gives the plugin none, or a serving loop that must not call
 * cudaMalloc / cudaFree (which can synchronise the device) on its request path.
 *
 * Computes exactly what sa_sparse_attn computes, with the same arguments apart from the
 * workspace, which is replaced by a SA_STATIC_SCRATCH_BYTES array that the library keeps in
 * device memory on every GPU that loads it, until the process exits.  Allocates nothing.
 *   status_out  optional device uint32: receives the call's status word (bit 0 set when an index
 *               outside [-1, rows) was seen, bit 1 when a kernel wait gave up, in which case o is
 *               not valid); NULL to skip.  The word is cleared at the start of every call; a call
 *               with b * s == 0 writes 0 to it.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current) and caches it: make that first call before any stream capture.  Every call
 * shares the one array, which keeps the last call's contents; calls whose work overlaps on the
 * GPU (unordered streams) race on it and must be serialised by the caller.
 * Returns SA_ERR_WORKSPACE when the kernel family the call runs in (as sa_sparse_attn routes it)
 * needs more scratch than SA_STATIC_SCRATCH_BYTES for this shape, otherwise as sa_sparse_attn.
 */
sa_status sa_sparse_attn_static_scratch(const void* q, const void* kv, const uint8_t* kv_scale,
                                        int kv_format, const float* sink, const int32_t* idx,
                                        float softmax_scale, int64_t b, int64_t s, int h, int d,
                                        int64_t rows, int topk, void* o, uint32_t* status_out,
                                        void* stream);

/*
 * Window index table (get_window_topk_idxs).
 *
 * Source: "Module attn" API page, Functions: window_topk_idxs and the ring-cache paragraph
 * (prefill of 12 tokens into 8 slots; decode reads the whole ring oldest first).
 *
 * Writes, for each of `nbatch` sequences, a [seqlen][window] block of int32 slot indices at
 * idx + bi * batch_stride, row r at + r * ld (ld >= window), so the table can be the leading
 * columns of a wider idx tensor:
 *   prefill (start_pos == 0): row i, column j -> i - window + 1 + j, or -1 when negative;
 *   decode  (seqlen == 1, start_pos = p > 0): column j -> (p - window + 1 + j) mod window, or
 *           -1 when p - window + 1 + j < 0 (the ring read oldest first).
 * start_pos > 0 with seqlen > 1 (chunked prefill) is not described by the source and returns
 * SA_ERR_UNSUPPORTED.  Requires window >= 1, ld >= window, batch_stride >= seqlen * ld.
 */
sa_status sa_window_idxs(int64_t start_pos, int64_t seqlen, int window, int32_t* idx, int64_t ld,
                         int64_t nbatch, int64_t batch_stride, void* stream);

/*
 * act_quant: fp8 e4m3 block quantisation with power-of-two (ue8m0) scales.
 *
 * Source: "Module attn" API page, Functions: act_quant_inplace and pow2_ceil; Constants:
 * FP8_BLOCK (32); the precision paragraph (the round trip is exact).
 *
 * For each of n rows (row i of x at x + i * x_stride elements) and each block of 32 consecutive
 * elements along d:
 *   amax = max |x_k|, floored at 1e-4;  s = pow2_ceil(amax / 448) (f32 division, round to
 *   nearest);  c_k = e4m3 of x_k / s (round to nearest even, saturating at +-448);
 * and writes any of:
 *   x_rt   bf16, the round trip c_k * s (row i at x_rt + i * rt_stride); may equal x (in place)
 *   codes  e4m3 bytes c_k (row i at codes + i * codes_stride)
 *   scales e8m0 bytes log2(s) + 127 (row i at scales + i * scales_stride)
 * Outputs passed as NULL are skipped (at least one must be given).  Requires d % 32 == 0,
 * d >= 32, strides >= the row's length in elements.
 */
sa_status sa_act_quant_fp8(const void* x, int64_t n, int d, int64_t x_stride,
                           void* x_rt, int64_t rt_stride,
                           uint8_t* codes, int64_t codes_stride,
                           uint8_t* scales, int64_t scales_stride, void* stream);

/*
 * Ring write: the window cache's write side, with act_quant fused.
 *
 * Source: "Module attn" API page, the ring-cache paragraph (the kv row of the token at position t
 * is kept in slot t mod window; a later token overwrites an earlier one in the same slot) and
 * act_quant_inplace (the kv row is quantised before it is stored).
 *
 * For each of `nbatch` sequences, the kv rows of `seqlen` new tokens at positions
 * start_pos .. start_pos + seqlen - 1 go to ring slot (position mod window) of that sequence,
 * quantised exactly as sa_act_quant_fp8 quantises a row.  When seqlen > window only the last
 * `window` tokens are written (each earlier token's slot is taken by a later one), so the ring ends
 * as if every token had been written in order.
 *   x            the new rows, bf16: row t of sequence bi at x + (bi * seqlen + t) * x_stride
 *                elements (x_stride >= d)
 *   ring_rt      bf16 round trip c * s: row `slot` of sequence bi at
 *                ring_rt + bi * rt_batch_stride + slot * rt_stride elements, or NULL
 *   ring_codes   e4m3 bytes, addressed the same way with codes_stride / codes_batch_stride, or NULL
 *   ring_scales  e8m0 bytes (d / 32 per row), scales_stride / scales_batch_stride, or NULL
 * At least one output; the ring rows of one sequence must not overlap those of another, and no
 * output may overlap x.  Requires d % 32 == 0, d >= 32, window >= 1, and non-negative nbatch,
 * seqlen and start_pos.  Returns SA_ERR_INVALID_ARG (nothing enqueued) for a bad argument and
 * SA_ERR_CUDA for a launch error; the caller owns every buffer.
 */
sa_status sa_window_write(const void* x, int64_t nbatch, int64_t seqlen, int d, int64_t x_stride,
                          int64_t start_pos, int window,
                          void* ring_rt, int64_t rt_stride, int64_t rt_batch_stride,
                          uint8_t* ring_codes, int64_t codes_stride, int64_t codes_batch_stride,
                          uint8_t* ring_scales, int64_t scales_stride, int64_t scales_batch_stride,
                          void* stream);

/*
 * Reads the status word in a workspace (synchronises `stream` first) and returns SA_OK or the
 * error recorded there: SA_ERR_TIMEOUT (a kernel wait gave up) before SA_ERR_INDEX (an index
 * outside [-1, rows) was seen).  With clear != 0 the word is reset to zero.
 */
sa_status sa_read_status(void* workspace, int clear, void* stream);

/* A static, human-readable name for a status code. */
const char* sa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int sa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H */
