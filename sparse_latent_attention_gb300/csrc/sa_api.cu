// The C ABI declared in include/sparse_attn.h: argument checks, workspace layout and dispatch.
// Nothing here allocates device memory; every kernel is enqueued on the caller's stream.

#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_internal.cuh"
#include "sparse_attn.h"

namespace {

constexpr int kVersion = 200;  // 0.2.0: tcgen05 family for head_dim 512 (bf16 and fp8 kv)

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

bool supported_shape(int64_t b, int64_t s, int h, int d, int64_t rows, int topk) {
    if (b < 0 || s < 0 || rows < 0 || topk < 0) return false;
    if (h < 1 || h > 128) return false;
    if (d < 64 || d > 512 || d % 64 != 0) return false;
    if (b * s * (int64_t)h >= (int64_t(1) << 31)) return false;
    if (rows >= (int64_t(1) << 31)) return false;
    return true;
}

sa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SA_OK : SA_ERR_CUDA; }

// The whole sparse_attn call; rope == nullptr for none (checked by the caller).
sa_status attn_call(const void* q, const void* kv, const uint8_t* kv_scale, int kv_format,
                    const float* sink, const int32_t* idx, float softmax_scale, int64_t b, int64_t s,
                    int h, int d, int64_t rows, int topk, void* o, void* workspace,
                    size_t workspace_bytes, const float* rope, int rope_dim, int64_t rope_pos0,
                    int family, void* stream);

}  // namespace

namespace sa {

// The family a call runs in (SA_FAMILY_AUTO resolved), or -1 when the requested one cannot run
// this shape.
int routed_family(int family, int h, int d, int kv_format, int64_t b, int64_t rows) {
    const bool tc = attn_tc_supports(h, d, kv_format, b, rows);
    if (family == SA_FAMILY_AUTO) return tc ? SA_FAMILY_TCGEN05 : SA_FAMILY_MMA_SYNC;
    if (family == SA_FAMILY_TCGEN05) return tc ? SA_FAMILY_TCGEN05 : -1;
    if (family == SA_FAMILY_MMA_SYNC) return SA_FAMILY_MMA_SYNC;
    return -1;
}

size_t routed_workspace_bytes(int family, int64_t b, int64_t s, int h, int d, int64_t rows,
                              int topk) {
    const size_t scratch = family == SA_FAMILY_TCGEN05 ? attn_tc_scratch_bytes(b, s, h, topk)
                                                       : attn_mma_scratch_bytes(b, s, h, d, topk);
    return SA_STATUS_BYTES + align_up(scratch, 256);
}

}  // namespace sa

extern "C" {

size_t sa_sparse_attn_workspace_size(int64_t b, int64_t s, int h, int d, int64_t rows, int topk,
                                     int kv_format) {
    if (kv_format != SA_KV_BF16 && kv_format != SA_KV_FP8_E4M3) return 0;
    if (!supported_shape(b, s, h, d, rows, topk)) return 0;
    // enough for either kernel family, whichever a call is routed to
    size_t scratch = sa::attn_mma_scratch_bytes(b, s, h, d, topk);
    if (sa::attn_tc_supports(h, d, kv_format, b, rows)) {
        const size_t tc_scratch = sa::attn_tc_scratch_bytes(b, s, h, topk);
        if (tc_scratch > scratch) scratch = tc_scratch;
    }
    return SA_STATUS_BYTES + sa::align_up(scratch, 256);
}

sa_status sa_sparse_attn(const void* q, const void* kv, const uint8_t* kv_scale, int kv_format,
                         const float* sink, const int32_t* idx, float softmax_scale,
                         int64_t b, int64_t s, int h, int d, int64_t rows, int topk,
                         void* o, void* workspace, size_t workspace_bytes, void* stream) {
    return attn_call(q, kv, kv_scale, kv_format, sink, idx, softmax_scale, b, s, h, d, rows, topk,
                     o, workspace, workspace_bytes, nullptr, 0, 0, SA_FAMILY_AUTO, stream);
}

sa_status sa_sparse_attn_family(const void* q, const void* kv, const uint8_t* kv_scale,
                                int kv_format, const float* sink, const int32_t* idx,
                                float softmax_scale, int64_t b, int64_t s, int h, int d,
                                int64_t rows, int topk, void* o, void* workspace,
                                size_t workspace_bytes, int family, void* stream) {
    if (family != SA_FAMILY_AUTO && family != SA_FAMILY_TCGEN05 && family != SA_FAMILY_MMA_SYNC)
        return SA_ERR_INVALID_ARG;
    return attn_call(q, kv, kv_scale, kv_format, sink, idx, softmax_scale, b, s, h, d, rows, topk,
                     o, workspace, workspace_bytes, nullptr, 0, 0, family, stream);
}

sa_status sa_sparse_attn_rope(const void* q, const void* kv, const uint8_t* kv_scale,
                              int kv_format, const float* sink, const int32_t* idx,
                              float softmax_scale, int64_t b, int64_t s, int h, int d,
                              int64_t rows, int topk, void* o, void* workspace,
                              size_t workspace_bytes, const float* rot, int64_t npos, int rope_dim,
                              int64_t start_pos, void* stream) {
    if (rope_dim < 2 || rope_dim % 2 != 0 || rope_dim > d || npos < 0 || start_pos < 0)
        return SA_ERR_INVALID_ARG;
    if (start_pos > npos - s) return SA_ERR_INVALID_ARG;  // positions start_pos .. start_pos + s - 1
    if (kv_format != SA_KV_BF16 && kv_format != SA_KV_FP8_E4M3) return SA_ERR_INVALID_ARG;
    // the rotation is fused into the tcgen05 kernel's epilogue only
    if (!sa::attn_tc_supports(h, d, kv_format, b, rows)) return SA_ERR_UNSUPPORTED;
    if (b * s > 0 && (!rot || !aligned(rot, 8))) return SA_ERR_INVALID_ARG;
    if (b * s > 0 && overlaps(o, (size_t)(b * s) * h * (size_t)d * 2, rot,
                              (size_t)npos * rope_dim * sizeof(float)))
        return SA_ERR_INVALID_ARG;
    return attn_call(q, kv, kv_scale, kv_format, sink, idx, softmax_scale, b, s, h, d, rows, topk,
                     o, workspace, workspace_bytes, rot, rope_dim, start_pos, SA_FAMILY_TCGEN05,
                     stream);
}

}  // extern "C"

namespace {

sa_status attn_call(const void* q, const void* kv, const uint8_t* kv_scale, int kv_format,
                    const float* sink, const int32_t* idx, float softmax_scale, int64_t b, int64_t s,
                    int h, int d, int64_t rows, int topk, void* o, void* workspace,
                    size_t workspace_bytes, const float* rope, int rope_dim, int64_t rope_pos0,
                    int family, void* stream) {
    if (kv_format != SA_KV_BF16 && kv_format != SA_KV_FP8_E4M3) return SA_ERR_INVALID_ARG;
    if (b < 0 || s < 0 || h < 1 || d < 1 || rows < 0 || topk < 0) return SA_ERR_INVALID_ARG;
    if (!supported_shape(b, s, h, d, rows, topk)) return SA_ERR_UNSUPPORTED;
    const int fam = sa::routed_family(family, h, d, kv_format, b, rows);
    if (fam < 0) return SA_ERR_UNSUPPORTED;
    if (kv_format == SA_KV_BF16 && kv_scale) return SA_ERR_INVALID_ARG;
    if (b * s == 0) return SA_OK;  // nothing to compute; pointers of empty tensors may be NULL
    // kv (and kv_scale) may be NULL only when there are no rows, idx only when topk == 0
    if (!q || !sink || !o || (rows > 0 && !kv) || (topk > 0 && !idx)) return SA_ERR_INVALID_ARG;
    if (kv_format == SA_KV_FP8_E4M3 && rows > 0 && !kv_scale) return SA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(o, 16) || !aligned(sink, 4) ||
        !aligned(idx, 4))
        return SA_ERR_INVALID_ARG;
    const size_t n_tok = (size_t)(b * s);
    const size_t o_bytes = n_tok * h * (size_t)d * 2;
    const size_t kv_bytes = (size_t)b * rows * d * (kv_format == SA_KV_BF16 ? 2 : 1);
    // every argument other than the workspace is checked before the workspace is looked at, so a
    // call without one validates the others (and enqueues nothing)
    if (overlaps(o, o_bytes, q, o_bytes) || overlaps(o, o_bytes, kv, kv_bytes) ||
        overlaps(o, o_bytes, idx, n_tok * topk * 4) || overlaps(o, o_bytes, sink, h * 4) ||
        (kv_scale && overlaps(o, o_bytes, kv_scale, (size_t)b * rows * (d / 32))))
        return SA_ERR_INVALID_ARG;
    // the family this call runs in needs no more than sa_sparse_attn_workspace_size returns
    const size_t need = sa::routed_workspace_bytes(fam, b, s, h, d, rows, topk);
    if (!workspace || workspace_bytes < need) return SA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return SA_ERR_INVALID_ARG;
    if (overlaps(o, o_bytes, workspace, need)) return SA_ERR_INVALID_ARG;

    sa::AttnCall c;
    c.q = q;
    c.kv = kv;
    c.kv_scale = kv_scale;
    c.kv_format = kv_format;
    c.sink = sink;
    c.idx = idx;
    c.softmax_scale = softmax_scale;
    c.b = b;
    c.s = s;
    c.h = h;
    c.d = d;
    c.rows = rows;
    c.topk = topk;
    c.o = o;
    c.status = reinterpret_cast<uint32_t*>(workspace);
    c.scratch = reinterpret_cast<uint8_t*>(workspace) + SA_STATUS_BYTES;
    c.scratch_bytes = workspace_bytes - SA_STATUS_BYTES;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    c.rope = rope;
    c.rope_dim = rope_dim;
    c.rope_pos0 = rope_pos0;
    if (fam == SA_FAMILY_TCGEN05) return from_cuda(sa::attn_tc_launch(c));
    return from_cuda(sa::attn_mma_launch(c));
}

}  // namespace

extern "C" {

sa_status sa_window_idxs(int64_t start_pos, int64_t seqlen, int window, int32_t* idx, int64_t ld,
                         int64_t nbatch, int64_t batch_stride, void* stream) {
    if (window < 1 || seqlen < 0 || start_pos < 0 || nbatch < 0 || ld < window)
        return SA_ERR_INVALID_ARG;
    if (nbatch > 1 && batch_stride < seqlen * ld) return SA_ERR_INVALID_ARG;
    if (start_pos > 0 && seqlen > 1) return SA_ERR_UNSUPPORTED;
    if (seqlen == 0 || nbatch == 0) return SA_OK;
    if (!idx || !aligned(idx, 4)) return SA_ERR_INVALID_ARG;
    return from_cuda(sa::window_idxs_launch(start_pos, seqlen, window, idx, ld, nbatch,
                                            batch_stride, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sa_act_quant_fp8(const void* x, int64_t n, int d, int64_t x_stride, void* x_rt,
                           int64_t rt_stride, uint8_t* codes, int64_t codes_stride,
                           uint8_t* scales, int64_t scales_stride, void* stream) {
    if (n < 0 || d < 32 || d % 32 != 0) return SA_ERR_INVALID_ARG;
    if (!x_rt && !codes && !scales) return SA_ERR_INVALID_ARG;
    if (n == 0) return SA_OK;
    if (!x || !aligned(x, 2) || x_stride < d) return SA_ERR_INVALID_ARG;
    if (x_rt && (!aligned(x_rt, 2) || rt_stride < d)) return SA_ERR_INVALID_ARG;
    if (codes && codes_stride < d) return SA_ERR_INVALID_ARG;
    if (scales && scales_stride < d / 32) return SA_ERR_INVALID_ARG;
    if (x_rt && x_rt != x && overlaps(x_rt, (size_t)((n - 1) * rt_stride + d) * 2, x,
                                      (size_t)((n - 1) * x_stride + d) * 2))
        return SA_ERR_INVALID_ARG;  // in place is allowed; a shifted overlap is not
    if (x_rt == x && rt_stride != x_stride) return SA_ERR_INVALID_ARG;
    return from_cuda(sa::act_quant_launch(x, n, d, x_stride, x_rt, rt_stride, codes, codes_stride,
                                          scales, scales_stride,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sa_window_write(const void* x, int64_t nbatch, int64_t seqlen, int d, int64_t x_stride,
                          int64_t start_pos, int window, void* ring_rt, int64_t rt_stride,
                          int64_t rt_batch_stride, uint8_t* ring_codes, int64_t codes_stride,
                          int64_t codes_batch_stride, uint8_t* ring_scales, int64_t scales_stride,
                          int64_t scales_batch_stride, void* stream) {
    if (nbatch < 0 || seqlen < 0 || start_pos < 0 || window < 1 || d < 32 || d % 32 != 0)
        return SA_ERR_INVALID_ARG;
    if (!ring_rt && !ring_codes && !ring_scales) return SA_ERR_INVALID_ARG;
    if (nbatch == 0 || seqlen == 0) return SA_OK;
    if (!x || !aligned(x, 2) || x_stride < d) return SA_ERR_INVALID_ARG;
    // each sequence's ring: its rows, and the batch stride that keeps the rings apart
    const int64_t w1 = window - 1;
    if (ring_rt && (!aligned(ring_rt, 2) || rt_stride < d ||
                    (nbatch > 1 && rt_batch_stride < w1 * rt_stride + d)))
        return SA_ERR_INVALID_ARG;
    if (ring_codes && (codes_stride < d || (nbatch > 1 && codes_batch_stride < w1 * codes_stride + d)))
        return SA_ERR_INVALID_ARG;
    if (ring_scales && (scales_stride < d / 32 ||
                        (nbatch > 1 && scales_batch_stride < w1 * scales_stride + d / 32)))
        return SA_ERR_INVALID_ARG;
    const size_t x_bytes = (size_t)((nbatch * seqlen - 1) * x_stride + d) * 2;
    if (ring_rt && overlaps(ring_rt, (size_t)((nbatch - 1) * rt_batch_stride + w1 * rt_stride + d) * 2,
                            x, x_bytes))
        return SA_ERR_INVALID_ARG;
    if (ring_codes && overlaps(ring_codes, (size_t)((nbatch - 1) * codes_batch_stride + w1 * codes_stride + d),
                               x, x_bytes))
        return SA_ERR_INVALID_ARG;
    if (ring_scales && overlaps(ring_scales,
                                (size_t)((nbatch - 1) * scales_batch_stride + w1 * scales_stride + d / 32),
                                x, x_bytes))
        return SA_ERR_INVALID_ARG;
    return from_cuda(sa::window_write_launch(x, nbatch, seqlen, d, x_stride, start_pos, window, ring_rt,
                                             rt_stride, rt_batch_stride, ring_codes, codes_stride,
                                             codes_batch_stride, ring_scales, scales_stride,
                                             scales_batch_stride, reinterpret_cast<cudaStream_t>(stream)));
}

sa_status sa_read_status(void* workspace, int clear, void* stream) {
    if (!workspace || !aligned(workspace, 4)) return SA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && clear) {
        e = cudaMemsetAsync(workspace, 0, sizeof word, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) return SA_ERR_CUDA;
    if (word & sa::kStatusTimeout) return SA_ERR_TIMEOUT;
    if (word & sa::kStatusBadIndex) return SA_ERR_INDEX;
    return SA_OK;
}

const char* sa_status_string(int status) {
    switch (status) {
        case SA_OK: return "ok";
        case SA_ERR_INVALID_ARG: return "invalid argument";
        case SA_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case SA_ERR_CUDA: return "CUDA error";
        case SA_ERR_INDEX: return "index outside [-1, rows) seen";
        case SA_ERR_WORKSPACE: return "workspace missing or too small";
        case SA_ERR_TIMEOUT: return "a kernel wait gave up (pipeline stalled)";
        default: return "unknown status";
    }
}

int sa_version(void) { return kVersion; }

}  // extern "C"
