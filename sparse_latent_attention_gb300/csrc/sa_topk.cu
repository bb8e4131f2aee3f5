// The indexer's selection of the compressed idx ("DeepSeek V4.1" attention page, Indexer.forward:
// visibility mask, topk, sort into position order, unreachable -> -1, the rest + offset) and its
// C ABI entry (include/sa_indexer.h).
//
// One CTA per query row.  The row's scores become order-preserving 32-bit keys in shared memory
// (a hidden position is never read: its key is the key of -inf).  A radix select over the keys,
// eight bits a pass from the top, finds the k-th largest key T and how many keys equal to T the
// k picks need; a compaction in position order then writes every key above T and the first
// `need` keys equal to T, so the picks come out sorted by position with no sort.

#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_indexer.h"

namespace {

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // the key of -inf

// Order-preserving map of an f32 bit pattern to an unsigned key: larger float, larger key.  -0 is
// taken as +0, so the two are one key.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
    if ((bits & 0x7FFFFFFFu) == 0u) bits = 0u;
    return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

template <int kThreads, bool kBf16>
__global__ void __launch_bounds__(kThreads)
    indexer_topk_kernel(const void* __restrict__ score, int64_t s, int n, int64_t start_pos,
                        int ratio, int k, int32_t offset, int32_t* __restrict__ idx, int64_t ld,
                        int64_t batch_stride) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ uint32_t keys[];  // n keys
    __shared__ uint32_t hist[256];
    __shared__ uint32_t warp_tot[2][kWarps][2];
    __shared__ uint32_t sel[2];  // the pass's digit, and the picks still needed inside it
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const int64_t bi = row / s, si = row - bi * s;
    // positions this query sees: (si + 1) / ratio <= n at a prefill, all of them at a decode step
    const int visible = start_pos == 0 ? (int)((si + 1) / ratio) : n;

    if constexpr (kBf16) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(score) + row * (int64_t)n;
#pragma unroll 4
        for (int t = tid; t < n; t += kThreads)
            keys[t] = t < visible ? order_key((uint32_t)__ldg(src + t) << 16) : kKeyNegInf;
    } else {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(score) + row * (int64_t)n;
#pragma unroll 4
        for (int t = tid; t < n; t += kThreads)
            keys[t] = t < visible ? order_key(__ldg(src + t)) : kKeyNegInf;
    }

    // radix select of the k-th largest key, 8 bits a pass; keys outside the prefix chosen so far
    // take no part.  k <= n, so the chosen bin always exists.
    uint32_t prefix = 0u, pmask = 0u;
    uint32_t krem = (uint32_t)k;
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreads) hist[i] = 0u;
        __syncthreads();
        for (int base = 0; base < n; base += kThreads) {
            const int t = base + tid;
            uint32_t dig = 256u;  // no bin
            if (t < n) {
                const uint32_t key = keys[t];
                if ((key & pmask) == prefix) dig = (key >> shift) & 255u;
            }
            // a plain shared atomic per key: measured faster than grouping equal digits of a warp
            // first (__match_any_sync), although the top digit of N(0, 1) scores falls in a few bins
            if (dig < 256u) atomicAdd(&hist[dig], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 255 - 8l down to 248 - 8l: lane order is descending digit order
            uint32_t c[8], sum = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - 8 * lane - j];
                sum += c[j];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const uint32_t excl = incl - sum;
            if (excl < krem && krem <= incl) {  // exactly one lane: the k-th key's bin is here
                uint32_t cum = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (cum + c[j] >= krem) {
                        sel[0] = (uint32_t)(255 - 8 * lane - j);
                        sel[1] = krem - cum;
                        break;
                    }
                    cum += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= sel[0] << shift;
        pmask |= 0xFFu << shift;
        krem = sel[1];
    }
    const uint32_t T = prefix;   // the k-th largest key
    const uint32_t need = krem;  // keys equal to T among the picks; the rest are above T

    // compaction in position order: a key above T goes after every pick before it; a key equal to
    // T is a pick when fewer than `need` equal keys come before it
    int32_t* out = idx + bi * batch_stride + si * ld;
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t run_gt = 0u, run_eq = 0u;
    int buf = 0;
    for (int base = 0; base < n; base += kThreads, buf ^= 1) {
        const int t = base + tid;
        const uint32_t key = t < n ? keys[t] : 0u;
        const bool gt = t < n && key > T, eq = t < n && key == T;
        const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) {
            warp_tot[buf][warp][0] = (uint32_t)__popc(bg);
            warp_tot[buf][warp][1] = (uint32_t)__popc(be);
        }
        __syncthreads();
        // this warp's offsets and the round's totals: a shuffle scan over the warps' counts
        uint32_t cg = lane < kWarps ? warp_tot[buf][lane][0] : 0u;
        uint32_t ce = lane < kWarps ? warp_tot[buf][lane][1] : 0u;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t vg = __shfl_up_sync(0xffffffffu, cg, off);
            const uint32_t ve = __shfl_up_sync(0xffffffffu, ce, off);
            if (lane >= off) {
                cg += vg;
                ce += ve;
            }
        }
        const uint32_t tg = __shfl_sync(0xffffffffu, cg, 31), te = __shfl_sync(0xffffffffu, ce, 31);
        const uint32_t wg = warp > 0 ? __shfl_sync(0xffffffffu, cg, warp - 1) : 0u;
        const uint32_t we = warp > 0 ? __shfl_sync(0xffffffffu, ce, warp - 1) : 0u;
        const uint32_t gbef = run_gt + wg + (uint32_t)__popc(bg & lt);
        const uint32_t ebef = run_eq + we + (uint32_t)__popc(be & lt);
        const int32_t v = t < visible ? t + offset : -1;
        // the select leaves exactly k - need keys above T, so a slot is always below k; the
        // check keeps every store inside the row regardless
        const uint32_t slot = gt ? gbef + min(ebef, need) : gbef + ebef;
        if ((gt || (eq && ebef < need)) && slot < (uint32_t)k) out[slot] = v;
        run_gt += tg;
        run_eq += te;
        if (run_gt + min(run_eq, need) >= (uint32_t)k) break;  // every pick written (uniform)
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int kThreads, bool kBf16>
cudaError_t launch(const void* score, int64_t rows, int64_t s, int n, int64_t start_pos, int ratio,
                   int k, int32_t offset, int32_t* idx, int64_t ld, int64_t batch_stride,
                   cudaStream_t stream) {
    const size_t smem = (size_t)n * sizeof(uint32_t);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(indexer_topk_kernel<kThreads, kBf16>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) return e;
    }
    indexer_topk_kernel<kThreads, kBf16><<<(unsigned)rows, kThreads, smem, stream>>>(
        score, s, n, start_pos, ratio, k, offset, idx, ld, batch_stride);
    return cudaGetLastError();
}

// Rows of up to 4096 positions take 128 threads (many rows per SM); longer rows more threads.
template <bool kBf16>
cudaError_t launch_any(const void* score, int64_t rows, int64_t s, int n, int64_t start_pos,
                       int ratio, int k, int32_t offset, int32_t* idx, int64_t ld,
                       int64_t batch_stride, cudaStream_t stream) {
    if (n <= 4096)
        return launch<128, kBf16>(score, rows, s, n, start_pos, ratio, k, offset, idx, ld,
                                  batch_stride, stream);
    if (n <= 16384)
        return launch<512, kBf16>(score, rows, s, n, start_pos, ratio, k, offset, idx, ld,
                                  batch_stride, stream);
    return launch<1024, kBf16>(score, rows, s, n, start_pos, ratio, k, offset, idx, ld,
                               batch_stride, stream);
}

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

extern "C" sa_status sa_indexer_topk(const void* score, int score_format, int64_t b, int64_t s,
                                     int64_t n_comp, int64_t start_pos, int ratio, int index_topk,
                                     int32_t offset, int32_t* idx, int64_t ld,
                                     int64_t batch_stride, void* stream) {
    if (score_format != SA_SCORE_F32 && score_format != SA_SCORE_BF16) return SA_ERR_INVALID_ARG;
    if (b < 0 || s < 0 || start_pos < 0 || ratio < 1 || index_topk < 0 || offset < 0)
        return SA_ERR_INVALID_ARG;
    if (n_comp != (start_pos + s) / ratio) return SA_ERR_INVALID_ARG;
    if (start_pos > 0 && s > 1) return SA_ERR_UNSUPPORTED;
    const int64_t k = index_topk < n_comp ? index_topk : n_comp;
    if (b * s == 0 || k == 0) return SA_OK;
    if (n_comp > SA_INDEXER_MAX_POSITIONS) return SA_ERR_UNSUPPORTED;
    if ((int64_t)offset + n_comp > INT32_MAX) return SA_ERR_INVALID_ARG;
    if (b * s >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
    if (!score || !idx || !aligned(idx, 4) || ld < k) return SA_ERR_INVALID_ARG;
    if (!aligned(score, score_format == SA_SCORE_F32 ? 4 : 2)) return SA_ERR_INVALID_ARG;
    if (b > 1 && batch_stride < (s - 1) * ld + k) return SA_ERR_INVALID_ARG;
    const size_t score_bytes = (size_t)(b * s * n_comp) * (score_format == SA_SCORE_F32 ? 4 : 2);
    const size_t idx_bytes = (size_t)((b - 1) * (b > 1 ? batch_stride : 0) + (s - 1) * ld + k) * 4;
    if (overlaps(score, score_bytes, idx, idx_bytes)) return SA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e =
        score_format == SA_SCORE_BF16
            ? launch_any<true>(score, b * s, s, (int)n_comp, start_pos, ratio, (int)k, offset, idx,
                               ld, batch_stride, st)
            : launch_any<false>(score, b * s, s, (int)n_comp, start_pos, ratio, (int)k, offset, idx,
                                ld, batch_stride, st);
    return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}
