// The indexer's two selection steps ("DeepSeek V4.1" source-layer attention page (indexer view)) and their C ABI entries
// (include/sa_indexer.h):
//   indexer_topk_kernel      Indexer.forward after the scores: visibility mask, the optional
//                            level-two candidate mask, topk, sort into position order,
//                            unreachable -> -1, the rest + offset
//   candidate_blocks_kernel  select_candidate_blocks: block maxima, the newest reachable block
//                            pinned, the top blocks kept (minus -inf picks), expanded to a mask
//
// One CTA per query row.  Scores become order-preserving 32-bit keys in shared memory (a
// position the query cannot reach is never read: its key is that of -inf).  A radix select
// over the keys, eight bits a pass from the top, finds the k-th largest key T and how many keys
// equal to T the k picks need.  One pass in position order then decides every key: a key above T
// is a pick, and a key equal to T is one when fewer than `need` equal keys come before it (equal
// scores are picked lowest position first), so picks come out in position order with no sort.

#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_indexer.h"

namespace {

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // the key of -inf
constexpr uint32_t kKeyPosInf = 0xFF800000u;  // the key of +inf

// Order-preserving map of an f32 bit pattern to an unsigned key: larger float, larger key.  -0 is
// taken as +0, so the two are one key.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
    if ((bits & 0x7FFFFFFFu) == 0u) bits = 0u;
    return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

template <bool kBf16>
__device__ __forceinline__ uint32_t load_key(const void* row, int t) {
    if constexpr (kBf16)
        return order_key((uint32_t)__ldg(reinterpret_cast<const uint16_t*>(row) + t) << 16);
    else
        return order_key(__ldg(reinterpret_cast<const uint32_t*>(row) + t));
}

struct SelectSmem {
    uint32_t hist[256];
    uint32_t warp_tot[2][32][2];
    uint32_t sel[2];  // a pass's digit, and the picks still needed inside it
};

// The k-th largest of keys[0, n) (1 <= k <= n): T, and need = how many of the k picks equal T
// (the other k - need are above T).  Every thread of the block calls it.
template <int kThreads>
__device__ void radix_select(const uint32_t* keys, int n, uint32_t k, SelectSmem& S, uint32_t& T,
                             uint32_t& need) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, pmask = 0u, krem = k;
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreads) S.hist[i] = 0u;
        __syncthreads();
        for (int t = tid; t < n; t += kThreads) {
            const uint32_t key = keys[t];
            // a plain shared atomic per key: measured faster than grouping a warp's equal digits
            // first (__match_any_sync), although the top digit of N(0, 1) scores falls in a few bins
            if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 255 - 8l down to 248 - 8l: lane order is descending digit order
            uint32_t c[8], sum = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = S.hist[255 - 8 * lane - j];
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
                        S.sel[0] = (uint32_t)(255 - 8 * lane - j);
                        S.sel[1] = krem - cum;
                        break;
                    }
                    cum += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= S.sel[0] << shift;
        pmask |= 0xFFu << shift;
        krem = S.sel[1];
    }
    T = prefix;
    need = krem;
}

// One pass over keys[0, n) in position order, kThreads positions a round.  For its position t of
// a round, every thread calls decide(t, pick, slot): pick tells whether t is one of the k picks
// and slot is its index among the picks in position order.  kStopEarly ends the pass once all k
// picks have been seen (nothing after them is needed).
template <int kThreads, bool kStopEarly, class Decide>
__device__ void rank_picks(const uint32_t* keys, int n, uint32_t k, uint32_t T, uint32_t need,
                           SelectSmem& S, Decide decide) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kThreads / 32;
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t run_gt = 0u, run_eq = 0u;
    int buf = 0;
    for (int base = 0; base < n; base += kThreads, buf ^= 1) {
        const int t = base + tid;
        const uint32_t key = t < n ? keys[t] : 0u;
        const bool gt = t < n && key > T, eq = t < n && key == T;
        const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) {
            S.warp_tot[buf][warp][0] = (uint32_t)__popc(bg);
            S.warp_tot[buf][warp][1] = (uint32_t)__popc(be);
        }
        __syncthreads();
        // this warp's offsets and the round's totals: a shuffle scan over the warps' counts
        uint32_t cg = lane < kWarps ? S.warp_tot[buf][lane][0] : 0u;
        uint32_t ce = lane < kWarps ? S.warp_tot[buf][lane][1] : 0u;
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
        const bool pick = gt || (eq && ebef < need);
        const uint32_t slot = gt ? gbef + min(ebef, need) : gbef + ebef;
        if (t < n) decide(t, pick, slot);
        run_gt += tg;
        run_eq += te;
        if (kStopEarly && run_gt + min(run_eq, need) >= k) break;  // uniform over the block
    }
}

// positions query si of a call sees: (si + 1) / ratio at a prefill, all n at a decode step
__device__ __forceinline__ int visible_of(int64_t si, int64_t start_pos, int ratio, int n) {
    return start_pos == 0 ? (int)((si + 1) / ratio) : n;
}

template <bool kBf16>
__device__ __forceinline__ const void* row_of(const void* base, int64_t row, int n) {
    if constexpr (kBf16) return reinterpret_cast<const uint16_t*>(base) + row * (int64_t)n;
    else return reinterpret_cast<const uint32_t*>(base) + row * (int64_t)n;
}

template <int kThreads, bool kBf16>
__global__ void __launch_bounds__(kThreads)
    indexer_topk_kernel(const void* __restrict__ score, const uint8_t* __restrict__ candidates,
                        int64_t s, int n, int64_t start_pos, int ratio, int k, int32_t offset,
                        int32_t* __restrict__ idx, int64_t ld, int64_t batch_stride) {
    extern __shared__ uint32_t keys[];  // n keys
    __shared__ SelectSmem S;
    const int64_t row = blockIdx.x;
    const int64_t bi = row / s, si = row - bi * s;
    const int visible = visible_of(si, start_pos, ratio, n);
    const void* src = row_of<kBf16>(score, row, n);
    const uint8_t* cand = candidates ? candidates + row * (int64_t)n : nullptr;
#pragma unroll 4
    for (int t = threadIdx.x; t < n; t += kThreads) {
        // outside the candidate blocks (level two) a score is -inf too
        const bool seen = t < visible && (cand == nullptr || __ldg(cand + t) != 0);
        keys[t] = seen ? load_key<kBf16>(src, t) : kKeyNegInf;
    }
    __syncthreads();
    uint32_t T, need;
    radix_select<kThreads>(keys, n, (uint32_t)k, S, T, need);
    int32_t* out = idx + bi * batch_stride + si * ld;
    rank_picks<kThreads, true>(keys, n, (uint32_t)k, T, need, S,
                               [&](int t, bool pick, uint32_t slot) {
                                   // a slot is always below k (k - need keys lie above T); the
                                   // check keeps every store inside the row regardless
                                   if (pick && slot < (uint32_t)k)
                                       out[slot] = t < visible ? t + offset : -1;
                               });
}

template <int kThreads, bool kBf16>
__global__ void __launch_bounds__(kThreads)
    candidate_blocks_kernel(const void* __restrict__ logits, int64_t s, int n, int64_t start_pos,
                            int ratio, int kb, int bs, uint8_t* __restrict__ mask) {
    extern __shared__ uint32_t keys[];  // one key per block
    __shared__ SelectSmem S;
    const int64_t row = blockIdx.x;
    const int64_t si = row % s;
    const int visible = visible_of(si, start_pos, ratio, n);
    const int nb = (n + bs - 1) / bs;
    const void* src = row_of<kBf16>(logits, row, n);
    // a block's score is its best reachable logit (-inf when it has none, and past the row's end);
    // the block holding the newest reachable position scores +inf
    const int pinned = visible > 0 ? (visible - 1) / bs : -1;
    for (int j = threadIdx.x; j < nb; j += kThreads) {
        uint32_t best = kKeyNegInf;
        const int t1 = min(j * bs + bs, visible);
        for (int t = j * bs; t < t1; ++t) best = max(best, load_key<kBf16>(src, t));
        keys[j] = j == pinned ? kKeyPosInf : best;
    }
    __syncthreads();
    const uint32_t k = (uint32_t)min(kb, nb);  // >= 1 (the host handles topk_blocks == 0)
    uint32_t T, need;
    radix_select<kThreads>(keys, nb, k, S, T, need);
    uint8_t* m = mask + row * (int64_t)n;
    rank_picks<kThreads, false>(keys, nb, k, T, need, S, [&](int j, bool pick, uint32_t) {
        // a pick that scores -inf is dropped
        const uint8_t kept = (pick && keys[j] != kKeyNegInf) ? 1 : 0;
        const int t1 = min(j * bs + bs, n);
        for (int t = j * bs; t < t1; ++t) m[t] = kept;
    });
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

// Launch a per-row kernel with `keys` 32-bit keys of shared memory per row: 128 threads for up
// to 4096 keys (many rows per SM), 1024 beyond (a long row's passes and rounds are its latency:
// 1024 threads took the 64 x 8192 decode selection from 24.6 to 18.4 us, where 512 ran before;
// more threads made the 2048-key rows slower).
// The same with the thread count chosen by `span`, the positions a row's threads read (the
// candidate blocks' threads read every position for the block maxima, then select among the far
// fewer block keys: 1024 threads for 8192 or 32768 positions took them from 16.4 / 52.3 to
// 12.3 / 30.7 us).
template <template <int, bool> class K, bool kBf16, class... Args>
cudaError_t launch_rows_n(int keys, int span, int64_t rows, cudaStream_t stream, Args... args) {
    const size_t smem = (size_t)keys * sizeof(uint32_t);
    auto go = [&](auto kernel, int threads) -> cudaError_t {
        if (smem > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(
                kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        kernel<<<(unsigned)rows, threads, smem, stream>>>(args...);
        return cudaGetLastError();
    };
    if (span <= 4096) return go(K<128, kBf16>::fn, 128);
    return go(K<1024, kBf16>::fn, 1024);
}

template <template <int, bool> class K, bool kBf16, class... Args>
cudaError_t launch_rows(int keys, int64_t rows, cudaStream_t stream, Args... args) {
    return launch_rows_n<K, kBf16>(keys, keys, rows, stream, args...);
}

template <int kThreads, bool kBf16>
struct TopkK {
    static constexpr auto fn = indexer_topk_kernel<kThreads, kBf16>;
};
template <int kThreads, bool kBf16>
struct CandK {
    static constexpr auto fn = candidate_blocks_kernel<kThreads, kBf16>;
};

// the shape checks both entries share
sa_status check_shape(int score_format, int64_t b, int64_t s, int64_t n_comp, int64_t start_pos,
                      int ratio) {
    if (score_format != SA_SCORE_F32 && score_format != SA_SCORE_BF16) return SA_ERR_INVALID_ARG;
    if (b < 0 || s < 0 || start_pos < 0 || ratio < 1) return SA_ERR_INVALID_ARG;
    if (n_comp != (start_pos + s) / ratio) return SA_ERR_INVALID_ARG;
    if (start_pos > 0 && s > 1) return SA_ERR_UNSUPPORTED;
    if (b * s >= (int64_t(1) << 31)) return SA_ERR_UNSUPPORTED;
    return SA_OK;
}

// a call that reads scores: present and aligned for their type
bool scores_ok(const void* score, int score_format) {
    return score && aligned(score, score_format == SA_SCORE_F32 ? 4 : 2);
}

}  // namespace

extern "C" sa_status sa_indexer_topk(const void* score, int score_format,
                                     const uint8_t* candidates, int64_t b, int64_t s,
                                     int64_t n_comp, int64_t start_pos, int ratio, int index_topk,
                                     int32_t offset, int32_t* idx, int64_t ld,
                                     int64_t batch_stride, void* stream) {
    const sa_status c = check_shape(score_format, b, s, n_comp, start_pos, ratio);
    if (c != SA_OK) return c;
    if (index_topk < 0 || offset < 0) return SA_ERR_INVALID_ARG;
    const int64_t k = index_topk < n_comp ? index_topk : n_comp;
    if (b * s == 0 || k == 0) return SA_OK;
    if (!scores_ok(score, score_format)) return SA_ERR_INVALID_ARG;
    if (n_comp > SA_INDEXER_MAX_POSITIONS) return SA_ERR_UNSUPPORTED;
    if ((int64_t)offset + n_comp > INT32_MAX) return SA_ERR_INVALID_ARG;
    if (!idx || !aligned(idx, 4) || ld < k) return SA_ERR_INVALID_ARG;
    if (b > 1 && batch_stride < (s - 1) * ld + k) return SA_ERR_INVALID_ARG;
    const size_t n_scores = (size_t)(b * s * n_comp);
    const size_t score_bytes = n_scores * (score_format == SA_SCORE_F32 ? 4 : 2);
    const size_t idx_bytes = (size_t)((b - 1) * (b > 1 ? batch_stride : 0) + (s - 1) * ld + k) * 4;
    if (overlaps(score, score_bytes, idx, idx_bytes)) return SA_ERR_INVALID_ARG;
    if (candidates && overlaps(candidates, n_scores, idx, idx_bytes)) return SA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int n = (int)n_comp;
    const cudaError_t e =
        score_format == SA_SCORE_BF16
            ? launch_rows<TopkK, true>(n, b * s, st, score, candidates, s, n, start_pos, ratio,
                                       (int)k, offset, idx, ld, batch_stride)
            : launch_rows<TopkK, false>(n, b * s, st, score, candidates, s, n, start_pos, ratio,
                                        (int)k, offset, idx, ld, batch_stride);
    return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

extern "C" sa_status sa_candidate_blocks(const void* logits, int score_format, int64_t b, int64_t s,
                                         int64_t n_comp, int64_t start_pos, int ratio,
                                         int topk_blocks, int block_size, uint8_t* mask,
                                         void* stream) {
    const sa_status c = check_shape(score_format, b, s, n_comp, start_pos, ratio);
    if (c != SA_OK) return c;
    if (topk_blocks < 0 || block_size < 1) return SA_ERR_INVALID_ARG;
    if (b * s == 0 || n_comp == 0) return SA_OK;
    if (!scores_ok(logits, score_format)) return SA_ERR_INVALID_ARG;
    const int64_t nb = (n_comp + block_size - 1) / block_size;
    if (nb > SA_INDEXER_MAX_POSITIONS || n_comp > INT32_MAX / 2) return SA_ERR_UNSUPPORTED;
    if (!mask) return SA_ERR_INVALID_ARG;
    const size_t n_scores = (size_t)(b * s * n_comp);
    if (overlaps(logits, n_scores * (score_format == SA_SCORE_F32 ? 4 : 2), mask, n_scores))
        return SA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (topk_blocks == 0)  // no block is kept
        return cudaMemsetAsync(mask, 0, n_scores, st) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
    const int n = (int)n_comp;
    const cudaError_t e =
        score_format == SA_SCORE_BF16
            ? launch_rows_n<CandK, true>((int)nb, n, b * s, st, logits, s, n, start_pos, ratio,
                                         topk_blocks, block_size, mask)
            : launch_rows_n<CandK, false>((int)nb, n, b * s, st, logits, s, n, start_pos, ratio,
                                          topk_blocks, block_size, mask);
    return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}
