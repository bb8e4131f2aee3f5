// hc_split_sinkhorn ("DeepSeek V4.1" attention-write page (decode)): a Hyper-Connections block's per-token mixes
// split into pre / post weights and a Sinkhorn-normalised comb matrix, and its C ABI entry
// (include/sa_hc.h).
//
// One thread per token.  A block's 256 rows of mixes are staged through shared memory (a
// coalesced copy in, one padded row per thread), computed in registers in f32, and the outputs
// leave through the same buffer as coalesced stores.  96 bytes in and 96 out per token at hc = 4;
// a normalisation takes one reciprocal of its sum and multiplies (the page divides each entry:
// one more rounding per step), since the ~640 divisions a token would otherwise take bound the
// kernel, not its bytes.  The reciprocal is the hardware's approximation refined by one
// Newton-Raphson step (within about one ulp; the sums are positive and normal).

#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_hc.h"

namespace {

constexpr int kTok = 256;  // tokens (threads) per block

// 1 / x for a positive normal f32: y0 = rcp.approx(x) (relative error below 2^-22), then one
// Newton-Raphson step for f(y) = 1 / y - x, y1 = y0 + y0 (1 - x y0), which squares the relative
// error.
__device__ __forceinline__ float recip(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return fmaf(y, fmaf(-x, y, 1.0f), y);
}

// f32 pairs (two lanes of one 64-bit register) for the packed add and multiply: each lane is the
// same round-to-nearest operation as a scalar one.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// recip() of both lanes: the two approximations, then the Newton-Raphson step in pairs.
__device__ __forceinline__ uint64_t recip2(uint64_t x) {
    float a, b, ya, yb;
    f2_split(x, a, b);
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(ya) : "f"(a));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(yb) : "f"(b));
    const uint64_t y = f2(ya, yb);
    const uint64_t e = ffma2(fmul2(x, f2(-1.f, -1.f)), y, f2(1.f, 1.f));  // 1 - x y (exact product)
    return ffma2(y, e, y);
}

template <int HC>
__global__ void __launch_bounds__(kTok)
    hc_split_sinkhorn_kernel(const float* __restrict__ mixes, int64_t n,
                             const float* __restrict__ scale, const float* __restrict__ base,
                             int iters, float eps, float* __restrict__ pre,
                             float* __restrict__ post, float* __restrict__ comb) {
    constexpr int kMix = (2 + HC) * HC;  // values a token has, in and out
    constexpr int kStride = kMix + 1;    // odd row stride: a thread's row reads are conflict-free
    __shared__ float rows[kTok * kStride];
    __shared__ float sb[kMix];
    __shared__ float ss[3];
    const int tid = threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    const int ntok = (int)min((int64_t)kTok, n - t0);
    const float* src = mixes + t0 * kMix;
    for (int e = tid; e < ntok * kMix; e += kTok) {
        const int r = e / kMix;
        rows[r * kStride + (e - r * kMix)] = __ldg(src + e);
    }
    if (tid < kMix) sb[tid] = __ldg(base + tid);
    if (tid < 3) ss[tid] = __ldg(scale + tid);
    __syncthreads();

    float pr[HC], po[HC], c[HC][HC];
    if (tid < ntok) {
        const float* m = rows + tid * kStride;
#pragma unroll
        for (int j = 0; j < HC; ++j) {
            pr[j] = 1.f / (1.f + expf(-(m[j] * ss[0] + sb[j]))) + eps;
            po[j] = 2.f / (1.f + expf(-(m[HC + j] * ss[1] + sb[HC + j])));
        }
#pragma unroll
        for (int j = 0; j < HC; ++j)
#pragma unroll
            for (int k = 0; k < HC; ++k)
                c[j][k] = m[2 * HC + j * HC + k] * ss[2] + sb[2 * HC + j * HC + k];
        // each row: softmax, plus eps
#pragma unroll
        for (int j = 0; j < HC; ++j) {
            float mx = c[j][0];
#pragma unroll
            for (int k = 1; k < HC; ++k) mx = fmaxf(mx, c[j][k]);
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < HC; ++k) {
                c[j][k] = expf(c[j][k] - mx);
                sum += c[j][k];
            }
            const float inv = recip(sum);
#pragma unroll
            for (int k = 0; k < HC; ++k) c[j][k] = c[j][k] * inv + eps;
        }
        // a column step, then iters - 1 rounds of a row step and a column step, on the matrix held
        // as pairs of columns (cp[j][q] = columns 2q, 2q + 1 of row j): a row's sum is one paired
        // add and one add, a pair of columns' sums three paired adds, the scaling paired multiplies
        static_assert(HC == 4, "the paired Sinkhorn rounds are written for hc = 4");
        uint64_t cp[HC][2];
#pragma unroll
        for (int j = 0; j < HC; ++j) {
            cp[j][0] = f2(c[j][0], c[j][1]);
            cp[j][1] = f2(c[j][2], c[j][3]);
        }
        const uint64_t eps2 = f2(eps, eps);
#pragma unroll 1
        for (int it = 0; it < iters; ++it) {
            if (it > 0) {
#pragma unroll
                for (int j = 0; j < HC; j += 2) {  // two rows' sums and reciprocals in a pair
                    float a0, b0, a1, b1;
                    f2_split(fadd2(cp[j][0], cp[j][1]), a0, b0);
                    f2_split(fadd2(cp[j + 1][0], cp[j + 1][1]), a1, b1);
                    float i0, i1;
                    f2_split(recip2(fadd2(f2(a0 + b0, a1 + b1), eps2)), i0, i1);
                    const uint64_t inv0 = f2(i0, i0), inv1 = f2(i1, i1);
                    cp[j][0] = fmul2(cp[j][0], inv0);
                    cp[j][1] = fmul2(cp[j][1], inv0);
                    cp[j + 1][0] = fmul2(cp[j + 1][0], inv1);
                    cp[j + 1][1] = fmul2(cp[j + 1][1], inv1);
                }
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint64_t sum = fadd2(fadd2(fadd2(cp[0][q], cp[1][q]), fadd2(cp[2][q], cp[3][q])), eps2);
                const uint64_t inv2 = recip2(sum);
#pragma unroll
                for (int j = 0; j < HC; ++j) cp[j][q] = fmul2(cp[j][q], inv2);
            }
        }
#pragma unroll
        for (int j = 0; j < HC; ++j) {
            f2_split(cp[j][0], c[j][0], c[j][1]);
            f2_split(cp[j][1], c[j][2], c[j][3]);
        }
    }
    __syncthreads();  // every row has been read: the buffer now takes the outputs
    if (tid < ntok) {
        float* o = rows + tid * kStride;
#pragma unroll
        for (int j = 0; j < HC; ++j) {
            o[j] = pr[j];
            o[HC + j] = po[j];
#pragma unroll
            for (int k = 0; k < HC; ++k) o[2 * HC + j * HC + k] = c[j][k];
        }
    }
    __syncthreads();
    for (int e = tid; e < ntok * HC; e += kTok) {
        const int r = e / HC, j = e - r * HC;
        pre[t0 * HC + e] = rows[r * kStride + j];
        post[t0 * HC + e] = rows[r * kStride + HC + j];
    }
    for (int e = tid; e < ntok * HC * HC; e += kTok) {
        const int r = e / (HC * HC);
        comb[t0 * HC * HC + e] = rows[r * kStride + 2 * HC + (e - r * HC * HC)];
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

extern "C" sa_status sa_hc_split_sinkhorn(const float* mixes, int64_t n, int hc,
                                          const float* hc_scale, const float* hc_base,
                                          int sinkhorn_iters, float eps, float* pre, float* post,
                                          float* comb, void* stream) {
    if (n < 0 || hc < 1 || sinkhorn_iters < 1) return SA_ERR_INVALID_ARG;
    if (hc != 4) return SA_ERR_UNSUPPORTED;
    if (n > (int64_t)INT32_MAX * kTok) return SA_ERR_INVALID_ARG;  // one block per 256 tokens
    if (n == 0) return SA_OK;
    if (!mixes || !hc_scale || !hc_base || !pre || !post || !comb) return SA_ERR_INVALID_ARG;
    if (!aligned(mixes, 16) || !aligned(hc_scale, 4) || !aligned(hc_base, 4) ||
        !aligned(pre, 4) || !aligned(post, 4) || !aligned(comb, 4))
        return SA_ERR_INVALID_ARG;
    const size_t mix = (size_t)(2 + hc) * hc;
    const size_t in_b = (size_t)n * mix * 4, pp_b = (size_t)n * hc * 4, c_b = (size_t)n * hc * hc * 4;
    const void* outs[3] = {pre, post, comb};
    const size_t out_b[3] = {pp_b, pp_b, c_b};
    for (int i = 0; i < 3; ++i) {
        if (overlaps(outs[i], out_b[i], mixes, in_b) || overlaps(outs[i], out_b[i], hc_scale, 12) ||
            overlaps(outs[i], out_b[i], hc_base, mix * 4))
            return SA_ERR_INVALID_ARG;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], out_b[i], outs[j], out_b[j])) return SA_ERR_INVALID_ARG;
    }
    const int64_t blocks = (n + kTok - 1) / kTok;
    hc_split_sinkhorn_kernel<4><<<(unsigned)blocks, kTok, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        mixes, n, hc_scale, hc_base, sinkhorn_iters, eps, pre, post, comb);
    return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}
