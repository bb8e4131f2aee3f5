// Input helpers on the sparse_attn path: the window index table and the fp8 block quantiser.
//
// Sources: "Module attn" API page (spark_model, deepseek_v41_ref/attn), Functions:
// window_topk_idxs, act_quant_inplace, pow2_ceil; Constants: FP8_BLOCK; the ring-cache and
// precision paragraphs.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_internal.cuh"

namespace sa {
namespace {

// ---------------------------------------------------------------------------------------------
// window_topk_idxs
// ---------------------------------------------------------------------------------------------

// One thread per output entry.  Prefill (start_pos == 0): row i column j holds the position
// i - window + 1 + j of the chunk, -1 before position 0.  Decode (one row at position p): the
// ring read oldest first, column j holds the slot of position p - window + 1 + j.
__global__ void window_idxs_kernel(int64_t start_pos, int64_t seqlen, int window, int32_t* idx,
                                   int64_t ld, int64_t nbatch, int64_t batch_stride) {
    const int64_t per_batch = seqlen * window;
    const int64_t total = per_batch * nbatch;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bi = e / per_batch;
        const int64_t rem = e - bi * per_batch;
        const int64_t i = rem / window;
        const int j = (int)(rem - i * window);
        int32_t v;
        if (start_pos == 0) {
            const int64_t pos = i - window + 1 + j;
            v = pos >= 0 ? (int32_t)pos : -1;
        } else {
            const int64_t pos = start_pos - window + 1 + j;
            v = pos >= 0 ? (int32_t)(pos % window) : -1;
        }
        idx[bi * batch_stride + i * ld + j] = v;
    }
}

// ---------------------------------------------------------------------------------------------
// act_quant (block 32, e4m3 values, power-of-two e8m0 scales)
// ---------------------------------------------------------------------------------------------

// 2^ceil(log2 v) for a positive normal f32, from its IEEE fields: the biased exponent plus one
// whenever a mantissa bit is set.
__device__ __forceinline__ float pow2_ceil_bits(float v) {
    const uint32_t u = __float_as_uint(v);
    const uint32_t e = (u >> 23) & 0xFFu;
    const uint32_t up = (u & 0x7FFFFFu) ? 1u : 0u;
    return __uint_as_float((e + up) << 23);
}

// f32 -> e4m3 byte, round to nearest even, saturating to +-448 (hardware conversion).
__device__ __forceinline__ uint8_t f32_to_e4m3_sat(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return (uint8_t)(r & 0xFFu);
}

// e4m3 byte -> f32 (exact, through the hardware e4m3x2 -> f16x2 conversion).
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
    uint32_t h2;
    const uint16_t in = c;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// One warp per 32-element block: lane k owns element k.  x_rt may alias x (in place): a lane
// reads its element before the block maximum is formed and writes it only afterwards.
// One 32-element block of a row, one element per lane of a converged warp: amax (floored at
// 1e-4), s = pow2_ceil(amax / 448), the e4m3 code of v / s and the bf16 round trip code * s;
// writes whichever of rt / code / scale (lane 0) are given.
__device__ __forceinline__ void quant_block32(float v, int lane, __nv_bfloat16* rt, uint8_t* code,
                                              uint8_t* scale) {
    // |v| orders like its bit pattern, so the block maximum is an integer max
    const uint32_t abits = __float_as_uint(v) & 0x7FFFFFFFu;
    float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, abits));
    if (amax < 1e-4f) amax = 1e-4f;
    const float sc = pow2_ceil_bits(__fdiv_rn(amax, 448.0f));
    const uint8_t c = f32_to_e4m3_sat(__fdiv_rn(v, sc));
    if (code) *code = c;
    if (rt) *rt = __float2bfloat16_rn(e4m3_to_f32(c) * sc);
    if (scale && lane == 0) *scale = (uint8_t)((__float_as_uint(sc) >> 23) & 0xFFu);
}

__global__ void act_quant_kernel(const __nv_bfloat16* x, int64_t n, int d,
                                 int64_t xs, __nv_bfloat16* x_rt, int64_t rts,
                                 uint8_t* __restrict__ codes, int64_t cs,
                                 uint8_t* __restrict__ scales, int64_t ss) {
    const int lane = threadIdx.x & 31;
    const int blocks_per_row = d / 32;
    const int64_t total = n * blocks_per_row;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t blk = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; blk < total;
         blk += warps) {
        const int64_t r = blk / blocks_per_row;
        const int cb = (int)(blk - r * blocks_per_row);
        const int64_t col = (int64_t)cb * 32 + lane;
        quant_block32(__bfloat162float(x[r * xs + col]), lane, x_rt ? x_rt + r * rts + col : nullptr,
                      codes ? codes + r * cs + col : nullptr, scales ? scales + r * ss + cb : nullptr);
    }
}

// Ring write ([attn-doc] ring-cache paragraph): new token t (of seqlen, at position
// start_pos + t) of sequence bi goes to ring slot (start_pos + t) mod window, quantised as
// act_quant_kernel quantises.  Only the last min(seqlen, window) tokens are written: an earlier
// token's slot belongs to a later one.  Source row (bi, t) at x + (bi * seqlen + t) * xs; ring row
// (bi, slot) at base + bi * batch stride + slot * row stride.
__global__ void window_write_kernel(const __nv_bfloat16* x, int64_t nbatch, int64_t seqlen, int d,
                                    int64_t xs, int64_t start_pos, int window,
                                    __nv_bfloat16* rt, int64_t rts, int64_t rtb,
                                    uint8_t* __restrict__ codes, int64_t cs, int64_t cbs,
                                    uint8_t* __restrict__ scales, int64_t ss, int64_t sbs) {
    const int lane = threadIdx.x & 31;
    const int blocks_per_row = d / 32;
    const int64_t t_first = seqlen > window ? seqlen - window : 0;
    const int64_t per_seq = seqlen - t_first;
    const int64_t total = nbatch * per_seq * blocks_per_row;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t blk = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; blk < total;
         blk += warps) {
        const int64_t row = blk / blocks_per_row;
        const int cb = (int)(blk - row * blocks_per_row);
        const int64_t bi = row / per_seq;
        const int64_t t = t_first + (row - bi * per_seq);
        const int64_t slot = (start_pos + t) % window;
        const int64_t col = (int64_t)cb * 32 + lane;
        quant_block32(__bfloat162float(x[(bi * seqlen + t) * xs + col]), lane,
                      rt ? rt + bi * rtb + slot * rts + col : nullptr,
                      codes ? codes + bi * cbs + slot * cs + col : nullptr,
                      scales ? scales + bi * sbs + slot * ss + cb : nullptr);
    }
}

int grid_for(int64_t work, int per_block) {
    int64_t g = (work + per_block - 1) / per_block;
    if (g < 1) g = 1;
    const int64_t cap = (int64_t)device_sm_count() * 32;  // grid-stride loops beyond this
    if (g > cap) g = cap;
    return (int)g;
}

}  // namespace

int device_sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && counts[dev]) return counts[dev];
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (n > kMaxSmCount) n = kMaxSmCount;
    if (dev >= 0 && dev < 64) counts[dev] = n;
    return n;
}

cudaError_t window_idxs_launch(int64_t start_pos, int64_t seqlen, int window, int32_t* idx,
                               int64_t ld, int64_t nbatch, int64_t batch_stride,
                               cudaStream_t stream) {
    const int64_t total = seqlen * window * nbatch;
    if (total == 0) return cudaSuccess;
    window_idxs_kernel<<<grid_for(total, 256), 256, 0, stream>>>(start_pos, seqlen, window, idx,
                                                                  ld, nbatch, batch_stride);
    return cudaGetLastError();
}

cudaError_t act_quant_launch(const void* x, int64_t n, int d, int64_t x_stride, void* x_rt,
                             int64_t rt_stride, uint8_t* codes, int64_t codes_stride,
                             uint8_t* scales, int64_t scales_stride, cudaStream_t stream) {
    const int64_t total_threads = n * (int64_t)d;
    if (total_threads == 0) return cudaSuccess;
    act_quant_kernel<<<grid_for(total_threads, 256), 256, 0, stream>>>(
        (const __nv_bfloat16*)x, n, d, x_stride, (__nv_bfloat16*)x_rt, rt_stride, codes,
        codes_stride, scales, scales_stride);
    return cudaGetLastError();
}

cudaError_t window_write_launch(const void* x, int64_t nbatch, int64_t seqlen, int d,
                                int64_t x_stride, int64_t start_pos, int window, void* ring_rt,
                                int64_t rt_stride, int64_t rt_batch_stride, uint8_t* codes,
                                int64_t codes_stride, int64_t codes_batch_stride, uint8_t* scales,
                                int64_t scales_stride, int64_t scales_batch_stride,
                                cudaStream_t stream) {
    const int64_t rows = nbatch * (seqlen < window ? seqlen : (int64_t)window);
    if (rows * d == 0) return cudaSuccess;
    window_write_kernel<<<grid_for(rows * d, 256), 256, 0, stream>>>(
        (const __nv_bfloat16*)x, nbatch, seqlen, d, x_stride, start_pos, window,
        (__nv_bfloat16*)ring_rt, rt_stride, rt_batch_stride, codes, codes_stride, codes_batch_stride,
        scales, scales_stride, scales_batch_stride);
    return cudaGetLastError();
}

}  // namespace sa
