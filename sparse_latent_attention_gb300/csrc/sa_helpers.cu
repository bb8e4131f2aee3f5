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
    pdl_wait();
    pdl_trigger();
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

// The same table, four columns per thread with one 16-byte store (window and ld multiples of 4,
// idx 16-byte aligned, fewer than 2^31 groups of four): 32-bit index arithmetic only.
__global__ void window_idxs4_kernel(int64_t start_pos, int seqlen, int window, int32_t* idx,
                                    int64_t ld, int nbatch, int64_t batch_stride) {
    pdl_wait();
    pdl_trigger();
    const int w4 = window >> 2;
    const int per_batch = seqlen * w4;
    const int total = per_batch * nbatch;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int bi = e / per_batch;
        const int rem = e - bi * per_batch;
        const int i = rem / w4;
        const int j = 4 * (rem - i * w4);
        // position of column j; the ring slot (decode) or the chunk position (prefill)
        const int64_t pos0 = (start_pos == 0 ? (int64_t)i : start_pos) - window + 1 + j;
        int32_t v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t pos = pos0 + k;
            v[k] = pos < 0 ? -1 : (int32_t)(start_pos == 0 ? pos : pos % window);
        }
        *reinterpret_cast<int4*>(idx + bi * batch_stride + i * ld + j) = make_int4(v[0], v[1], v[2], v[3]);
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
    pdl_wait();
    pdl_trigger();
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
    pdl_wait();
    pdl_trigger();
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

// Eight consecutive elements of one 32-element block per lane, four lanes per block (lanes
// 4k .. 4k + 3 of a warp, which enter and leave together): the block maximum takes two shuffles
// within the group.  The arithmetic is quant_block32's: amax floored at 1e-4, s = pow2_ceil(amax /
// 448) (f32 division, round to nearest), e4m3 of v / s (v times the exact power-of-two 1 / s),
// bf16 of code * s.  Writes whichever of rt (8 bf16), code (8 bytes) and scale (the group's first
// lane) are given.  in holds the eight elements as bf16 pairs.
__device__ __forceinline__ void quant_group8(uint4 in, __nv_bfloat16* rt, uint8_t* code, uint8_t* scale,
                                             bool first) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    float v[8];
    uint32_t amax_bits = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        amax_bits = max(amax_bits, max((w[i] << 16) & 0x7FFFFFFFu, (w[i] & 0x7FFF0000u)));
    }
    const unsigned grp = 0xFu << (threadIdx.x & 28);
    amax_bits = max(amax_bits, __shfl_xor_sync(grp, amax_bits, 1, 4));
    amax_bits = max(amax_bits, __shfl_xor_sync(grp, amax_bits, 2, 4));
    float amax = __uint_as_float(amax_bits);
    if (amax < 1e-4f) amax = 1e-4f;
    const float sc = pow2_ceil_bits(__fdiv_rn(amax, 448.0f));
    const uint32_t se = (__float_as_uint(sc) >> 23) & 0xFFu;  // 2^(se - 127); 105 <= se <= 254
    const float inv = __uint_as_float((254u - se) << 23);      // 1 / s, exact
    uint32_t cw[2] = {0u, 0u};
    uint32_t rw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint16_t c2;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c2) : "f"(v[2 * i + 1] * inv), "f"(v[2 * i] * inv));
        cw[i >> 1] |= (uint32_t)c2 << (16 * (i & 1));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
        const float a = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * sc;
        const float b = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * sc;
        __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
        rw[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    if (code) *reinterpret_cast<uint2*>(code) = make_uint2(cw[0], cw[1]);
    if (rt) *reinterpret_cast<uint4*>(rt) = make_uint4(rw[0], rw[1], rw[2], rw[3]);
    if (scale && first) *scale = (uint8_t)se;
}

// act_quant over n rows, eight elements per thread (see quant_group8).  Row r at x + r xs; the
// outputs at the same row offsets with their own strides.  Requires x and x_rt 16-byte aligned,
// strides in elements multiples of 8 (codes: 8 bytes), fewer than 2^31 groups of eight.
__global__ void act_quant8_kernel(const __nv_bfloat16* x, int64_t n, int d, int64_t xs,
                                  __nv_bfloat16* x_rt, int64_t rts, uint8_t* codes, int64_t cs,
                                  uint8_t* scales, int64_t ss) {
    pdl_wait();
    pdl_trigger();
    const int g8 = d >> 3;
    const int total = (int)(n * g8);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int r = e / g8;
        const int c = 8 * (e - r * g8);
        const uint4 in = *reinterpret_cast<const uint4*>(x + (int64_t)r * xs + c);
        quant_group8(in, x_rt ? x_rt + (int64_t)r * rts + c : nullptr,
                     codes ? codes + (int64_t)r * cs + c : nullptr,
                     scales ? scales + (int64_t)r * ss + (c >> 5) : nullptr, (c & 31) == 0);
    }
}

// The ring write with act_quant fused, eight elements per thread (window_write_kernel's mapping;
// the same alignment conditions as act_quant8_kernel, the batch strides multiples of 8 too).
__global__ void window_write8_kernel(const __nv_bfloat16* x, int64_t nbatch, int64_t seqlen, int d,
                                     int64_t xs, int64_t start_pos, int window,
                                     __nv_bfloat16* rt, int64_t rts, int64_t rtb,
                                     uint8_t* codes, int64_t cs, int64_t cbs,
                                     uint8_t* scales, int64_t ss, int64_t sbs) {
    pdl_wait();
    pdl_trigger();
    const int g8 = d >> 3;
    const int64_t t_first = seqlen > window ? seqlen - window : 0;
    const int per_seq = (int)(seqlen - t_first);
    const int total = (int)(nbatch * per_seq * g8);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        const int row = e / g8;
        const int c = 8 * (e - row * g8);
        const int bi = row / per_seq;
        const int64_t t = t_first + (row - bi * per_seq);
        const int64_t slot = (start_pos + t) % window;
        const uint4 in = *reinterpret_cast<const uint4*>(x + ((int64_t)bi * seqlen + t) * xs + c);
        quant_group8(in, rt ? rt + bi * rtb + slot * rts + c : nullptr,
                     codes ? codes + bi * cbs + slot * cs + c : nullptr,
                     scales ? scales + bi * sbs + slot * ss + (c >> 5) : nullptr, (c & 31) == 0);
    }
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool a8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

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
    if (window % 4 == 0 && ld % 4 == 0 && (nbatch == 1 || batch_stride % 4 == 0) && a16(idx) &&
        total / 4 < (int64_t(1) << 31) && seqlen < (int64_t(1) << 31)) {
        return launch_pdl(window_idxs4_kernel, dim3(grid_for(total / 4, 256)), dim3(256), 0, stream,
                          start_pos, (int)seqlen, window, idx, ld, (int)nbatch, batch_stride);
    }
    return launch_pdl(window_idxs_kernel, dim3(grid_for(total, 256)), dim3(256), 0, stream,
                      start_pos, seqlen, window, idx, ld, nbatch, batch_stride);
}

cudaError_t act_quant_launch(const void* x, int64_t n, int d, int64_t x_stride, void* x_rt,
                             int64_t rt_stride, uint8_t* codes, int64_t codes_stride,
                             uint8_t* scales, int64_t scales_stride, cudaStream_t stream) {
    const int64_t total_threads = n * (int64_t)d;
    if (total_threads == 0) return cudaSuccess;
    if (a16(x) && x_stride % 8 == 0 && (!x_rt || (a16(x_rt) && rt_stride % 8 == 0)) &&
        (!codes || (a8(codes) && codes_stride % 8 == 0)) && total_threads / 8 < (int64_t(1) << 31)) {
        return launch_pdl(act_quant8_kernel, dim3(grid_for(total_threads / 8, 256)), dim3(256), 0,
                          stream, (const __nv_bfloat16*)x, n, d, x_stride, (__nv_bfloat16*)x_rt,
                          rt_stride, codes, codes_stride, scales, scales_stride);
    }
    return launch_pdl(act_quant_kernel, dim3(grid_for(total_threads, 256)), dim3(256), 0, stream,
                      (const __nv_bfloat16*)x, n, d, x_stride, (__nv_bfloat16*)x_rt, rt_stride,
                      codes, codes_stride, scales, scales_stride);
}

cudaError_t window_write_launch(const void* x, int64_t nbatch, int64_t seqlen, int d,
                                int64_t x_stride, int64_t start_pos, int window, void* ring_rt,
                                int64_t rt_stride, int64_t rt_batch_stride, uint8_t* codes,
                                int64_t codes_stride, int64_t codes_batch_stride, uint8_t* scales,
                                int64_t scales_stride, int64_t scales_batch_stride,
                                cudaStream_t stream) {
    const int64_t rows = nbatch * (seqlen < window ? seqlen : (int64_t)window);
    if (rows * d == 0) return cudaSuccess;
    if (a16(x) && x_stride % 8 == 0 &&
        (!ring_rt || (a16(ring_rt) && rt_stride % 8 == 0 && rt_batch_stride % 8 == 0)) &&
        (!codes || (a8(codes) && codes_stride % 8 == 0 && codes_batch_stride % 8 == 0)) &&
        rows * d / 8 < (int64_t(1) << 31)) {
        return launch_pdl(window_write8_kernel, dim3(grid_for(rows * d / 8, 256)), dim3(256), 0,
                          stream, (const __nv_bfloat16*)x, nbatch, seqlen, d, x_stride, start_pos,
                          window, (__nv_bfloat16*)ring_rt, rt_stride, rt_batch_stride, codes,
                          codes_stride, codes_batch_stride, scales, scales_stride,
                          scales_batch_stride);
    }
    return launch_pdl(window_write_kernel, dim3(grid_for(rows * d, 256)), dim3(256), 0, stream,
                      (const __nv_bfloat16*)x, nbatch, seqlen, d, x_stride, start_pos, window,
                      (__nv_bfloat16*)ring_rt, rt_stride, rt_batch_stride, codes, codes_stride,
                      codes_batch_stride, scales, scales_stride, scales_batch_stride);
}

}  // namespace sa
