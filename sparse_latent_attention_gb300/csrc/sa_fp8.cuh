// e4m3 + e8m0 (block 32) kv rows widened to bf16, shared by both sparse_attn kernel families.
//
// An e4m3 code times a power-of-two scale has at most four significant bits, so the product
// is exact in bf16: the widened row equals the act_quant round trip of the original row ("Module
// attn" API page, act_quant_inplace and the precision paragraph).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace sa {
namespace fp8 {

// 2^(e - 127) for an e8m0 byte (e = 0 is 2^-127, a subnormal f32).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
    return e == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);
}

// Sixteen e4m3 codes times one power-of-two scale -> sixteen bf16 values (exact): elements
// 0..7 in lo, 8..15 in hi, lowest element in the low half of each word.  Per pair of codes: one
// conversion to f16 (exact), two widenings to f32, one paired multiply by the scale (two
// round-to-nearest f32 products in one instruction) and one packing to bf16.
__device__ __forceinline__ void dequant16(uint4 c, float sc, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint64_t sc2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(sc2) : "f"(sc));
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint16_t pair = (uint16_t)(w[i] >> (16 * half));
            uint32_t h2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
            const float a = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
            const float b = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
            uint64_t ab;
            asm("{\n .reg .b64 t;\n mov.b64 t, {%1, %2};\n mul.rn.f32x2 %0, t, %3;\n}"
                : "=l"(ab) : "f"(a), "f"(b), "l"(sc2));
            float as, bs;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(as), "=f"(bs) : "l"(ab));
            __nv_bfloat162 v = __floats2bfloat162_rn(as, bs);
            out[2 * i + half] = *reinterpret_cast<uint32_t*>(&v);
        }
    }
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

}  // namespace fp8
}  // namespace sa
