// sparse_attn, warp-level mma.sync family.
//
// Source: "Module attn" API page (spark_model, deepseek_v41_ref/attn), Functions: sparse_attn
// and the precision paragraph; "DeepSeek V4.1" attention page, Attention.forward.
//
// One CTA takes one query token and up to 64 of its heads.  The kv rows that token's idx names
// are gathered once per tile of 64 rows into shared memory (cp.async, -1 rows zero-filled and
// masked) and serve both products:
//   S  = Q K^T      (16 heads x 64 rows per warp, K = head_dim)
//   O += P V        (16 heads x head_dim/2 per warp; the two warps of a head group split d)
// with an online softmax in f32 (base-2 exponent, running max per head) and the sink added to
// the denominator only at the end.  When the token count is too small to fill the GPU (decode),
// the idx columns are split over several CTAs that write (m, l, O) partials to the workspace and
// a second kernel merges them.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_fp8.cuh"
#include "sa_internal.cuh"

namespace sa {
namespace {

constexpr int kHeadsPerCta = 64;
constexpr int kTN = 64;            // gathered rows per tile
constexpr int kPad = 8;            // bf16 padding per smem row: conflict-free ldmatrix
constexpr int kThreads = 256;      // 4 head groups x 2 d-halves
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    const __nv_bfloat16* q;
    const void* kv;
    const uint8_t* kv_scale;
    const float* sink;
    const int32_t* idx;
    __nv_bfloat16* o;
    float* part_ml;   // [tokens][splits][h][2]  (running max in log2 units, sum)
    float* part_o;    // [tokens][splits][h][d]
    uint32_t* status;
    float scale_log2;
    int64_t s_len;
    int h;
    int64_t rows;
    int topk;
    int n_tiles;
    int n_splits;
    int tiles_per_split;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

using fp8::dequant16;
using fp8::e8m0_to_f32;

template <int D, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) attn_mma_kernel(Params p) {
    constexpr int LD = D + kPad;          // smem row stride in elements
    constexpr int DH = D / 2;             // d columns per warp
    constexpr int NT_O = DH / 8;          // O n-tiles per warp
    constexpr int NT_S = kTN / 8;         // S n-tiles
    constexpr int CH = D / 8;             // 16-byte chunks per bf16 row

    extern __shared__ __align__(128) uint8_t smem[];
    __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
    __nv_bfloat16* sKV = sQ + kHeadsPerCta * LD;
    int* sRow = reinterpret_cast<int*>(sKV + 2 * kTN * LD);

    // every global access of this kernel comes after the work queued before it on the stream
    pdl_wait();
    pdl_trigger();
    const int64_t token = blockIdx.x;
    const int split = blockIdx.y;
    const int h0 = blockIdx.z * kHeadsPerCta;
    const int hc = min(kHeadsPerCta, p.h - h0);
    const int n_hg = (hc + 15) >> 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hg = warp >> 1, dh = warp & 1;
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t bi = token / p.s_len;
    const int t_begin = split * p.tiles_per_split;
    const int t_end = min(p.n_tiles, t_begin + p.tiles_per_split);
    const int32_t* idx_tok = p.idx + token * (int64_t)p.topk;

    // Q rows of this CTA's heads (rows past hc zeroed up to the head-group boundary)
    {
        const __nv_bfloat16* qsrc = p.q + (token * p.h + h0) * (int64_t)D;
        for (int c = threadIdx.x; c < n_hg * 16 * CH; c += kThreads) {
            const int r = c / CH, k = c - r * CH;
            __nv_bfloat16* dst = sQ + r * LD + k * 8;
            if (r < hc)
                cp_async16(dst, qsrc + (int64_t)r * D + k * 8, 16);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
    }

    // Gather the kv rows of tile t into stage st.  Every thread resolves the index of the rows
    // it copies; an index outside [-1, rows) counts as -1 and raises the status bit.
    auto gather = [&](int t, int st) {
        __nv_bfloat16* base = sKV + st * kTN * LD;
        if constexpr (!kFp8) {
            const __nv_bfloat16* kvb =
                reinterpret_cast<const __nv_bfloat16*>(p.kv) + bi * p.rows * (int64_t)D;
            for (int c = threadIdx.x; c < kTN * CH; c += kThreads) {
                const int r = c / CH, k = c - r * CH;
                const int col = t * kTN + r;
                int j = col < p.topk ? idx_tok[col] : -1;
                if (j < -1 || j >= p.rows) {
                    if (k == 0) atomicOr(p.status, kStatusBadIndex);
                    j = -1;
                }
                if (k == 0) sRow[st * kTN + r] = j;
                // a zero-byte copy (empty slot) still names a valid address: q's first row
                const void* src = j >= 0 ? (const void*)(kvb + (int64_t)j * D + k * 8)
                                         : (const void*)p.q;
                cp_async16(base + r * LD + k * 8, src, j >= 0 ? 16 : 0);
            }
        } else {
            const uint8_t* kvb = reinterpret_cast<const uint8_t*>(p.kv) + bi * p.rows * (int64_t)D;
            const uint8_t* scb = p.kv_scale + bi * p.rows * (int64_t)(D / 32);
            constexpr int CH8 = D / 16;  // 16-code chunks per row
            for (int c = threadIdx.x; c < kTN * CH8; c += kThreads) {
                const int r = c / CH8, k = c - r * CH8;
                const int col = t * kTN + r;
                int j = col < p.topk ? idx_tok[col] : -1;
                if (j < -1 || j >= p.rows) {
                    if (k == 0) atomicOr(p.status, kStatusBadIndex);
                    j = -1;
                }
                if (k == 0) sRow[st * kTN + r] = j;
                uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                if (j >= 0) {
                    const uint4 codes =
                        __ldg(reinterpret_cast<const uint4*>(kvb + (int64_t)j * D + k * 16));
                    const float sc = e8m0_to_f32(__ldg(scb + (int64_t)j * (D / 32) + k / 2));
                    dequant16(codes, sc, lo, hi);
                }
                uint4* dst = reinterpret_cast<uint4*>(base + r * LD + k * 16);
                dst[0] = lo;
                dst[1] = hi;
            }
        }
    };

    if (t_begin < t_end) gather(t_begin, 0);
    cp_async_commit();

    float O[NT_O][4];
#pragma unroll
    for (int i = 0; i < NT_O; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max (log2 units), rows g and g + 8
    float l0 = 0.f, l1 = 0.f;              // this thread's share of the running sums

    const bool active = hg < n_hg;
    const uint32_t q_base = smem_u32(sQ + (hg * 16) * LD);

    for (int t = t_begin; t < t_end; ++t) {
        const int st = (t - t_begin) & 1;
        if (t + 1 < t_end) gather(t + 1, st ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        if (active) {
            const __nv_bfloat16* kvs = sKV + st * kTN * LD;
            const uint32_t kv_base = smem_u32(kvs);
            float S[NT_S][4];
#pragma unroll
            for (int i = 0; i < NT_S; ++i) S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;

            // S = Q K^T over the full head_dim
#pragma unroll 4
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                {
                    const int mi = lane >> 3, r = lane & 7;
                    const int row = r + (mi & 1) * 8, col = ks * 16 + (mi >> 1) * 8;
                    ldsm_x4(q_base + (row * LD + col) * 2, a0, a1, a2, a3);
                }
#pragma unroll
                for (int np = 0; np < NT_S / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int mi = lane >> 3, r = lane & 7;
                    const int row = np * 16 + r + (mi >> 1) * 8, col = ks * 16 + (mi & 1) * 8;
                    ldsm_x4(kv_base + (row * LD + col) * 2, b0, b1, b2, b3);
                    mma_bf16(S[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_bf16(S[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }

            // mask empty slots, scale into log2 units, online softmax
            const int* rows_st = sRow + st * kTN;
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NT_S; ++nt) {
                const int c0 = nt * 8 + 2 * t4;
                const bool v0 = rows_st[c0] >= 0, v1 = rows_st[c0 + 1] >= 0;
                S[nt][0] = v0 ? S[nt][0] * p.scale_log2 : -INFINITY;
                S[nt][1] = v1 ? S[nt][1] * p.scale_log2 : -INFINITY;
                S[nt][2] = v0 ? S[nt][2] * p.scale_log2 : -INFINITY;
                S[nt][3] = v1 ? S[nt][3] * p.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(S[nt][0], S[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(S[nt][2], S[nt][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = mn0 == -INFINITY ? 1.f : fast_exp2(m0 - mn0);
            const float al1 = mn1 == -INFINITY ? 1.f : fast_exp2(m1 - mn1);
            const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
            const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
            m0 = mn0;
            m1 = mn1;
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT_S; ++nt) {
                S[nt][0] = fast_exp2(S[nt][0] - mu0);
                S[nt][1] = fast_exp2(S[nt][1] - mu0);
                S[nt][2] = fast_exp2(S[nt][2] - mu1);
                S[nt][3] = fast_exp2(S[nt][3] - mu1);
                rs0 += S[nt][0] + S[nt][1];
                rs1 += S[nt][2] + S[nt][3];
            }
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
#pragma unroll
            for (int i = 0; i < NT_O; ++i) {
                O[i][0] *= al0;
                O[i][1] *= al0;
                O[i][2] *= al1;
                O[i][3] *= al1;
            }

            // O += P V: P straight from the S registers, V = the same kv tile (rows as k)
#pragma unroll
            for (int kc = 0; kc < kTN / 16; ++kc) {
                const uint32_t a0 = pack_bf16(S[2 * kc][0], S[2 * kc][1]);
                const uint32_t a1 = pack_bf16(S[2 * kc][2], S[2 * kc][3]);
                const uint32_t a2 = pack_bf16(S[2 * kc + 1][0], S[2 * kc + 1][1]);
                const uint32_t a3 = pack_bf16(S[2 * kc + 1][2], S[2 * kc + 1][3]);
#pragma unroll
                for (int np = 0; np < NT_O / 2; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int mi = lane >> 3, r = lane & 7;
                    const int row = kc * 16 + r + (mi & 1) * 8;
                    const int col = dh * DH + np * 16 + (mi >> 1) * 8;
                    ldsm_x4_t(kv_base + (row * LD + col) * 2, b0, b1, b2, b3);
                    mma_bf16(O[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_bf16(O[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    if (!active) return;
    // complete the row sums across the quad
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
    const float mu0 = m0 == -INFINITY ? 0.f : m0;
    const float mu1 = m1 == -INFINITY ? 0.f : m1;
    const int r0 = hg * 16 + g, r1 = r0 + 8;  // local head rows

    if (p.n_splits == 1) {
        // the sink joins the denominator only: den = l + 2^(sink * log2e - m)
        float inv0 = 0.f, inv1 = 0.f;
        if (r0 < hc && l0 > 0.f) inv0 = 1.f / (l0 + fast_exp2(p.sink[h0 + r0] * kLog2e - mu0));
        if (r1 < hc && l1 > 0.f) inv1 = 1.f / (l1 + fast_exp2(p.sink[h0 + r1] * kLog2e - mu1));
        __nv_bfloat16* orow0 = p.o + (token * p.h + h0 + r0) * (int64_t)D + dh * DH;
        __nv_bfloat16* orow1 = p.o + (token * p.h + h0 + r1) * (int64_t)D + dh * DH;
#pragma unroll
        for (int nt = 0; nt < NT_O; ++nt) {
            const int c = nt * 8 + 2 * t4;
            if (r0 < hc)
                *reinterpret_cast<uint32_t*>(orow0 + c) = pack_bf16(O[nt][0] * inv0, O[nt][1] * inv0);
            if (r1 < hc)
                *reinterpret_cast<uint32_t*>(orow1 + c) = pack_bf16(O[nt][2] * inv1, O[nt][3] * inv1);
        }
    } else {
        const int64_t pbase = (token * p.n_splits + split) * (int64_t)p.h + h0;
        if (t4 == 0) {
            if (r0 < hc) {
                p.part_ml[(pbase + r0) * 2 + 0] = mu0;
                p.part_ml[(pbase + r0) * 2 + 1] = l0;
            }
            if (r1 < hc) {
                p.part_ml[(pbase + r1) * 2 + 0] = mu1;
                p.part_ml[(pbase + r1) * 2 + 1] = l1;
            }
        }
        float* po0 = p.part_o + (pbase + r0) * (int64_t)D + dh * DH;
        float* po1 = p.part_o + (pbase + r1) * (int64_t)D + dh * DH;
#pragma unroll
        for (int nt = 0; nt < NT_O; ++nt) {
            const int c = nt * 8 + 2 * t4;
            if (r0 < hc) *reinterpret_cast<float2*>(po0 + c) = make_float2(O[nt][0], O[nt][1]);
            if (r1 < hc) *reinterpret_cast<float2*>(po1 + c) = make_float2(O[nt][2], O[nt][3]);
        }
    }
}

// Merge the split partials of one token: M = max_s m_s;
// o = sum_s 2^(m_s - M) O_s / (2^(sink log2e - M) + sum_s 2^(m_s - M) l_s), zero when no row.
// One block of d / 4 threads per (token, head): thread i merges columns 4 i .. 4 i + 3 of the
// split partials in one pass over the splits, four at a time (their statistics and partial
// columns are loaded together, so the loads of a group overlap), rescaling its running sums
// whenever a split raises the maximum.  Splits with l = 0 (no row) are skipped.
__global__ void attn_combine_kernel(const float* __restrict__ part_ml,
                                    const float* __restrict__ part_o,
                                    const float* __restrict__ sink, __nv_bfloat16* __restrict__ o,
                                    int h, int d, int n_splits) {
    // the attention kernel this launch depends on has completed and its partials are visible
    // after this point
    pdl_wait();
    pdl_trigger();
    const int64_t th = blockIdx.x;  // token * h + head
    const int hh = (int)(th % h);
    const int64_t token = th / h;
    const int c = 4 * threadIdx.x;
    const float2* ml0 = reinterpret_cast<const float2*>(part_ml) + token * n_splits * (int64_t)h + hh;
    const float* po0 = part_o + (token * n_splits * (int64_t)h + hh) * d + c;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n_splits; s0 += 4) {
        float2 ml[4];
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool in = s0 + i < n_splits;
            ml[i] = in ? ml0[(int64_t)(s0 + i) * h] : make_float2(0.f, 0.f);
            v[i] = in ? *reinterpret_cast<const float4*>(po0 + (int64_t)(s0 + i) * h * d)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (!(ml[i].y > 0.f)) continue;
            if (ml[i].x > M) {  // a new maximum: rescale what was summed so far (0 at the start)
                const float r = M == -INFINITY ? 0.f : fast_exp2(M - ml[i].x);
                L *= r;
                acc.x *= r;
                acc.y *= r;
                acc.z *= r;
                acc.w *= r;
                M = ml[i].x;
            }
            const float w = fast_exp2(ml[i].x - M);
            L += w * ml[i].y;
            acc.x += w * v[i].x;
            acc.y += w * v[i].y;
            acc.z += w * v[i].z;
            acc.w += w * v[i].w;
        }
    }
    const float Mu = M == -INFINITY ? 0.f : M;
    const float inv = L > 0.f ? 1.f / (L + fast_exp2(sink[hh] * kLog2e - Mu)) : 0.f;
    uint2 out;
    out.x = pack_bf16(acc.x * inv, acc.y * inv);
    out.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(o + th * (int64_t)d + c) = out;
}

struct Geometry {
    int n_tiles, n_splits, tiles_per_split, hblocks;
};

// The idx columns of a token are split over several CTAs when the tokens alone would not give
// two CTAs per SM.  The split count grows with the SM count, so a workspace sized for
// kMaxSmCount SMs covers every device.
Geometry geometry(int64_t n_tokens, int h, int topk, int sms) {
    Geometry g;
    g.n_tiles = (topk + kTN - 1) / kTN;
    g.hblocks = (h + kHeadsPerCta - 1) / kHeadsPerCta;
    const int64_t base = n_tokens * g.hblocks;
    const int64_t kTargetCtas = 2 * (int64_t)sms;
    int splits = 1;
    if (g.n_tiles > 1 && base < kTargetCtas) {
        splits = (int)((kTargetCtas + base - 1) / base);
        if (splits > g.n_tiles) splits = g.n_tiles;
    }
    g.tiles_per_split = splits > 1 ? (g.n_tiles + splits - 1) / splits : (g.n_tiles > 0 ? g.n_tiles : 1);
    g.n_splits = splits > 1 ? (g.n_tiles + g.tiles_per_split - 1) / g.tiles_per_split : 1;
    return g;
}

size_t smem_bytes(int d) {
    return (size_t)(kHeadsPerCta + 2 * kTN) * (d + kPad) * 2 + 2 * kTN * sizeof(int);
}

template <int D, bool kFp8>
cudaError_t launch_t(const AttnCall& c, const Params& p, dim3 grid) {
    static bool configured[64] = {};  // per template instance and device
    const size_t smem = smem_bytes(D);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(attn_mma_kernel<D, kFp8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[dev] = true;
    }
    return launch_pdl(attn_mma_kernel<D, kFp8>, grid, dim3(kThreads), smem, c.stream, p);
}

template <bool kFp8>
cudaError_t launch_d(const AttnCall& c, const Params& p, dim3 grid) {
    switch (c.d) {
        case 64: return launch_t<64, kFp8>(c, p, grid);
        case 128: return launch_t<128, kFp8>(c, p, grid);
        case 192: return launch_t<192, kFp8>(c, p, grid);
        case 256: return launch_t<256, kFp8>(c, p, grid);
        case 320: return launch_t<320, kFp8>(c, p, grid);
        case 384: return launch_t<384, kFp8>(c, p, grid);
        case 448: return launch_t<448, kFp8>(c, p, grid);
        case 512: return launch_t<512, kFp8>(c, p, grid);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t attn_mma_scratch_bytes(int64_t b, int64_t s, int h, int d, int topk) {
    const Geometry g = geometry(b * s, h, topk, kMaxSmCount);
    if (g.n_splits == 1) return 0;
    const size_t ntok = (size_t)(b * s);
    const size_t ml = align_up(ntok * g.n_splits * h * 2 * sizeof(float), 256);
    const size_t po = ntok * g.n_splits * h * (size_t)d * sizeof(float);
    return ml + po;
}

cudaError_t attn_mma_launch(const AttnCall& c) {
    const int64_t n_tokens = c.b * c.s;
    const Geometry g = geometry(n_tokens, c.h, c.topk, device_sm_count());
    Params p;
    p.q = reinterpret_cast<const __nv_bfloat16*>(c.q);
    p.kv = c.kv;
    p.kv_scale = c.kv_scale;
    p.sink = c.sink;
    p.idx = c.idx;
    p.o = reinterpret_cast<__nv_bfloat16*>(c.o);
    p.status = c.status;
    p.scale_log2 = c.softmax_scale * kLog2e;
    p.s_len = c.s;
    p.h = c.h;
    p.rows = c.rows;
    p.topk = c.topk;
    p.n_tiles = g.n_tiles;
    p.n_splits = g.n_splits;
    p.tiles_per_split = g.tiles_per_split;
    p.part_ml = nullptr;
    p.part_o = nullptr;
    if (g.n_splits > 1) {
        const size_t ml = align_up((size_t)n_tokens * g.n_splits * c.h * 2 * sizeof(float), 256);
        p.part_ml = reinterpret_cast<float*>(c.scratch);
        p.part_o = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(c.scratch) + ml);
    }
    if (n_tokens > 0x7FFFFFFF) return cudaErrorInvalidValue;
    dim3 grid((unsigned)n_tokens, g.n_splits, g.hblocks);
    cudaError_t e = c.kv_format == SA_KV_BF16 ? launch_d<false>(c, p, grid) : launch_d<true>(c, p, grid);
    if (e != cudaSuccess || g.n_splits == 1) return e;
    return attn_combine_launch(p.part_ml, p.part_o, c.sink, p.o, n_tokens, c.h, c.d, g.n_splits,
                               c.stream);
}

cudaError_t attn_combine_launch(const float* part_ml, const float* part_o, const float* sink,
                                void* o, int64_t n_tokens, int h, int d, int n_splits,
                                cudaStream_t stream) {
    if (n_tokens * h == 0) return cudaSuccess;
    // a programmatic dependent of the attention kernel just queued on the stream: its blocks can
    // be scheduled while that kernel drains, and wait for its partials
    return launch_pdl(attn_combine_kernel, dim3((unsigned)(n_tokens * h)), dim3((unsigned)(d / 4)), 0,
                      stream, part_ml, part_o, sink, reinterpret_cast<__nv_bfloat16*>(o), h, d,
                      n_splits);
}

}  // namespace sa
