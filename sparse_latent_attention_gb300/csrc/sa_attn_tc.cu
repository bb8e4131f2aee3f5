// sparse_attn on the 5th-generation tensor cores (tcgen05, accumulators in TMEM), head_dim 512.
//
// Source: "Module attn" API page (spark_model, deepseek_v41_ref/attn), Functions: sparse_attn
// and the precision paragraph; "DeepSeek V4.1" attention page, Attention.forward.
//
// Formulation.  All heads of a query token read the same gathered kv rows, and the rows serve as
// both keys and values.  Rows are gathered 64 at a time (a tile) into one of two shared-memory
// buffers, so that one tile is gathered while the tensor core works on the other:
//   S[64 heads x 64 rows]   = Q[64 x 512] . KV_tile^T                   (32 MMAs, M = 64)
//   O^T[512 x 64 heads]    += KV_tile^T[512 x 64] . P^T[64 rows x 64]    (4 M-chunks x 4 MMAs)
// With head_dim 512 an f32 accumulator of O for 64 heads needs 256 TMEM columns; as O^T (d on
// the lanes) it leaves the other 256 columns for two S buffers.  S has the heads as its M
// dimension, and an M = 64 accumulator puts head 16 w + i on TMEM lane 32 w + i: a softmax
// thread owns one head and half of the tile's columns (the other half sits with the thread 16
// lanes up), so the row maximum and sum need one shuffle and no exchange across warps.  The
// same swizzled shared-memory tile is the K-major B operand of the first product and the
// MN-major A operand of the second; P (bf16) is the K-major B operand of the second.  A
// running maximum is only raised (and O rescaled) when a new logit exceeds it by more than 2^8,
// so the rescale is rare.  The sink joins the denominator once, in the epilogue:
// o = O / (l + 2^(sink log2e - m)).
//
// Roles (persistent CTAs, one 64-head block of one query token per task, 480 threads):
//   warp 0      logits issue (one elected lane) and TMEM allocation
//   warp 14     P.V issue (one elected lane).  Two issuing warps, each blocked on its own
//               barriers, keep one product's bookkeeping off the other's path: the tensor pipe
//               takes the MMAs of both as they come, so the gather of one buffer, the logits of
//               its tile and the softmax and P.V of the other tile overlap
//   warp 1      Q loads (TMA, 128-byte swizzle) and an L2 prefetch of the next task's Q
//   warps 2-5   kv row gather: the 128 idx columns of a pair of tiles at a time, one per thread;
//               cp.async 16 B into the swizzled layout (fp8 rows are staged raw and widened in
//               place); rows already resident from the previous pair are kept -- see below
//   warps 6-9   softmax: S -> P (bf16, shared memory), running max and sum, O rescale
//   warps 10-13 epilogue: O^T -> o (bf16) or split partials; with fp8 kv, between epilogues,
//               they widen the second half (d 256-511) of every staged tile
// Every wait is bounded; a wait that gives up raises the timeout bit and every role unwinds.
//
// Row placement.  The order of the gathered rows inside a tile does not matter (the softmax and
// P.V sum over rows; masking uses each tile's set of claimed slots).  The 128 idx columns of a
// pair of tiles are placed together: when their valid rows have distinct residues mod 128, row
// j goes to slot j mod 128 (slots 0-63 in the pair's first tile, 64-127 in its second);
// otherwise column r of the pair goes to slot r.  A row already sitting in its slot from the
// previous pair is not copied again.  A CTA takes a contiguous block of tasks, so consecutive
// query tokens of a sliding window (127 of 128 rows shared) reload one row per token.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "sa_fp8.cuh"
#include "sa_internal.cuh"
#include "sa_tc.cuh"

namespace sa {
namespace {

using namespace tc;

constexpr int kD = 512;           // head_dim handled by this kernel
constexpr int kRows = 64;         // gathered rows per tile (N of the logits, K of P.V)
constexpr int kHeads = 64;        // heads per task (M of the logits, N of P.V)
constexpr int kChunks = 4;        // 128-d chunks of O^T (M of P.V)
constexpr int kProdWarps = 4;                       // kv gather warps (one pair column per thread)
constexpr int kProdThreads = 32 * kProdWarps;       // = the 128 columns of a pair of tiles
constexpr int kWarpSoftmax = 2 + kProdWarps;        // first softmax warp
constexpr int kWarpEpilogue = kWarpSoftmax + 4;     // first epilogue warp
constexpr int kWarpPv = kWarpEpilogue + 4;         // P.V issue
constexpr int kThreads = 32 * (kWarpPv + 1);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// TMEM columns: O^T chunks (4 x 64), the two S buffers (2 x 64)
constexpr uint32_t kColO = 0, kColS = 256;

// Shared-memory map (dynamic, 1024-byte aligned base)
// The two kv buffers are interleaved by 64-d block: [8 blocks of 64 d][buffer][64 rows][128 B]
constexpr uint32_t kBlkBytes = kRows * 128;       // 8 KB: one buffer's [64 rows x 64 d]
constexpr uint32_t kDBlkBytes = 2 * kBlkBytes;    // 16 KB: a 64-d block of both buffers
constexpr uint32_t kKvBytes = 8 * kDBlkBytes;     // 128 KB
constexpr uint32_t kQBlkBytes = kHeads * 128;     // 8 KB: [64 heads x 64 d] of Q
constexpr uint32_t kQBytes = kHeads * kD * 2;     // 64 KB: 8 blocks of [64 heads x 128 B]
constexpr uint32_t kPBytes = kHeads * kRows * 2;  // 8 KB: [64 heads x 128 B] per P buffer
constexpr uint32_t kOffKv = 0;
constexpr uint32_t kOffQ = kOffKv + kKvBytes;
constexpr uint32_t kOffP = kOffQ + kQBytes;
constexpr uint32_t kOffMisc = kOffP + 2 * kPBytes;

struct Misc {
    uint64_t q_full, q_empty;
    uint64_t kv_full[2], kv_empty[2];  // per kv buffer
    uint64_t staged[2];                // fp8: a tile's raw codes have landed (per kv buffer)
    uint64_t s_full[2], s_empty[2];    // per S buffer (TMEM)
    uint64_t p_full[2], p_empty[2];    // per P buffer (shared memory)
    uint64_t o_full, o_empty[kChunks];
    uint64_t stats_full[2], stats_empty[2];
    uint64_t sm_bar, pr_bar, done;
    uint32_t tmem_base;
    int abort;
    int need_corr[3];                  // per tile, in rotation: some head raised its maximum
    alignas(8) uint16_t vmask16[2][4];  // claimed slots of the tile in each kv buffer, 16 a piece
    uint32_t ring_bits[3][4];          // per pair, in rotation: residues mod 128 of valid rows
    int ring_count[3];                 // number of valid rows of a pair
    int64_t pair_seq[3];               // sequence whose rows a pair holds
    int row_id[2 * kRows];             // kv row held by each slot of the two buffers, -1 = none
    int2 copy_list[kProdWarps][2][32];  // per producer warp and tile: (kv row, slot) to copy
    int copy_n[kProdWarps][2];          // the lengths of those lists
    float alpha[2][kHeads];            // rescale factor of the tile, per tile parity
    float stats_m[2][kHeads];          // final max (0 when none) per task parity
    float stats_l[2][kHeads];          // final sum per task parity
    alignas(16) float inv[4][kHeads];  // epilogue: 1 / denominator, a table per epilogue warp
    float sink[kHeads];                // the sinks of the CTA's head block
    alignas(16) uint8_t fp8_sc[2 * kRows][16];  // e8m0 scales of the rows an fp8 tile widens
};
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
    const __nv_bfloat16* q;    // for the L2 prefetch of the next task's rows
    const __nv_bfloat16* kv;   // bf16 rows (bf16 kv)
    const uint8_t* kv8;        // e4m3 rows and their e8m0 scales (fp8 kv)
    const uint8_t* kv_scale;
    const float* sink;
    const int32_t* idx;
    __nv_bfloat16* o;
    float* part_ml;
    float* part_o;
    uint32_t* status;
    float scale_log2;
    int64_t s_len;
    int h;
    int hblocks;
    int64_t rows;
    int topk;
    int n_tiles;
    int n_splits;
    int tiles_per_split;  // even when the columns are split, so that pairs never straddle tasks
    int64_t n_units;      // (token, split) units; each is one task per head block
    const float* rope;    // inverse rotation of o's last rope_dim dims, or nullptr (see AttnCall)
    int rope_dim;
    int64_t rope_pos0;
};

struct Task {
    int64_t token, seq, pos;  // query token (flat), its sequence and position in it
    int hb, split, t0, t1;
};

// A CTA serves one head block, blockIdx.x % hblocks; the CTAs of one group (blockIdx.x /
// hblocks) serve the same (token, split) units at the same time, so every kv row a group gathers
// is read from HBM once and from L2 by the group's other CTAs.  A group takes a contiguous block
// of units [begin, end), so that consecutive query tokens of one sequence (which share most
// window rows) run back to back on the same SM.
__device__ __forceinline__ void task_range(const Params& p, int64_t& begin, int64_t& end) {
    const int64_t g = gridDim.x / p.hblocks, i = blockIdx.x / p.hblocks;
    const int64_t base = p.n_units / g, rem = p.n_units % g;
    begin = i * base + (i < rem ? i : rem);
    end = begin + base + (i < rem ? 1 : 0);
}

// The task of unit tau (token tau / n_splits, split tau % n_splits) for this CTA's head block.
__device__ __forceinline__ Task task_of(const Params& p, int64_t tau) {
    Task t;
    t.split = (int)(tau % p.n_splits);
    t.hb = (int)(blockIdx.x % p.hblocks);
    t.token = tau / p.n_splits;
    t.seq = t.token / p.s_len;
    t.pos = t.token - t.seq * p.s_len;
    t.t0 = t.split * p.tiles_per_split;
    t.t1 = min(p.n_tiles, t.t0 + p.tiles_per_split);
    if (t.t1 < t.t0) t.t1 = t.t0;
    return t;
}

// The task of the next unit (splits fastest, then tokens), without divisions.
__device__ __forceinline__ void task_step(const Params& p, Task& t) {
    if (++t.split == p.n_splits) {
        t.split = 0;
        ++t.token;
        if (++t.pos == p.s_len) {
            t.pos = 0;
            ++t.seq;
        }
    }
    t.t0 = t.split * p.tiles_per_split;
    t.t1 = min(p.n_tiles, t.t0 + p.tiles_per_split);
    if (t.t1 < t.t0) t.t1 = t.t0;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Three-input maximum and minimum, and f32 pairs (two lanes of one 64-bit register) for the packed
// FMA and add.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// The maximum (kMax) or minimum of 32 raw f32 words, as a tree of three-input operations.
template <bool kMax>
__device__ __forceinline__ float reduce32(const uint32_t (&r)[32]) {
    auto op3 = [](float a, float b, float c) { return kMax ? max3f(a, b, c) : min3f(a, b, c); };
    auto op2 = [](float a, float b) { return kMax ? fmaxf(a, b) : fminf(a, b); };
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i)
        a[i] = op3(__uint_as_float(r[3 * i]), __uint_as_float(r[3 * i + 1]), __uint_as_float(r[3 * i + 2]));
    a[10] = op2(__uint_as_float(r[30]), __uint_as_float(r[31]));
    const float b0 = op3(a[0], a[1], a[2]), b1 = op3(a[3], a[4], a[5]), b2 = op3(a[6], a[7], a[8]);
    return op3(b0, b1, op3(b2, a[9], a[10]));
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint32_t pack_bf16_2(uint64_t v) {
    float lo, hi;
    f2_split(v, lo, hi);
    return pack_bf16(lo, hi);
}

// mbar_wait by every lane of a converged warp, with a warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// Barrier among the 128 threads of one warpgroup, on an mbarrier so that it is bounded.
__device__ __forceinline__ bool wg_sync(uint32_t bar, uint32_t& phase, volatile int* abort) {
    mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase & 1, abort);
    ++phase;
    return ok;
}

// A 16-byte cp.async at constant offsets from a shared and a global base address.
template <uint32_t kSOff, int kGOff>
__device__ __forceinline__ void cp_async16_at(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%3], 16;" ::"r"(dst), "l"(src), "n"(kSOff),
                 "n"(kGOff));
}

// Byte offset, inside the kv buffers, of 16-byte unit u (of 64) of the row in slot ps (bit 6 =
// the buffer, bits 0-5 = the row of the tile): 64-d block u / 8, 128-byte swizzle.
__device__ __forceinline__ uint32_t kv_unit_off(int ps, int u) {
    return (uint32_t)(u >> 3) * kDBlkBytes + (uint32_t)(ps >> 6) * kBlkBytes + (uint32_t)(ps & 63) * 128 +
           ((((uint32_t)u & 7) ^ ((uint32_t)ps & 7)) << 4);
}

// Widens 128-d chunks c0 .. c1 - 1 of the fp8 rows a warp lists, in place: the e4m3 codes of chunk
// c sit raw in 64-d block 2c + 1 of the row's slot and become bf16 in blocks 2c and 2c + 1 (exact:
// see sa_fp8.cuh).  Lane l moves 16-code unit l % 8 (`unit`) of list entries l / 8 + 4 i (ent[i],
// x < 0 = none); the row's 16 e8m0 scales are in fp8_sc.
__device__ __forceinline__ void widen_fp8(uint32_t s_kv, const Misc& M, const int2 (&ent)[8], int unit,
                                          int c0, int c1) {
    // Per entry, once: the slot's offset inside a 64-d block (buffer and row) and the byte offset
    // of this lane's first bf16 unit in it.  Unit u = 16 c + 2 unit of the row sits in block
    // u / 8 = 2 c + unit / 4 at swizzled position (u % 8) ^ (slot % 8), u % 8 = 2 (unit % 4); unit
    // u + 1 is the same address with bit 4 flipped (u is even).
    uint32_t rb[8], xo[8];
    const uint32_t uo = (uint32_t)(2 * (unit & 3)) << 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t r = (uint32_t)ent[i].y;
        rb[i] = (r >> 6) * kBlkBytes + (r & 63) * 128;
        xo[i] = rb[i] + (uo ^ ((r & 7) << 4));
    }
    const uint8_t* sc_base = &M.fp8_sc[0][0] + (unit >> 1);
#pragma unroll 1
    for (int cw = c0; cw < c1; ++cw) {
        const uint32_t code_at = s_kv + (2 * cw + 1) * kDBlkBytes + unit * 16;
        const uint32_t out_at = s_kv + (2 * cw + (unit >> 2)) * kDBlkBytes;
        // entries in two groups of four; a row's 8 lanes read all its codes before any writes
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            uint4 code[4];
            float sc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int2 en = ent[4 * g + i];
                if (en.x < 0) break;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(code[i].x), "=r"(code[i].y), "=r"(code[i].z), "=r"(code[i].w)
                             : "r"(code_at + rb[4 * g + i])
                             : "memory");
                sc[i] = fp8::e8m0_to_f32(sc_base[en.y * 16 + 4 * cw]);
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int2 en = ent[4 * g + i];
                if (en.x < 0) break;
                uint4 lo, hi;
                fp8::dequant16(code[i], sc[i], lo, hi);
                const uint32_t at = out_at + xo[4 * g + i];
                st_shared_v4(at, lo.x, lo.y, lo.z, lo.w);
                st_shared_v4(at ^ 16u, hi.x, hi.y, hi.z, hi.w);
            }
        }
    }
}

// kRope: the inverse rotation of o's rope dims is fused into the epilogue (a separate
// instantiation, so that the plain kernel carries none of its code)
template <bool kFp8, bool kRope>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap q_map, Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    Misc& M = *reinterpret_cast<Misc*>(smem + kOffMisc);
    const uint32_t s_kv = smem_addr(smem + kOffKv);
    const uint32_t s_q = smem_addr(smem + kOffQ);
    const uint32_t s_p = smem_addr(smem + kOffP);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &M.abort;
    const int hb = (int)(blockIdx.x % p.hblocks);
    pdl_trigger();  // the next launch on the stream may be scheduled from now on

    if (tid == 0) {
        mbar_init(smem_addr(&M.q_full), 1);
        mbar_init(smem_addr(&M.q_empty), 1);
        for (int b = 0; b < 2; ++b) {
            // fp8: the epilogue warps widen half of every tile, so they arrive too
            mbar_init(smem_addr(&M.kv_full[b]), kFp8 ? kProdThreads + 128 : kProdThreads);
            mbar_init(smem_addr(&M.staged[b]), kProdThreads);
            mbar_init(smem_addr(&M.kv_empty[b]), 1);
            mbar_init(smem_addr(&M.s_full[b]), 1);
            mbar_init(smem_addr(&M.s_empty[b]), 128);
            mbar_init(smem_addr(&M.p_full[b]), 128);
            mbar_init(smem_addr(&M.p_empty[b]), 1);
            mbar_init(smem_addr(&M.stats_full[b]), 128);
            mbar_init(smem_addr(&M.stats_empty[b]), 128);
        }
        mbar_init(smem_addr(&M.o_full), 1);
        for (int c = 0; c < kChunks; ++c) mbar_init(smem_addr(&M.o_empty[c]), 128);
        mbar_init(smem_addr(&M.sm_bar), 128);
        mbar_init(smem_addr(&M.pr_bar), kProdThreads);
        mbar_init(smem_addr(&M.done), 2);
        M.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(&M.tmem_base), 512);
        tmem_relinquish();
    }
    // every slot starts as a finite (zero) row that no tile claims
    for (int i = tid; i < 2 * kRows; i += kThreads) M.row_id[i] = -1;
    if (tid < 12) (&M.ring_bits[0][0])[tid] = 0;
    if (tid < 3) {
        M.ring_count[tid] = 0;
        M.pair_seq[tid] = -1;
        M.need_corr[tid] = 0;
    }
    for (uint32_t i = tid; i < kKvBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kOffKv)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1 && lane == 0) tma_prefetch_desc(&q_map);
    // the set-up above touches no global memory; everything below may read what the work queued
    // before this launch writes
    pdl_wait();
    for (int i = tid; i < kHeads; i += kThreads)
        M.sink[i] = hb * kHeads + i < p.h ? p.sink[hb * kHeads + i] : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = M.tmem_base;
    int64_t tb, te;
    task_range(p, tb, te);

    if (warp == 0) {
        // ------------------------------------------------------------------ logits issue
        // The whole warp runs this loop (descriptors stay in uniform registers); each MMA and
        // commit is issued by one elected lane, and every lane waits on the barriers.  A wait's
        // result is made warp-uniform so that a time-out cannot split the warp.
        constexpr uint32_t id_s = idesc_bf16_f32(kHeads, kRows, false, false);
        const uint64_t a_s0 = smem_desc_sw128(s_q, 16, 1024);   // Q, K-major
        const uint64_t b_s0 = smem_desc_sw128(s_kv, 16, 1024);  // tile rows, K-major
        bool ok = true;
        int64_t k = 0;
        uint32_t T = 0;
        Task t = task_of(p, tb);
        for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
            if (p.n_tiles == 0) {  // no idx columns: keep the Q phases in step
                ok = warp_wait(smem_addr(&M.q_full), (uint32_t)(k & 1), abort);
                mma_commit_elect(smem_addr(&M.q_empty));
                continue;
            }
            for (int ti = t.t0; ti < t.t1 && ok; ++ti, ++T) {
                const uint32_t b = T & 1, use = T >> 1;
                ok = warp_wait(smem_addr(&M.kv_full[b]), use & 1, abort) &&
                     warp_wait(smem_addr(&M.s_empty[b]), (use & 1) ^ 1, abort) &&
                     (ti != t.t0 || warp_wait(smem_addr(&M.q_full), (uint32_t)(k & 1), abort));
                if (!ok) break;
                tc_fence_after();
                // S = Q . tile^T: K step 4 kb + kq (16 of 512) = block kb of Q and of the tile,
                // 32 B per step inside a 128-byte row
                const uint32_t s_col = tmem + kColS + 64 * b;
                const uint32_t ahi = (uint32_t)(a_s0 >> 32), bhi = (uint32_t)(b_s0 >> 32);
                uint32_t alo = (uint32_t)a_s0, blo = (uint32_t)b_s0 + b * (kBlkBytes >> 4);
#pragma unroll 1
                for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq)
                        mma_lohi_elect(s_col, alo + kq * 2, ahi, blo + kq * 2, bhi, id_s, (kb | kq) != 0);
                    alo += kQBlkBytes >> 4;
                    blo += kDBlkBytes >> 4;
                }
                if (ti == t.t1 - 1) mma_commit_elect(smem_addr(&M.q_empty));
                mma_commit_elect(smem_addr(&M.s_full[b]));
            }
        }
        // let every issued MMA finish before the accumulators are released
        mma_commit_elect(smem_addr(&M.done));
        warp_wait(smem_addr(&M.done), 0, abort);
    } else if (warp == kWarpPv) {
        // ------------------------------------------------------------------ P.V issue
        constexpr uint32_t id_o = idesc_bf16_f32(128, kHeads, true, false);
        const uint64_t a_o0 = smem_desc_sw128(s_kv, kDBlkBytes, 1024);  // tile^T, MN-major
        const uint64_t b_o0 = smem_desc_sw128(s_p, 16, 1024);           // P, K-major
        bool ok = true;
        int64_t k = 0;
        uint32_t T = 0;
        Task t = task_of(p, tb);
        for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
            if (p.n_tiles == 0) {  // no idx columns: keep the O phases in step
                for (int c = 0; c < kChunks && ok; ++c)
                    ok = warp_wait(smem_addr(&M.o_empty[c]), (uint32_t)(k & 1) ^ 1, abort);
                mma_commit_elect(smem_addr(&M.o_full));
                continue;
            }
            for (int ti = t.t0; ti < t.t1 && ok; ++ti, ++T) {
                // O^T += KV^T . P^T for tile T (T & 1 = its kv and P buffer)
                const uint32_t b = T & 1;
                const bool first = ti == t.t0;
                if (!(ok = warp_wait(smem_addr(&M.p_full[b]), (T >> 1) & 1, abort))) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kChunks && ok; ++c) {
                    if (first) {  // the epilogue has read this chunk of the last task's O
                        if (!(ok = warp_wait(smem_addr(&M.o_empty[c]), (uint32_t)(k & 1) ^ 1, abort))) break;
                        tc_fence_after();
                    }
                    // K step ks = rows 16 ks .. 16 ks + 15 (2 KB of the two 64-d blocks of chunk c)
                    const uint32_t alo = (uint32_t)a_o0 + b * (kBlkBytes >> 4) + c * (2 * kDBlkBytes >> 4);
                    const uint32_t blo = (uint32_t)b_o0 + b * (kPBytes >> 4);
                    const uint32_t ahi = (uint32_t)(a_o0 >> 32), bhi = (uint32_t)(b_o0 >> 32);
#pragma unroll
                    for (int ks = 0; ks < kRows / 16; ++ks)
                        mma_lohi_elect(tmem + kColO + 64 * c, alo + ks * (16 * 128 >> 4), ahi, blo + ks * 2,
                                       bhi, id_o, !(first && ks == 0));
                }
                if (!ok) break;
                mma_commit_elect(smem_addr(&M.kv_empty[b]));  // the tile's rows are read
                mma_commit_elect(smem_addr(&M.p_empty[b]));
                if (ti == t.t1 - 1) mma_commit_elect(smem_addr(&M.o_full));
            }
        }
        // (done completes once both issuing warps' MMAs have)
        mma_commit_elect(smem_addr(&M.done));
        warp_wait(smem_addr(&M.done), 0, abort);
    } else if (warp == 1) {
        // ------------------------------------------------------------------ Q loads (TMA)
        if (lane == 0) {
            int64_t k = 0;
            bool ok = true;
            Task t = task_of(p, tb);
            const int hc = min(kHeads, p.h - hb * kHeads);
            for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
                const int32_t y = (int32_t)(t.token * p.h + (int64_t)t.hb * kHeads);
                ok = mbar_wait(smem_addr(&M.q_empty), (uint32_t)(k & 1) ^ 1, abort);
                if (!ok) break;
                const uint32_t bar = smem_addr(&M.q_full);
                mbar_arrive_expect_tx(bar, kQBytes);
#pragma unroll 1
                for (int c = 0; c < 8; ++c)  // 8 boxes of [64 heads x 64 d], 128-byte swizzle
                    tma_load_2d(s_q + c * 8192, &q_map, 64 * c, y, bar);
                // the next task's rows (when it is another token) into L2 meanwhile
                if (tau + 1 < te && t.split == p.n_splits - 1) {
                    const __nv_bfloat16* qn = p.q + ((t.token + 1) * p.h + (int64_t)hb * kHeads) * kD;
#pragma unroll 1
                    for (int i = 0; i < hc; i += 8)
                        prefetch_l2(qn + (int64_t)i * kD, (uint32_t)(min(8, hc - i) * kD * 2));
                }
            }
            // after a failed wait, let the last Q load land before the CTA exits
            if (!ok && k > 0) mbar_drain(smem_addr(&M.q_full), (uint32_t)((k - 1) & 1));
        }
        __syncwarp();
    } else if (warp < kWarpSoftmax) {
        // ------------------------------------------------------------------ kv gather
        // Each thread resolves one of the 128 columns of a pair of tiles; every warp lists the
        // rows it copies into each of the pair's tiles, and copies a tile's rows (cp.async, one
        // commit group) as soon as the P.V two tiles back has released that kv buffer.  Warp w
        // resolves columns 16 w .. 16 w + 15 of each tile (lanes 0-15 the first tile, 16-31 the
        // second), so that every warp has rows to copy into both tiles.
        const int pw = warp - 2;  // producer warp 0 .. kProdWarps - 1
        const int pt = (lane >> 4) * kRows + 16 * pw + (lane & 15);  // its pair column (and slot)
        uint32_t T = 0, pr_phase = 0, g3 = 0;
        bool ok = true;
        Task t = task_of(p, tb);
        for (int64_t tau = tb; tau < te && ok; ++tau, task_step(p, t)) {
            const int64_t bi = t.seq;
            const int32_t* idx_tok = p.idx + t.token * (int64_t)p.topk;
            const int colend = min(p.topk, t.t1 * kRows);
            for (int ti = t.t0; ti < t.t1 && ok; ti += 2) {
                const int nt = min(2, t.t1 - ti);  // tiles of this pair
                const uint32_t gprev = g3 == 0 ? 2 : g3 - 1, gnext = g3 == 2 ? 0 : g3 + 1;
                const int col = ti * kRows + pt;
                int j = col < colend ? __ldg(idx_tok + col) : -1;
                if (j < -1 || j >= p.rows) {
                    atomicOr(p.status, kStatusBadIndex);
                    j = -1;
                }
                // ring placement (slot = j mod 128) when the valid rows' residues are distinct
                // (the per-pair records rotate over three entries; the previous pair's is cleared
                // after this pair's barrier, when nobody reads it any more, and is next written
                // by the pair after the next, after the next pair's barrier.  The next pair's
                // own entry must not be touched here: a fast thread may be filling it already.)
                {
                    // per warp: the residue bits of each of the four words or-reduced, and the count
                    // of valid rows, added by one lane
                    const uint32_t w = (uint32_t)(j & 127) >> 5, bit = j >= 0 ? 1u << (j & 31) : 0u;
                    uint32_t wb[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) wb[q] = __reduce_or_sync(0xffffffffu, w == (uint32_t)q ? bit : 0u);
                    const uint32_t nv = (uint32_t)__popc(__ballot_sync(0xffffffffu, j >= 0));
                    if (lane == 0) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (wb[q]) atomicOr(&M.ring_bits[g3][q], wb[q]);
                        if (nv) atomicAdd(&M.ring_count[g3], (int)nv);
                    }
                }
                if (pt == 0) M.pair_seq[g3] = bi;
                if (!(ok = wg_sync(smem_addr(&M.pr_bar), pr_phase, abort))) break;
                // a slot's row can be kept only if it belongs to this same sequence
                const bool same_seq = M.pair_seq[gprev] == bi;
                const bool ring = nt == 2 &&
                                  __popc(M.ring_bits[g3][0]) + __popc(M.ring_bits[g3][1]) +
                                          __popc(M.ring_bits[g3][2]) + __popc(M.ring_bits[g3][3]) ==
                                      M.ring_count[g3];
                // this thread's own slot is empty unless a row claims it
                const bool claimed = ring ? ((M.ring_bits[g3][pt >> 5] >> (pt & 31)) & 1) != 0 : j >= 0;
                const int slot = ring ? (j & 127) : pt;
                // slot s of the pair is row s % 64 of the kv buffer of tile T + s / 64 (every
                // slot of both buffers is rewritten, so a one-tile pair forgets the other buffer)
                const int ps_own = (int)((((T + (uint32_t)(pt >> 6)) & 1) << 6) | (uint32_t)(pt & 63));
                const int ps = (int)((((T + (uint32_t)(slot >> 6)) & 1) << 6) | (uint32_t)(slot & 63));
                if (!claimed) M.row_id[ps_own] = -1;
                const bool copy = j >= 0 && !(same_seq && M.row_id[ps] == j);
                if (j >= 0) M.row_id[ps] = j;
                if (pt == 0) {
                    M.ring_bits[gprev][0] = M.ring_bits[gprev][1] = 0;
                    M.ring_bits[gprev][2] = M.ring_bits[gprev][3] = 0;
                    M.ring_count[gprev] = 0;
                }
                g3 = gnext;
                // the claimed slots (16 of each tile: slots 16 pw .. 16 pw + 15 in the first
                // tile's half of the ballot, the second tile's in the other) and the rows it copies
                // into each tile, compacted into lists (ballot prefix counts)
                const uint32_t m_claim = __ballot_sync(0xFFFFFFFFu, claimed);
                const int half = slot >> 6;
                const uint32_t mh0 = __ballot_sync(0xFFFFFFFFu, copy && half == 0);
                const uint32_t mh1 = __ballot_sync(0xFFFFFFFFu, copy && half == 1);
                if constexpr (kFp8) {
                    // the epilogue warps read the previous pair's lists until they have widened
                    // its tiles (their arrival completes a tile's kv_full)
                    if (T > 0 && !(ok = mbar_wait(smem_addr(&M.kv_full[(T - 1) & 1]), ((T - 1) >> 1) & 1, abort)))
                        break;
                    if (T > 1 && !(ok = mbar_wait(smem_addr(&M.kv_full[(T - 2) & 1]), ((T - 2) >> 1) & 1, abort)))
                        break;
                    if (lane == 0) {
                        M.copy_n[pw][0] = __popc(mh0);
                        M.copy_n[pw][1] = __popc(mh1);
                    }
                }
                if (copy) {
                    const uint32_t mh = half ? mh1 : mh0;
                    M.copy_list[pw][half][__popc(mh & ((1u << lane) - 1u))] = make_int2(j, ps);
                    // the buffers are usually still in use: pull the new rows into L2 now, so
                    // that the copies issued once a buffer is released hit L2
                    if constexpr (kFp8) {
                        prefetch_l2(p.kv8 + (bi * p.rows + j) * (int64_t)kD, kD);
                        prefetch_l2(p.kv_scale + (bi * p.rows + j) * (int64_t)(kD / 32), kD / 32);
                    } else {
                        prefetch_l2(p.kv + (bi * p.rows + j) * (int64_t)kD, kD * 2);
                    }
                }
                __syncwarp();
                if constexpr (kFp8) {
                    // e4m3 rows: chunk c's 128 codes of each listed row are staged raw in block
                    // 2c + 1 of the row's slot (dead until the row is written), then widened in
                    // place to bf16 in blocks 2c and 2c + 1.  Lane l moves 16-code unit l % 8 of
                    // rows l / 8 + 4 i.
                    const uint8_t* kvb8 = p.kv8 + bi * p.rows * (int64_t)kD;
                    const uint8_t* scb = p.kv_scale + bi * p.rows * (int64_t)(kD / 32);
                    const int unit = lane & 7;
                    // stage each tile as soon as its buffer is released (one commit group per
                    // tile), then widen them in order: the first tile's widening overlaps the
                    // second's copies
                    // (a tile's list entries (lane / 8) + 4 i are read from the list where needed)
                    auto load_ent = [&](int hx, int2 (&ent)[8]) {
                        const int ncopy = __popc(hx ? mh1 : mh0);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int e = (lane >> 3) + 4 * i;
                            ent[i] = e < ncopy ? M.copy_list[pw][hx][e] : make_int2(-1, 0);
                        }
                    };
#pragma unroll
                    for (int hx = 0; hx < 2; ++hx) {
                        if (hx >= nt || !ok) break;
                        const uint32_t Tx = T + hx, b = Tx & 1;
                        const int ncopy = __popc(hx ? mh1 : mh0);
                        int2 ent8[8];
                        load_ent(hx, ent8);
                        if (!(ok = mbar_wait(smem_addr(&M.kv_empty[b]), ((Tx >> 1) & 1) ^ 1, abort))) break;
                        M.vmask16[b][pw] = (uint16_t)(hx ? m_claim >> 16 : m_claim);
                        if (lane < ncopy) {  // the row's 16 scales
                            const int2 en = M.copy_list[pw][hx][lane];
                            cp_async16(smem_addr(&M.fp8_sc[en.y][0]), scb + (int64_t)en.x * (kD / 32), 16u);
                        }
                        // per row one shared and one global base, chunk c at constant offsets
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (ent8[i].x < 0) break;
                            const uint32_t r = (uint32_t)ent8[i].y;
                            const uint32_t sb =
                                s_kv + kDBlkBytes + (r >> 6) * kBlkBytes + (r & 63) * 128 + unit * 16;
                            const uint8_t* gb = kvb8 + (int64_t)ent8[i].x * kD + unit * 16;
                            cp_async16_at<0, 0>(sb, gb);
                            cp_async16_at<2 * kDBlkBytes, 128>(sb, gb);
                            cp_async16_at<4 * kDBlkBytes, 256>(sb, gb);
                            cp_async16_at<6 * kDBlkBytes, 384>(sb, gb);
                        }
                        cp_async_commit();
                    }
#pragma unroll
                    for (int hx = 0; hx < 2; ++hx) {
                        if (hx >= nt || !ok) break;
                        const uint32_t b = (T + hx) & 1;
                        if (hx == 0 && nt == 2) cp_async_wait<1>();
                        else cp_async_wait<0>();
                        __syncwarp();  // every lane's staged codes are visible to the warp
                        // the epilogue warps widen chunks 2 and 3 of the tile, this warp 0 and 1
                        mbar_arrive(smem_addr(&M.staged[b]));
                        int2 ent8[8];
                        load_ent(hx, ent8);
                        widen_fp8(s_kv, M, ent8, unit, 0, 2);
                        fence_proxy_async_smem();
                        mbar_arrive(smem_addr(&M.kv_full[b]));
                    }
                    T += nt;
                    continue;
                }
                const __nv_bfloat16* kvb = p.kv + bi * p.rows * (int64_t)kD;
                // a tile with at most two new rows (e.g. the next token of a sliding window):
                // load them into registers now, while the buffers are still in use; lane l
                // holds 16-byte units l and 32 + l of a row
                uint4 v[2][2][2];
                int2 ent_r[2][2];
#pragma unroll
                for (int hx = 0; hx < 2; ++hx) {
                    const int n = __popc(hx ? mh1 : mh0);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        ent_r[hx][e] = (hx < nt && n <= 2 && e < n) ? M.copy_list[pw][hx][e] : make_int2(-1, 0);
                        if (ent_r[hx][e].x >= 0) {
                            const uint4* src = reinterpret_cast<const uint4*>(kvb + (int64_t)ent_r[hx][e].x * kD);
                            v[hx][e][0] = __ldg(src + lane);
                            v[hx][e][1] = __ldg(src + 32 + lane);
                        }
                    }
                }
#pragma unroll
                for (int hx = 0; hx < 2; ++hx) {
                    if (hx >= nt || !ok) break;
                    const uint32_t Tx = T + hx, b = Tx & 1;
                    const int ncopy = __popc(hx ? mh1 : mh0);
                    if (!(ok = mbar_wait(smem_addr(&M.kv_empty[b]), ((Tx >> 1) & 1) ^ 1, abort))) break;
                    M.vmask16[b][pw] = (uint16_t)(hx ? m_claim >> 16 : m_claim);
                    if (ncopy <= 2) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if (ent_r[hx][e].x < 0) continue;
                            const int r = ent_r[hx][e].y;
                            const uint4 w0 = v[hx][e][0], w1 = v[hx][e][1];
                            st_shared_v4(s_kv + kv_unit_off(r, lane), w0.x, w0.y, w0.z, w0.w);
                            st_shared_v4(s_kv + kv_unit_off(r, 32 + lane), w1.x, w1.y, w1.z, w1.w);
                        }
                    } else {
                        // list entries lane / 16 + 2 i (two rows per instruction); lane % 16 moves
                        // 16-byte unit u = 16 c + lane % 16 of quarter c of the row.  One shared and
                        // one global base address per row, the quarters at constant offsets: unit u
                        // sits in 64-d block u / 8 = 2 c + (lane % 16) / 8 at swizzled position
                        // (lane % 8) ^ (slot % 8), i.e. bits 4-6 of the 1024-byte aligned base
                        // (the instruction count of this loop bounds the gather)
                        const uint32_t s_lane = s_kv + (uint32_t)((lane & 15) >> 3) * kDBlkBytes +
                                                ((uint32_t)lane & 7) * 16;
                        const char* g_lane = reinterpret_cast<const char*>(kvb) + (lane & 15) * 16;
#pragma unroll 1
                        for (int e = lane >> 4; e < ncopy; e += 2) {
                            const int2 en = M.copy_list[pw][hx][e];
                            const uint32_t ps = (uint32_t)en.y;
                            const uint32_t sb = (s_lane ^ ((ps & 7) << 4)) + (ps >> 6) * kBlkBytes +
                                                (ps & 63) * 128;
                            const char* gb = g_lane + (int64_t)en.x * (kD * 2);
                            cp_async16_at<0, 0>(sb, gb);
                            cp_async16_at<2 * kDBlkBytes, 256>(sb, gb);
                            cp_async16_at<4 * kDBlkBytes, 512>(sb, gb);
                            cp_async16_at<6 * kDBlkBytes, 768>(sb, gb);
                        }
                        cp_async_commit();
                        cp_async_wait<0>();
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(smem_addr(&M.kv_full[b]));
                }
                T += nt;
            }
        }
        cp_async_wait<0>();
    } else if (warp < kWarpEpilogue) {
        // ------------------------------------------------------------------ softmax
        // Per tile: the head's maximum over the tile -> running max m (raised only past the
        // threshold), p = 2^(x - m) written as the head's P row, and the running sum
        // l = alpha l + sum p; O is rescaled (rarely) before the tile's P.V.
        const int q4 = warp & 3;
        const int hf = lane >> 4;                // which 32 of the tile's 64 columns
        const int hh = 16 * q4 + (lane & 15);    // the head (within the block) of this thread
        const int st = tid - 32 * kWarpSoftmax;  // 0 .. 127
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint32_t T = 0, sm_phase = 0, c3 = 0;
        int64_t k = 0;
        bool ok = true;
        Task t = task_of(p, tb);
        for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
            const int kpar = (int)(k & 1);
            float m = -INFINITY, mu = 0.f, l = 0.f;
            for (int ti = t.t0; ti < t.t1 && ok; ++ti, ++T) {
                const uint32_t b = T & 1, use = T >> 1;
                const bool first = ti == t.t0;
                ok = mbar_wait(smem_addr(&M.kv_full[b]), use & 1, abort);  // the tile's slot set
                if (ok) ok = mbar_wait(smem_addr(&M.s_full[b]), use & 1, abort);
                if (!ok) break;
                tc_fence_after();
                uint32_t r[32];
                tmem_ld_16x32bx2_x32<32>(tmem + lane_base + kColS + 64 * b, r);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(smem_addr(&M.s_empty[b]));
                // scaled logits (log2 units); an unclaimed slot's become -inf
                const uint32_t vm = reinterpret_cast<const uint32_t*>(M.vmask16[b])[hf];
                // every one of the 32 slots claimed (the usual case): the maximum of the raw logits
                // (the minimum for a negative scale) times the scale, and p = 2^(s scale - m) in one
                // FMA; otherwise the scaled logits replace the raw ones, -inf where unclaimed
                const bool full = vm == 0xFFFFFFFFu;
                float mt, sc = p.scale_log2;
                if (full) {
                    mt = (sc >= 0.f ? reduce32<true>(r) : reduce32<false>(r)) * sc;
                } else {
                    mt = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float xi = ((vm >> i) & 1u) ? __uint_as_float(r[i]) * sc : -INFINITY;
                        r[i] = __float_as_uint(xi);
                        mt = fmaxf(mt, xi);
                    }
                    sc = 1.f;
                }
                mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 16));
                float al = 1.f, mn = mt;
                if (!first) {
                    mn = mt > m + kRescaleThreshold ? mt : m;
                    if (mn != m) al = fast_exp2(m - mn);  // 0 when m = -inf (nothing summed yet)
                }
                if (hf == 0) {
                    M.alpha[b][hh] = al;
                    if (!first && mn != m) M.need_corr[c3] = 1;
                }
                m = mn;
                mu = mn == -INFINITY ? 0.f : mn;
                // p = 2^(x - m): this thread's 32 columns are 16-byte units 4 hf .. 4 hf + 3 of
                // the head's 128-byte P row (swizzled like every K-major operand)
                // (pairs of columns through the packed FMA and add; two running pair sums)
                uint32_t pk[16];
                const uint64_t sc2 = f2(sc, sc), nm2 = f2(-mu, -mu);
                uint64_t acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    const uint64_t s2 = f2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    f2_split(ffma2(s2, sc2, nm2), x0, x1);
                    const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
                    acc[i & 1] = fadd2(acc[i & 1], f2(e0, e1));
                    pk[i] = pack_bf16(e0, e1);
                }
                float a0, a1, a2, a3;
                f2_split(acc[0], a0, a1);
                f2_split(acc[1], a2, a3);
                const float ps = (a0 + a1) + (a2 + a3);
                l = first ? ps : fmaf(al, l, ps);
                // the P buffer is free once the P.V two tiles back has completed
                if (!(ok = mbar_wait(smem_addr(&M.p_empty[b]), (use & 1) ^ 1, abort))) break;
                const uint32_t prow = s_p + b * kPBytes + (uint32_t)hh * 128;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    st_shared_v4(prow + ((((uint32_t)(4 * hf + u)) ^ ((uint32_t)hh & 7)) << 4), pk[4 * u],
                                 pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                if (!(ok = wg_sync(smem_addr(&M.sm_bar), sm_phase, abort))) break;
                const bool corr = !first && M.need_corr[c3] != 0;
                // (clear the entry of the tile after next: its writers are past the next barrier)
                if (st == 0) M.need_corr[c3 == 0 ? 2 : c3 - 1] = 0;
                c3 = c3 == 2 ? 0 : c3 + 1;
                if (corr) {
                    // O must hold the previous tile's P.V before it is rescaled
                    const uint32_t pb = (T - 1) & 1;
                    if (!(ok = mbar_wait(smem_addr(&M.p_empty[pb]), ((T - 1) >> 1) & 1, abort))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 2 * kChunks; ++c) {  // O^T in 8 blocks of 32 heads
                        uint32_t o[32];
                        const uint32_t ta = tmem + lane_base + kColO + 32 * c;
                        tmem_ld_32x32b_x32(ta, o);
                        tmem_wait_ld();
                        const float* alc = &M.alpha[b][32 * (c & 1)];
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alc[i]);
                        tmem_st_32x32b_x32(ta, o);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_addr(&M.p_full[b]));
            }
            if (!ok) break;
            // the task's statistics, once the epilogue has read those of two tasks back
            if (!(ok = mbar_wait(smem_addr(&M.stats_empty[kpar]), (uint32_t)((k >> 1) & 1) ^ 1, abort))) break;
            l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
            if (hf == 0) {
                M.stats_m[kpar][hh] = t.t1 > t.t0 ? mu : 0.f;
                M.stats_l[kpar][hh] = t.t1 > t.t0 ? l : 0.f;
            }
            mbar_arrive(smem_addr(&M.stats_full[kpar]));
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        // O^T chunk c (128 d x 64 heads) leaves TMEM at once (the MMA may refill it), is scaled by
        // 1 / denominator and packed to bf16.  Each warp holds 32 d of every head; neighbouring
        // lanes trade halves so that each lane holds one head's pair of d, and each store
        // instruction writes two heads' 64 contiguous bytes of o (a staged TMA store was measured
        // slower on a sliding window, where the epilogue follows every second tile).  Every
        // thread passes every barrier of a task, even after a failed wait, so the warpgroup's
        // barriers never split.
        const int q4 = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const int odd = lane & 1;
        const uint32_t sel = odd ? 0x3276u : 0x5410u;
        int64_t k = 0;
        bool ok = true;
        Task t = task_of(p, tb);
        // fp8: the next tile whose chunks 2 and 3 this warpgroup widens (warp q4 takes the rows
        // producer warp q4 listed)
        int64_t wtau = p.n_tiles > 0 ? tb : te;
        int wsplit = t.split, wt0 = t.t0, wt1 = t.t1, wti = t.t0;
        uint32_t wT = 0;
        for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
            const int kpar = (int)(k & 1);
            const int h0 = t.hb * kHeads;
            const int hc = min(kHeads, p.h - h0);
            // the cos / sin of this thread's pair in the last O chunk (where the rope dims sit),
            // loaded now so that the load's latency hides behind the wait for O
            float2 rope_last = make_float2(1.f, 0.f);
            if constexpr (kRope) {
                const int dd = 128 * (kChunks - 1) + 32 * q4 + lane, first = kD - p.rope_dim;
                if (dd >= first)
                    rope_last = reinterpret_cast<const float2*>(
                        p.rope)[(p.rope_pos0 + t.pos) * (p.rope_dim / 2) + ((dd - first) >> 1)];
            }
            if constexpr (kFp8) {
                // widen every tile the producers have staged until this task's O is complete
                // (its last tile needs this warpgroup's widening first); the poll is bounded
                uint32_t idle = 0;
                while (true) {
                    if (wtau < te &&
                        __all_sync(0xffffffffu, mbar_test_wait(smem_addr(&M.staged[wT & 1]), (wT >> 1) & 1))) {
                        const int hx = (wti - wt0) & 1;
                        const int ncopy = M.copy_n[q4][hx];
                        int2 ent8[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int e = (lane >> 3) + 4 * i;
                            ent8[i] = e < ncopy ? M.copy_list[q4][hx][e] : make_int2(-1, 0);
                        }
                        widen_fp8(s_kv, M, ent8, lane & 7, 2, 4);
                        fence_proxy_async_smem();
                        mbar_arrive(smem_addr(&M.kv_full[wT & 1]));
                        ++wT;
                        if (++wti == wt1) {  // the next unit's tiles (splits fastest, as task_step)
                            ++wtau;
                            if (++wsplit == p.n_splits) wsplit = 0;
                            wt0 = wsplit * p.tiles_per_split;
                            wt1 = min(p.n_tiles, wt0 + p.tiles_per_split);
                            wti = wt0;
                        }
                        idle = 0;
                        continue;
                    }
                    if (__all_sync(0xffffffffu, mbar_test_wait(smem_addr(&M.o_full), (uint32_t)kpar))) break;
                    if (__any_sync(0xffffffffu, *abort != 0) || ++idle > (1u << 22)) {
                        *abort = 1;
                        ok = false;
                        break;
                    }
                    if (idle > 64) __nanosleep(32);
                }
            }
            ok = ok && mbar_wait(smem_addr(&M.o_full), (uint32_t)kpar, abort);
            if (ok) ok = mbar_wait(smem_addr(&M.stats_full[kpar]), (uint32_t)((k >> 1) & 1), abort);
            tc_fence_after();
            const bool split = p.n_splits > 1;
            const int64_t pbase = (t.token * p.n_splits + t.split) * (int64_t)p.h + h0;
            // the denominators: lane l finishes heads l and l + 32 into the warp's own table
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                const int h = lane + 32 * hq;
                const float l = M.stats_l[kpar][h], mu = M.stats_m[kpar][h];
                float inv = 0.f;
                if (ok && h < hc) {
                    if (split) {
                        if (q4 == 0) {
                            p.part_ml[(pbase + h) * 2 + 0] = mu;
                            p.part_ml[(pbase + h) * 2 + 1] = l;
                        }
                    } else if (l > 0.f) {
                        inv = 1.f / (l + fast_exp2(M.sink[h] * kLog2e - mu));
                    }
                }
                M.inv[q4][h] = inv;
            }
            mbar_arrive(smem_addr(&M.stats_empty[kpar]));
            __syncwarp();
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c) {
                uint32_t r[kHeads];
                tmem_ld_32x32b_x64(tmem + lane_base + kColO + 64 * c, r);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(smem_addr(&M.o_empty[c]));  // the MMA may refill this chunk now
                if (kRope && 128 * c + 32 * q4 + 32 > kD - p.rope_dim) {
                    // the inverse rotation of the rope dims ("DeepSeek V4.1" attention page,
                    // apply_rotary_emb with inverse, on o[..., -rope_dim:]): lanes 2k and 2k + 1
                    // hold the real and imaginary part of one pair of every head; (a + i b)
                    // (c - i s) = (a c + b s) + i (b c - a s), on the f32 O before any rounding
                    // (split partials too: the merge is linear)
                    const int dd = 128 * c + 32 * q4 + lane, first = kD - p.rope_dim;
                    const bool mine = dd >= first, odd = (lane & 1) != 0;
                    float2 w = rope_last;  // the last chunk's pair was loaded before the wait
                    if (c != kChunks - 1 && mine)
                        w = reinterpret_cast<const float2*>(
                            p.rope)[(p.rope_pos0 + t.pos) * (p.rope_dim / 2) + ((dd - first) >> 1)];
                    const float cs = w.x, sn = w.y;
#pragma unroll
                    for (int i = 0; i < kHeads; ++i) {
                        const float v = __uint_as_float(r[i]);
                        const float u = __shfl_xor_sync(0xffffffffu, v, 1);
                        const float rv = odd ? fmaf(v, cs, -u * sn) : fmaf(v, cs, u * sn);
                        r[i] = __float_as_uint(mine ? rv : v);
                    }
                }
                if (split) {
                    if (ok) {
                        float* po = p.part_o + pbase * kD + 128 * c + 32 * q4 + lane;
#pragma unroll
                        for (int i = 0; i < kHeads; ++i)
                            if (i < hc) po[(int64_t)i * kD] = __uint_as_float(r[i]);
                    }
                    continue;
                }
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) {  // heads 32 rh .. 32 rh + 31 of the block
                    // Lanes 2k and 2k + 1 hold d = 2k and 2k + 1 of every head.  Heads a and a + 1
                    // are packed per word, the neighbours swap words, and the even lane keeps head
                    // a's (d, d + 1) pair, the odd lane head a + 1's.  (O^T is always finite, so a
                    // head with inv = 0 comes out as zeros.)
                    uint32_t out[16];
#pragma unroll
                    for (int mq = 0; mq < 8; ++mq) {
                        const float4 w = *reinterpret_cast<const float4*>(&M.inv[q4][32 * rh + 4 * mq]);
                        const int a = 32 * rh + 4 * mq;
                        // (pairs of heads scaled by one paired multiply: the same two products)
                        const uint32_t pk0 = pack_bf16_2(
                            fmul2(f2(__uint_as_float(r[a]), __uint_as_float(r[a + 1])), f2(w.x, w.y)));
                        const uint32_t pk1 = pack_bf16_2(
                            fmul2(f2(__uint_as_float(r[a + 2]), __uint_as_float(r[a + 3])), f2(w.z, w.w)));
                        out[2 * mq] = __byte_perm(pk0, __shfl_xor_sync(0xffffffffu, pk0, 1), sel);
                        out[2 * mq + 1] = __byte_perm(pk1, __shfl_xor_sync(0xffffffffu, pk1, 1), sel);
                    }
                    // word jj: head 32 rh + 2 jj + odd, d pair 2 (lane / 2) of this warp's 32 d
                    if (ok) {
                        uint32_t* og = reinterpret_cast<uint32_t*>(
                            p.o + ((int64_t)t.token * p.h + h0 + 32 * rh + odd) * kD + 128 * c + 32 * q4 +
                            2 * (lane >> 1));
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            if (32 * rh + 2 * jj + odd < hc) og[(int64_t)jj * kD] = out[jj];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0 && M.abort) atomicOr(p.status, kStatusTimeout);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &f, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

struct TcGeometry {
    int n_tiles, hblocks, n_splits, tiles_per_split;
};

// Split the idx columns of a token over several tasks only when the tokens alone cannot fill
// the GPU's SMs (decode), at pair-of-tiles boundaries.  The split count grows with the SM count,
// so a workspace sized for kMaxSmCount SMs covers every device.
TcGeometry tc_geometry(int64_t n_tokens, int h, int topk, int sms) {
    TcGeometry g;
    g.n_tiles = (topk + kRows - 1) / kRows;
    g.hblocks = (h + kHeads - 1) / kHeads;
    const int pairs = (g.n_tiles + 1) / 2;
    const int64_t base = n_tokens * g.hblocks;
    int splits = 1;
    if (pairs > 1 && base < sms) {
        splits = (int)(sms / base);
        if (splits > pairs) splits = pairs;
        if (splits < 1) splits = 1;
    }
    if (splits > 1) {
        g.tiles_per_split = 2 * ((pairs + splits - 1) / splits);
        g.n_splits = (g.n_tiles + g.tiles_per_split - 1) / g.tiles_per_split;
    } else {
        g.tiles_per_split = g.n_tiles > 0 ? g.n_tiles : 1;
        g.n_splits = 1;
    }
    return g;
}

}  // namespace

bool attn_tc_supports(int h, int d, int kv_format, int64_t b, int64_t rows) {
    (void)h;
    (void)b;
    (void)rows;
    return d == kD && (kv_format == SA_KV_BF16 || kv_format == SA_KV_FP8_E4M3);
}

size_t attn_tc_scratch_bytes(int64_t b, int64_t s, int h, int topk) {
    const TcGeometry g = tc_geometry(b * s, h, topk, kMaxSmCount);
    if (g.n_splits == 1) return 0;
    const size_t ntok = (size_t)(b * s);
    const size_t ml = align_up(ntok * g.n_splits * h * 2 * sizeof(float), 256);
    return ml + ntok * g.n_splits * h * (size_t)kD * sizeof(float);
}

cudaError_t attn_tc_launch(const AttnCall& c) {
    const int64_t n_tokens = c.b * c.s;
    if (c.topk == 0)  // no row at all: o is the zero of an empty sum (rotated or not)
        return cudaMemsetAsync(c.o, 0, (size_t)n_tokens * c.h * kD * 2, c.stream);
    const TcGeometry g = tc_geometry(n_tokens, c.h, c.topk, device_sm_count());
    auto encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap qmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)kD, (cuuint64_t)(n_tokens * c.h)};
    const cuuint64_t gstride[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(c.q), gdim,
                        gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

    Params p;
    const bool fp8 = c.kv_format == SA_KV_FP8_E4M3;
    p.q = reinterpret_cast<const __nv_bfloat16*>(c.q);
    p.rope = c.rope;
    p.rope_dim = c.rope_dim;
    p.rope_pos0 = c.rope_pos0;
    p.kv = fp8 ? nullptr : reinterpret_cast<const __nv_bfloat16*>(c.kv);
    p.kv8 = fp8 ? reinterpret_cast<const uint8_t*>(c.kv) : nullptr;
    p.kv_scale = fp8 ? c.kv_scale : nullptr;
    p.sink = c.sink;
    p.idx = c.idx;
    p.o = reinterpret_cast<__nv_bfloat16*>(c.o);
    p.status = c.status;
    p.scale_log2 = c.softmax_scale * kLog2e;
    p.s_len = c.s;
    p.h = c.h;
    p.hblocks = g.hblocks;
    p.rows = c.rows;
    p.topk = c.topk;
    p.n_tiles = g.n_tiles;
    p.n_splits = g.n_splits;
    p.tiles_per_split = g.tiles_per_split;
    p.n_units = n_tokens * g.n_splits;
    p.part_ml = nullptr;
    p.part_o = nullptr;
    if (g.n_splits > 1) {
        const size_t ml = align_up((size_t)n_tokens * g.n_splits * c.h * 2 * sizeof(float), 256);
        p.part_ml = reinterpret_cast<float*>(c.scratch);
        p.part_o = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(c.scratch) + ml);
    }

    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !configured[dev]) {
        void (*const fns[4])(const CUtensorMap, Params) = {
            attn_tc_kernel<false, false>, attn_tc_kernel<true, false>, attn_tc_kernel<false, true>,
            attn_tc_kernel<true, true>};
        for (auto fn : fns) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
            if (e != cudaSuccess) return e;
        }
        if (dev < 64) configured[dev] = true;
    }
    int64_t groups = device_sm_count() / g.hblocks;  // CTA groups, one CTA per head block
    if (groups > p.n_units) groups = p.n_units;
    if (groups < 1) groups = 1;
    const int64_t grid = groups * g.hblocks;
    const bool rope = c.rope != nullptr;
    auto kernel = fp8 ? (rope ? attn_tc_kernel<true, true> : attn_tc_kernel<true, false>)
                      : (rope ? attn_tc_kernel<false, true> : attn_tc_kernel<false, false>);
    e = launch_pdl(kernel, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, c.stream, qmap, p);
    if (e != cudaSuccess || g.n_splits == 1) return e;
    return attn_combine_launch(p.part_ml, p.part_o, c.sink, c.o, n_tokens, c.h, kD, g.n_splits,
                               c.stream);
}

}  // namespace sa
