// sparse_attn on the 5th-generation tensor cores (tcgen05, accumulators in TMEM), head_dim 512.
//
// Source: "Module attn" API page (spark_model, deepseek_v41_ref/attn), Functions: sparse_attn
// and the precision paragraph; "DeepSeek V4.1" attention page, Attention.forward.
//
// Formulation.  All heads of a query token read the same gathered kv rows, and the rows serve as
// both keys and values.  With head_dim 512 an f32 accumulator of O for 64 heads needs 256 TMEM
// columns in any orientation, while with heads as the MMA's M dimension O takes all 512 columns
// (the full TMEM) and leaves no room for the logits.  So the gathered rows are the M dimension:
//   S^T[128 rows x 64 heads]  = KV_tile[128 x 512] . Q^T            (4 x 8 MMAs, K = 512)
//   O^T[512 x 64 heads]      += KV_tile^T[512 x 128] . P^T[128 x 64] (4 M-chunks x 8 MMAs)
// TMEM holds O^T (256 columns), two S^T buffers (2 x 64), an all-ones bf16 operand (8 columns)
// and the softmax denominators (64 columns): l = ones . P^T is one more MMA per K step, so the
// row sums come from the same bf16 P that multiplies V and are rescaled together with O.  The same swizzled shared-memory
// tile is the K-major A operand of the first product and the MN-major A operand of the second.
// The softmax runs down the columns of S^T (one TMEM lane = one gathered row per thread): the
// column maximum is a warp max reduction plus a 4-warp exchange, and a running maximum is only
// raised (and O rescaled) when a new logit exceeds it by more than 2^8, so the rescale is rare.
// The sink joins the denominator once, in the epilogue: o = O / (l + 2^(sink log2e - m)).
//
// Roles (persistent CTAs, one 64-head block of one query token per task, 384 threads):
//   warp 0      MMA issue (one thread) and TMEM allocation
//   warp 1      Q loads (TMA, 128-byte swizzle)
//   warps 2-3   kv row gather (cp.async 16 B, swizzled in place; rows already resident from the
//               previous tile are kept -- see below)
//   warps 4-7   softmax: S^T -> P^T (bf16, shared memory), running max, O rescale
//   warps 8-11  epilogue: O^T -> o (bf16) or split partials
// Every wait is bounded; a wait that gives up raises the timeout bit and every role unwinds.
//
// Row placement.  The order of the gathered rows inside a tile does not matter (the softmax and
// P.V sum over rows; masking uses the recorded row id of each slot).  When the valid rows of a
// tile have distinct residues mod 128, row j goes to slot j mod 128; otherwise row r of the tile
// goes to slot r.  A row already sitting in its slot from the previous tile is not copied again.
// A CTA takes a contiguous block of tasks, so consecutive query tokens of a sliding window (127
// of 128 rows shared) reload one row per token.

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
constexpr int kRows = 128;        // gathered rows per tile (MMA M)
constexpr int kHeads = 64;        // heads per task (MMA N)
constexpr int kGroups = 4;        // 128-wide d groups (pipeline granularity)
constexpr int kProdWarps = 4;                      // kv gather warps (one tile slot per thread)
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kWarpSoftmax = 2 + kProdWarps;        // first softmax warp
constexpr int kWarpEpilogue = kWarpSoftmax + 4;     // first epilogue warp
constexpr int kThreads = 32 * (kWarpEpilogue + 4);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// TMEM columns: O^T chunks, the two S^T buffers, the all-ones operand, the row sums
constexpr uint32_t kColO = 0, kColS = 256, kColOnes = 384, kColSum = 448;

// Shared-memory map (dynamic, 1024-byte aligned base)
constexpr uint32_t kKvBytes = kRows * kD * 2;     // 128 KB: 8 blocks of [128 rows x 128 B]
constexpr uint32_t kQBytes = kHeads * kD * 2;     // 64 KB: 8 blocks of [64 heads x 128 B]
constexpr uint32_t kPBytes = kRows * kHeads * 2;  // 16 KB: [128 rows x 128 B]
constexpr uint32_t kOffKv = 0;
constexpr uint32_t kOffQ = kOffKv + kKvBytes;
constexpr uint32_t kOffP = kOffQ + kQBytes;
// o staging: one [32 heads x 32 d] box of 64-byte rows (no swizzle) per epilogue warp
constexpr uint32_t kStageBoxBytes = 32 * 64;
constexpr uint32_t kOffStage = kOffP + kPBytes;
constexpr uint32_t kOffMisc = kOffStage + 4 * kStageBoxBytes;

struct Misc {
    uint64_t q_full, q_empty;
    uint64_t kv_full[kGroups], kv_empty[kGroups];  // per 128-d chunk of the kv tile
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full, p_empty;
    uint64_t o_full, o_empty[kGroups];
    uint64_t stats_full[2];
    uint64_t sm_bar, ep_bar, pr_bar, done;
    uint32_t tmem_base;
    int abort;
    int need_corr[2];
    int row_id[2][kRows];              // kv row held by each slot per tile parity, -1 = none
    uint32_t ring_bits[2][4];          // residues mod 128 of a tile's valid rows
    int ring_count[2];                 // number of valid rows of a tile
    int64_t tile_seq[2];               // sequence whose rows a tile holds (-1 = none)
    int2 copy_list[kProdWarps][32];    // per producer warp: (kv row, slot) of the rows to copy
    float colred[4][kHeads];           // per-warp column max of the current tile
    float m[kHeads];                   // running max (log2 units)
    alignas(16) float mu[kHeads];      // the running max with -inf replaced by 0
    float alpha[kHeads];               // rescale factor of this tile
    float stats_m[2][kHeads];          // final max (0 when none) per task parity
    alignas(16) float inv[4][kHeads];  // epilogue: 1 / denominator, a table per epilogue warp
    float sink[128];                   // the sinks of every head
    alignas(16) uint8_t fp8_sc[kRows][16];  // e8m0 scales of the rows an fp8 tile widens, by slot
};
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
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
    int tiles_per_split;
    int64_t n_units;  // (token, split) units; each is one task per head block
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

// A 4-byte shared-memory store in asm without a memory clobber: the compiler may move the
// surrounding shared-memory reads across it (they never touch the same bytes).
__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
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

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap o_map,
                   Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    Misc& M = *reinterpret_cast<Misc*>(smem + kOffMisc);
    const uint32_t s_kv = smem_addr(smem + kOffKv);
    const uint32_t s_q = smem_addr(smem + kOffQ);
    const uint32_t s_p = smem_addr(smem + kOffP);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort = &M.abort;

    if (tid == 0) {
        mbar_init(smem_addr(&M.q_full), 1);
        mbar_init(smem_addr(&M.q_empty), 1);
        for (int c = 0; c < kGroups; ++c) {
            mbar_init(smem_addr(&M.kv_full[c]), kProdThreads);
            mbar_init(smem_addr(&M.kv_empty[c]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&M.s_full[b]), 1);
            mbar_init(smem_addr(&M.s_empty[b]), 128);
            mbar_init(smem_addr(&M.stats_full[b]), 1);
        }
        mbar_init(smem_addr(&M.p_full), 128);
        mbar_init(smem_addr(&M.p_empty), 1);
        mbar_init(smem_addr(&M.o_full), 1);
        for (int c = 0; c < kGroups; ++c) mbar_init(smem_addr(&M.o_empty[c]), 128);
        mbar_init(smem_addr(&M.sm_bar), 128);
        mbar_init(smem_addr(&M.ep_bar), 128);
        mbar_init(smem_addr(&M.pr_bar), kProdThreads);
        mbar_init(smem_addr(&M.done), 1);
        M.abort = 0;
        M.need_corr[0] = M.need_corr[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(&M.tmem_base), 512);
        tmem_relinquish();
    }
    // every slot starts as a finite (zero) row that no tile claims
    for (int i = tid; i < 2 * kRows; i += kThreads) (&M.row_id[0][0])[i] = -1;
    if (tid < 8) (&M.ring_bits[0][0])[tid] = 0;
    if (tid < 2) {
        M.ring_count[tid] = 0;
        M.tile_seq[tid] = -1;
    }
    for (int i = tid; i < p.h; i += kThreads) M.sink[i] = p.sink[i];
    for (uint32_t i = tid; i < kKvBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kOffKv)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1 && lane == 0) tma_prefetch_desc(&q_map);
    if (warp == kWarpEpilogue && lane == 0) tma_prefetch_desc(&o_map);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = M.tmem_base;
    if (warp >= kWarpSoftmax && warp < kWarpEpilogue) {  // all-ones bf16 A operand for the row sums
        tmem_st_32x32b_x8(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kColOnes, 0x3F803F80u);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int64_t tb, te;
    task_range(p, tb, te);


    if (warp == 0) {
        // ------------------------------------------------------------------ MMA issue
        // The whole warp runs this loop (descriptors stay in uniform registers); each MMA and
        // commit is issued by one elected lane, and every lane waits on the barriers.  A wait's
        // result is made warp-uniform so that a time-out cannot split the warp.
        {
            constexpr uint32_t id_s = idesc_bf16_f32(kRows, kHeads, false, false);
            constexpr uint32_t id_o = idesc_bf16_f32(kRows, kHeads, true, true);
            constexpr uint32_t id_l = idesc_bf16_f32(kRows, kHeads, false, true);
            // base descriptors; the per-instruction ones add a start-address offset (>> 4)
            const uint64_t a_s0 = smem_desc_sw128(s_kv, 16, 1024);
            const uint64_t b_s0 = smem_desc_sw128(s_q, 16, 1024);
            const uint64_t a_o0 = smem_desc_sw128(s_kv, 16384, 1024);
            const uint64_t b_o0 = smem_desc_sw128(s_p, 8192, 1024);
            uint32_t T = 0;
            int64_t k = 0;
            bool ok = true;
            Task t = task_of(p, tb);
            for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
                const uint32_t kp = (uint32_t)(k & 1);
                if (t.t0 == t.t1) {  // nothing listed for this task: keep every phase in step
                    ok = warp_wait(smem_addr(&M.q_full), kp, abort);
                    mma_commit_elect(smem_addr(&M.q_empty));
                    for (int c = 0; c < kGroups && ok; ++c)
                        ok = warp_wait(smem_addr(&M.o_empty[c]), kp ^ 1, abort);
                    mma_commit_elect(smem_addr(&M.o_full));
                    continue;
                }
                for (int ti = t.t0; ti < t.t1 && ok; ++ti, ++T) {
                    const uint32_t b = T & 1, use = (T >> 1) & 1, tp = T & 1;
                    const uint32_t s_col = tmem + kColS + 64 * b;
                    // S^T = KV . Q^T: every wait first, then the 32 MMAs back to back
                    ok = warp_wait(smem_addr(&M.s_empty[b]), use ^ 1, abort);
                    if (ok && ti == t.t0) ok = warp_wait(smem_addr(&M.q_full), kp, abort);
                    if (!ok) break;
                    // K step ks (16 of 512): block ks / 4 of the tile / Q, 32 B per step inside
                    // a 128-byte row (2 in the descriptor's 16-byte address units); each 128-d
                    // chunk of the tile as soon as it has landed (the chunk loop is kept rolled: the
                    // issuing warp shares its instruction cache with three other roles)
#pragma unroll 1
                    for (int c = 0; c < kGroups; ++c) {
                        if (!(ok = warp_wait(smem_addr(&M.kv_full[c]), tp, abort))) break;
                        tc_fence_after();
#pragma unroll
                        for (int ks = 8 * c; ks < 8 * c + 8; ++ks)
                            mma_bf16_ss_elect(s_col, a_s0 + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2),
                                        b_s0 + (uint64_t)((ks >> 2) * 512 + (ks & 3) * 2), id_s,
                                        ks != 0);
                    }
                    if (!ok) break;
                    if (ti == t.t1 - 1) mma_commit_elect(smem_addr(&M.q_empty));
                    mma_commit_elect(smem_addr(&M.s_full[b]));
                    // O^T += KV^T . P^T
                    ok = warp_wait(smem_addr(&M.p_full), tp, abort);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < kGroups; ++c) {
                        if (ti == t.t0) {  // the epilogue has read this chunk of the last task's O
                            if (!(ok = warp_wait(smem_addr(&M.o_empty[c]), kp ^ 1, abort))) break;
                            tc_fence_after();
                        }
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)  // 16 rows = 2 KB per K step
                            mma_bf16_ss_elect(tmem + kColO + 64 * c, a_o0 + (uint64_t)(c * 2048 + ks * 128),
                                        b_o0 + (uint64_t)(ks * 128), id_o, !(ti == t.t0 && ks == 0));
                        mma_commit_elect(smem_addr(&M.kv_empty[c]));  // chunk c of the tile is read
                    }
                    if (!ok) break;
                    // l += ones . P^T (every element of the A operand is 1, so one 8-column
                    // block of TMEM serves every K step)
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_bf16_ts_elect(tmem + kColSum, tmem + kColOnes, b_o0 + (uint64_t)(ks * 128),
                                    id_l, !(ti == t.t0 && ks == 0));
                    mma_commit_elect(smem_addr(&M.p_empty));
                    if (ti == t.t1 - 1) mma_commit_elect(smem_addr(&M.o_full));
                }
            }
            // let every issued MMA finish before the accumulators are released
            mma_commit_elect(smem_addr(&M.done));
            warp_wait(smem_addr(&M.done), 0, abort);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ Q loads (TMA)
        if (lane == 0) {
            int64_t k = 0;
            bool ok = true;
            Task t = task_of(p, tb);
            for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
                const int32_t y = (int32_t)(t.token * p.h + (int64_t)t.hb * kHeads);
                ok = mbar_wait(smem_addr(&M.q_empty), (uint32_t)(k & 1) ^ 1, abort);
                if (!ok) break;
                const uint32_t bar = smem_addr(&M.q_full);
                mbar_arrive_expect_tx(bar, kQBytes);
#pragma unroll 1
                for (int c = 0; c < 8; ++c)  // 8 boxes of [64 heads x 64 d], 128-byte swizzle
                    tma_load_2d(s_q + c * 8192, &q_map, 64 * c, y, bar);
            }
            // after a failed wait, let the last Q load land before the CTA exits
            if (!ok && k > 0) mbar_drain(smem_addr(&M.q_full), (uint32_t)((k - 1) & 1));
        }
        __syncwarp();
    } else if (warp < kWarpSoftmax) {
        // ------------------------------------------------------------------ kv gather
        // Each thread resolves one of the tile's 128 slots; every warp lists the rows it copies
        // and copies each 128-d chunk of them (cp.async, one commit group per chunk) as soon as
        // the previous tile's P.V has finished reading that chunk; chunk c is signalled once the
        // group has landed.
        const int pw = warp - 2;       // producer warp 0 .. kProdWarps - 1
        const int pt_id = tid - 64;    // the tile slot (column placement) this thread resolves
        uint32_t T = 0, pr_phase = 0;
        bool ok = true;
        Task t = task_of(p, tb);
        for (int64_t tau = tb; tau < te && ok; ++tau, task_step(p, t)) {
            const int64_t bi = t.seq;
            const int32_t* idx_tok = p.idx + t.token * (int64_t)p.topk;
            const __nv_bfloat16* kvb = p.kv + bi * p.rows * (int64_t)kD;
            for (int ti = t.t0; ti < t.t1 && ok; ++ti, ++T) {
                const uint32_t tp = T & 1;
                const int col = ti * kRows + pt_id;
                int j = col < p.topk ? __ldg(idx_tok + col) : -1;
                if (j < -1 || j >= p.rows) {
                    atomicOr(p.status, kStatusBadIndex);
                    j = -1;
                }
                // placement: ring (slot = j mod 128) when the valid rows' residues are distinct.
                // (row_id[tp] is only written after the tile barrier below: the softmax of the
                // tile two back, which has the same parity, may still be reading it until then.)
                if (j >= 0) {
                    atomicOr(&M.ring_bits[tp][(j & 127) >> 5], 1u << (j & 31));
                    atomicAdd(&M.ring_count[tp], 1);
                }
                if (pt_id == 0) M.tile_seq[tp] = bi;
                if (!(ok = wg_sync(smem_addr(&M.pr_bar), pr_phase, abort))) break;
                // a slot's row can be kept only if it belongs to this same sequence
                const bool same_seq = M.tile_seq[tp ^ 1] == bi;
                const bool ring = __popc(M.ring_bits[tp][0]) + __popc(M.ring_bits[tp][1]) +
                                      __popc(M.ring_bits[tp][2]) + __popc(M.ring_bits[tp][3]) ==
                                  M.ring_count[tp];
                // this thread's own slot is empty unless a row claims it
                const bool claimed = ring ? ((M.ring_bits[tp][pt_id >> 5] >> (pt_id & 31)) & 1) != 0
                                          : j >= 0;
                if (!claimed) M.row_id[tp][pt_id] = -1;
                const int slot = ring ? (j & 127) : pt_id;
                const bool copy = j >= 0 && (!same_seq || M.row_id[tp ^ 1][slot] != j);
                if (j >= 0) M.row_id[tp][slot] = j;
                if (pt_id == 0) {  // the next tile (other parity) starts from a clean slate
                    M.ring_bits[tp ^ 1][0] = M.ring_bits[tp ^ 1][1] = 0;
                    M.ring_bits[tp ^ 1][2] = M.ring_bits[tp ^ 1][3] = 0;
                    M.ring_count[tp ^ 1] = 0;
                }
                // the rows this warp copies, compacted into a list (ballot prefix count)
                const uint32_t m0 = __ballot_sync(0xFFFFFFFFu, copy);
                const int ncopy = __popc(m0);
                if (copy) M.copy_list[pw][__popc(m0 & ((1u << lane) - 1u))] = make_int2(j, slot);
                // the previous tile is usually still in use: pull this tile's new rows into L2
                // now, so that the copies issued once its chunks are released hit L2
                if (copy) {
                    if constexpr (kFp8) {
                        prefetch_l2(p.kv8 + (bi * p.rows + j) * (int64_t)kD, kD);
                        prefetch_l2(p.kv_scale + (bi * p.rows + j) * (int64_t)(kD / 32), kD / 32);
                    } else {
                        prefetch_l2(kvb + (int64_t)j * kD, kD * 2);
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
                    int2 ent8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int e = (lane >> 3) + 4 * i;
                        ent8[i] = e < ncopy ? M.copy_list[pw][e] : make_int2(-1, 0);
                    }
                    // stage every chunk as soon as P.V has released it ...
#pragma unroll
                    for (int c = 0; c < kGroups; ++c) {
                        if (ok) ok = mbar_wait(smem_addr(&M.kv_empty[c]), tp ^ 1, abort);
                        if (ok) {
                            if (c == 0 && lane < ncopy) {  // the row's 16 scales
                                const int2 en = M.copy_list[pw][lane];
                                cp_async16(smem_addr(&M.fp8_sc[en.y][0]),
                                           scb + (int64_t)en.x * (kD / 32), 16u);
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                if (ent8[i].x < 0) break;
                                cp_async16(s_kv + (2 * c + 1) * 16384 + ent8[i].y * 128 + unit * 16,
                                           kvb8 + (int64_t)ent8[i].x * kD + 128 * c + unit * 16, 16u);
                            }
                        }
                        cp_async_commit();
                    }
                    // ... then widen them in order, each once its group has landed
#pragma unroll
                    for (int cw = 0; cw < kGroups; ++cw) {
                        if (cw == 0) cp_async_wait<3>();
                        else if (cw == 1) cp_async_wait<2>();
                        else if (cw == 2) cp_async_wait<1>();
                        else cp_async_wait<0>();
                        __syncwarp();  // every lane's staged codes are visible to the warp
                        uint4 code[8];
                        float sc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (ent8[i].x < 0) break;
                            const int r = ent8[i].y;
                            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                         : "=r"(code[i].x), "=r"(code[i].y), "=r"(code[i].z), "=r"(code[i].w)
                                         : "r"(s_kv + (2 * cw + 1) * 16384 + r * 128 + unit * 16)
                                         : "memory");
                            sc[i] = fp8::e8m0_to_f32(M.fp8_sc[r][4 * cw + (unit >> 1)]);
                        }
                        __syncwarp();  // all codes read before any lane overwrites them
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (ent8[i].x < 0) break;
                            const int r = ent8[i].y;
                            uint4 lo, hi;
                            fp8::dequant16(code[i], sc[i], lo, hi);
                            const int u = 16 * cw + 2 * unit;  // 16-byte bf16 units u, u + 1
                            const uint32_t row = s_kv + (u >> 3) * 16384 + r * 128;
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             row + ((((u & 7) ^ (r & 7)) & 7) << 4)),
                                         "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w)
                                         : "memory");
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             row + (((((u + 1) & 7) ^ (r & 7)) & 7) << 4)),
                                         "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                                         : "memory");
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(smem_addr(&M.kv_full[cw]));
                    }
                    if (!ok) break;
                    continue;
                }
                if (ncopy <= 2) {
                    // few new rows (e.g. the next token of a sliding window): load them into
                    // registers now, while the previous tile is still being used, and write them
                    // to their slots chunk by chunk as the tile is released
                    uint4 v[2][2];
                    int2 ent[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        ent[e] = e < ncopy ? M.copy_list[pw][e] : make_int2(-1, 0);
                        if (ent[e].x >= 0) {
                            const uint4* src = reinterpret_cast<const uint4*>(kvb + (int64_t)ent[e].x * kD);
                            v[e][0] = __ldg(src + lane);
                            v[e][1] = __ldg(src + 32 + lane);
                        }
                    }
                    // chunk c (units 16 c .. 16 c + 15) is held by the lanes with lane / 16 ==
                    // c % 2, in v[.][c / 2]; each chunk is written and signalled as soon as P.V
                    // has released it
#pragma unroll
                    for (int c = 0; c < kGroups; ++c) {
                        if (ok) ok = mbar_wait(smem_addr(&M.kv_empty[c]), tp ^ 1, abort);
                        if (ok && (lane >> 4) == (c & 1)) {
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                if (ent[e].x < 0) continue;
                                const int r = ent[e].y;
                                const int u = 32 * (c >> 1) + lane;  // 16-byte unit of the 1 KB row
                                const uint4 w = v[e][c >> 1];
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                                 s_kv + (u >> 3) * 16384 + r * 128 +
                                                 ((((u & 7) ^ (r & 7)) & 7) << 4)),
                                             "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                                             : "memory");
                            }
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(smem_addr(&M.kv_full[c]));
                    }
                    if (!ok) break;
                    continue;
                }
                // this lane's rows of the list: entries lane / 16 + 2 i (two rows per instruction)
                int2 ent[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int e = (lane >> 4) + 2 * i;
                    ent[i] = e < ncopy ? M.copy_list[pw][e] : make_int2(-1, 0);
                }
                // chunk c = 16-byte units 16 c .. 16 c + 15 of each row (blocks 2 c and 2 c + 1)
#pragma unroll
                for (int c = 0; c < kGroups; ++c) {
                    if (ok) ok = mbar_wait(smem_addr(&M.kv_empty[c]), tp ^ 1, abort);
                    if (ok) {
                        const int u = 16 * c + (lane & 15);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (ent[i].x < 0) break;
                            const int r = ent[i].y;
                            const uint32_t dst =
                                s_kv + (u >> 3) * 16384 + r * 128 + ((((u & 7) ^ (r & 7)) & 7) << 4);
                            cp_async16(dst, kvb + (int64_t)ent[i].x * kD + u * 8, 16u);
                        }
                    }
                    cp_async_commit();  // (an empty group after a failed wait keeps the count)
                }
                if (!ok) break;
                cp_async_wait<3>();
                fence_proxy_async_smem();
                mbar_arrive(smem_addr(&M.kv_full[0]));
                cp_async_wait<2>();
                fence_proxy_async_smem();
                mbar_arrive(smem_addr(&M.kv_full[1]));
                cp_async_wait<1>();
                fence_proxy_async_smem();
                mbar_arrive(smem_addr(&M.kv_full[2]));
                cp_async_wait<0>();
                fence_proxy_async_smem();
                mbar_arrive(smem_addr(&M.kv_full[3]));
            }
        }
        cp_async_wait<0>();
    } else if (warp < kWarpEpilogue) {
        // ------------------------------------------------------------------ softmax
        // Per tile: column max of the logits -> running max m (raised only past the threshold),
        // p = 2^(x - m) written as P^T, and the tile's column sums; the sums are folded into the
        // running l = alpha * l + sum at the next tile (and once more at the end of the task).
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;  // TMEM lane = tile row
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint32_t T = 0, sm_phase = 0;
        int64_t k = 0;
        bool ok = true;
        Task t = task_of(p, tb);
        for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
            const int kpar = (int)(k & 1);
            for (int ti = t.t0; ti < t.t1 && ok; ++ti, ++T) {
                const uint32_t b = T & 1, use = (T >> 1) & 1, tp = T & 1;
                const bool first = ti == t.t0;
                ok = mbar_wait(smem_addr(&M.kv_full[0]), tp, abort);  // the tile's row ids
                if (ok) ok = mbar_wait(smem_addr(&M.s_full[b]), use, abort);
                if (!ok) break;
                // an empty slot's logits become -inf (pass 1) and its P^T row zeros (pass 2)
                const bool valid = M.row_id[tp][row] >= 0;
                const float row_bias = valid ? 0.f : -INFINITY;
                const uint32_t row_mask = valid ? 0xFFFFFFFFu : 0u;
                const uint32_t s_addr = tmem + lane_base + kColS + 64 * b;
                tc_fence_after();
                // pass 1: column maximum of the scaled logits over the 128 rows; lane i keeps the
                // warp maxima of heads i and 32 + i
                {
                    uint32_t r[kHeads];
                    tmem_ld_32x32b_x64(s_addr, r);
                    tmem_wait_ld();
                    float mine0 = -INFINITY, mine1 = -INFINITY;
#pragma unroll
                    for (int i = 0; i < kHeads; ++i) {
                        const float x = fmaf(__uint_as_float(r[i]), p.scale_log2, row_bias);
                        float mx;
                        asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx) : "f"(x));
                        if (i < 32) {
                            if (lane == i) mine0 = mx;
                        } else {
                            if (lane == i - 32) mine1 = mx;
                        }
                    }
                    M.colred[q4][lane] = mine0;
                    M.colred[q4][32 + lane] = mine1;
                }
                if (!(ok = wg_sync(smem_addr(&M.sm_bar), sm_phase, abort))) break;
                if (row < kHeads) {
                    const int h = row;
                    const float cm = fmaxf(fmaxf(M.colred[0][h], M.colred[1][h]),
                                           fmaxf(M.colred[2][h], M.colred[3][h]));
                    const float mo = M.m[h];
                    float mn, al = 1.f;
                    if (first) {
                        mn = cm;
                    } else {
                        mn = cm > mo + kRescaleThreshold ? cm : mo;
                        if (mn != mo) {
                            al = fast_exp2(mo - mn);  // 0 when mo = -inf (nothing summed yet)
                            M.need_corr[tp] = 1;
                        }
                    }
                    M.m[h] = mn;
                    M.mu[h] = mn == -INFINITY ? 0.f : mn;
                    M.alpha[h] = al;
                }
                if (!(ok = wg_sync(smem_addr(&M.sm_bar), sm_phase, abort))) break;
                const bool corr = !first && M.need_corr[tp];
                if (row == 0) M.need_corr[tp ^ 1] = 0;

                // P buffer free and the previous PV done (O stable)
                ok = mbar_wait(smem_addr(&M.p_empty), tp ^ 1, abort);
                if (!ok) break;
                if (corr) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 2 * kGroups + 2; ++c) {  // O^T (8 blocks), then l (2)
                        uint32_t r[32];
                        const uint32_t ta = tmem + lane_base +
                                            (c < 2 * kGroups ? kColO + 32 * c : kColSum + 32 * (c & 1));
                        tmem_ld_32x32b_x32(ta, r);
                        tmem_wait_ld();
                        const float* al = &M.alpha[32 * (c & 1)];
#pragma unroll
                        for (int h = 0; h < 32; ++h)
                            r[h] = __float_as_uint(__uint_as_float(r[h]) * al[h]);
                        tmem_st_32x32b_x32(ta, r);
                    }
                    tmem_wait_st();
                }
                // pass 2: p = 2^(x - m) as the P^T row (128-byte swizzled MN-major operand); the
                // sums are accumulated by the tensor core from P^T
                {
                    uint32_t r[kHeads];
                    tmem_ld_32x32b_x64(s_addr, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 8; ++u) {  // 16-byte unit u of the row: heads 8u .. 8u + 7
                        const float4 ma = *reinterpret_cast<const float4*>(&M.mu[8 * u]);
                        const float4 mb = *reinterpret_cast<const float4*>(&M.mu[8 * u + 4]);
                        const float mu8[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
                        float e[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            e[i] = fast_exp2(fmaf(__uint_as_float(r[8 * u + i]), p.scale_log2, -mu8[i]));
                        const uint32_t dst = s_p + row * 128 + (((u ^ (row & 7)) & 7) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                                     "r"(pack_bf16(e[0], e[1]) & row_mask),
                                     "r"(pack_bf16(e[2], e[3]) & row_mask),
                                     "r"(pack_bf16(e[4], e[5]) & row_mask),
                                     "r"(pack_bf16(e[6], e[7]) & row_mask));
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_addr(&M.s_empty[b]));
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_addr(&M.p_full));
            }
            if (!ok) break;
            // final statistics of the task: the running max per head (the sums are in TMEM)
            if (!(ok = wg_sync(smem_addr(&M.sm_bar), sm_phase, abort))) break;
            if (row < kHeads) {
                const float mh = t.t1 > t.t0 ? M.m[row] : -INFINITY;
                M.stats_m[kpar][row] = mh == -INFINITY ? 0.f : mh;
            }
            if (!(ok = wg_sync(smem_addr(&M.sm_bar), sm_phase, abort))) break;
            if (row == 0) mbar_arrive(smem_addr(&M.stats_full[kpar]));
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        // O^T chunk c (128 d x 64 heads) leaves TMEM at once (the MMA may refill it), is scaled by
        // 1 / denominator and packed to bf16.  Each warp (32 d) transposes its part through its
        // own [32 heads x 32 d] shared-memory box and stores it to o with TMA, synchronising only
        // with itself.  Every thread passes every barrier of a task, even after a failed wait, so
        // the warpgroup's barriers never split.
        const int q4 = warp & 3;
        const int et = tid - 32 * kWarpEpilogue;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        // this warp's box: 32 rows (heads) of 64 bytes (32 d); this thread's word in a row holds
        // the d pair 2 (lane / 2), 2 (lane / 2) + 1
        const uint32_t s_box = smem_addr(smem + kOffStage) + q4 * kStageBoxBytes;
        const int odd = lane & 1;
        const uint32_t sel = odd ? 0x3276u : 0x5410u;
        const uint32_t st_base = s_box + 4 * (lane >> 1) + 64 * odd;
        int64_t k = 0;
        bool ok = true;
        Task t = task_of(p, tb);
        for (int64_t tau = tb; tau < te && ok; ++tau, ++k, task_step(p, t)) {
            const int kpar = (int)(k & 1);
            const int h0 = t.hb * kHeads;
            const int hc = min(kHeads, p.h - h0);
            ok = mbar_wait(smem_addr(&M.o_full), (uint32_t)kpar, abort);
            if (ok) ok = mbar_wait(smem_addr(&M.stats_full[kpar]), (uint32_t)((k >> 1) & 1), abort);
            tc_fence_after();
            const bool split = p.n_splits > 1;
            const int64_t pbase = (t.token * p.n_splits + t.split) * (int64_t)p.h + h0;
            // the denominators: every TMEM lane of the sum block holds the same row sums, so
            // each warp reads them all and lane l finishes heads l and l + 32 into the warp's own
            // table (no barrier across the warps)
            {
                float lsum[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem + lane_base + kColSum + 32 * hh, r);
                    tmem_wait_ld();
                    float v = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (lane == i) v = __uint_as_float(r[i]);
                    lsum[hh] = t.t1 > t.t0 ? v : 0.f;
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = lane + 32 * hh;
                    const float l = lsum[hh], mu = M.stats_m[kpar][h];
                    float inv = 0.f;
                    if (ok && h < hc) {
                        if (split) {
                            if (q4 == 0) {
                                p.part_ml[(pbase + h) * 2 + 0] = mu;
                                p.part_ml[(pbase + h) * 2 + 1] = l;
                            }
                        } else if (l > 0.f) {
                            inv = 1.f / (l + fast_exp2(M.sink[h0 + h] * kLog2e - mu));
                        }
                    }
                    M.inv[q4][h] = inv;
                }
                __syncwarp();
            }
#pragma unroll 1
            for (int c = 0; c < kGroups; ++c) {
                uint32_t r[kHeads];
                tmem_ld_32x32b_x64(tmem + lane_base + 64 * c, r);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(smem_addr(&M.o_empty[c]));  // the MMA may refill this chunk now
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
                    // a's (d, d + 1) pair, the odd lane head a + 1's: rows a and a + 1 of the box
                    // are 64 bytes apart, in opposite halves of the banks.  (O^T is always finite,
                    // so a head with inv = 0 comes out as zeros.)
                    uint32_t out[16];
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float4 w = *reinterpret_cast<const float4*>(&M.inv[q4][32 * rh + 4 * m]);
                        const int a = 32 * rh + 4 * m;
                        const uint32_t pk0 = pack_bf16(__uint_as_float(r[a]) * w.x,
                                                       __uint_as_float(r[a + 1]) * w.y);
                        const uint32_t pk1 = pack_bf16(__uint_as_float(r[a + 2]) * w.z,
                                                       __uint_as_float(r[a + 3]) * w.w);
                        out[2 * m] = __byte_perm(pk0, __shfl_xor_sync(0xffffffffu, pk0, 1), sel);
                        out[2 * m + 1] = __byte_perm(pk1, __shfl_xor_sync(0xffffffffu, pk1, 1), sel);
                    }
                    // the box is free once this warp's previous store has read it
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 16; ++j) st_shared_b32(st_base + 128 * j, out[j]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && ok && h0 + 32 * rh < p.h) {
                        tma_store_3d(&o_map, s_box, 128 * c + 32 * q4, h0 + 32 * rh,
                                     (int32_t)t.token);
                        bulk_commit();
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
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

int sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 64 && counts[dev]) return counts[dev];
    int n = 148;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev < 64) counts[dev] = n;
    return n;
}

struct TcGeometry {
    int n_tiles, hblocks, n_splits, tiles_per_split;
};

// Split the idx columns of a token over several tasks only when the tokens alone cannot fill
// the GPU (decode); the split count is device-independent so the workspace size is too.
TcGeometry tc_geometry(int64_t n_tokens, int h, int topk) {
    constexpr int kAssumedSms = 152;
    TcGeometry g;
    g.n_tiles = (topk + kRows - 1) / kRows;
    g.hblocks = (h + kHeads - 1) / kHeads;
    const int64_t base = n_tokens * g.hblocks;
    int splits = 1;
    if (g.n_tiles > 1 && base < kAssumedSms) {
        splits = (int)(kAssumedSms / base);
        if (splits > g.n_tiles) splits = g.n_tiles;
        if (splits < 1) splits = 1;
    }
    g.tiles_per_split = splits > 1 ? (g.n_tiles + splits - 1) / splits : (g.n_tiles > 0 ? g.n_tiles : 1);
    g.n_splits = splits > 1 ? (g.n_tiles + g.tiles_per_split - 1) / g.tiles_per_split : 1;
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
    const TcGeometry g = tc_geometry(b * s, h, topk);
    if (g.n_splits == 1) return 0;
    const size_t ntok = (size_t)(b * s);
    const size_t ml = align_up(ntok * g.n_splits * h * 2 * sizeof(float), 256);
    return ml + ntok * g.n_splits * h * (size_t)kD * sizeof(float);
}

cudaError_t attn_tc_launch(const AttnCall& c) {
    const int64_t n_tokens = c.b * c.s;
    const TcGeometry g = tc_geometry(n_tokens, c.h, c.topk);
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
    // o as [tokens][h][512]: a [1 x 32 x 32] box is clipped at h for a partial head block
    CUtensorMap omap;
    const cuuint64_t odim[3] = {(cuuint64_t)kD, (cuuint64_t)c.h, (cuuint64_t)n_tokens};
    const cuuint64_t ostride[2] = {(cuuint64_t)kD * 2, (cuuint64_t)c.h * kD * 2};
    const cuuint32_t obox[3] = {32, (cuuint32_t)(c.h < 32 ? c.h : 32), 1};
    const cuuint32_t oestride[3] = {1, 1, 1};
    r = encode(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, c.o, odim, ostride, obox, oestride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

    Params p;
    const bool fp8 = c.kv_format == SA_KV_FP8_E4M3;
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
        e = cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_tc_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev < 64) configured[dev] = true;
    }
    int64_t groups = sm_count() / g.hblocks;  // CTA groups, one CTA per head block
    if (groups > p.n_units) groups = p.n_units;
    if (groups < 1) groups = 1;
    const int64_t grid = groups * g.hblocks;
    if (fp8)
        attn_tc_kernel<true><<<(unsigned)grid, kThreads, kSmemBytes, c.stream>>>(qmap, omap, p);
    else
        attn_tc_kernel<false><<<(unsigned)grid, kThreads, kSmemBytes, c.stream>>>(qmap, omap, p);
    e = cudaGetLastError();
    if (e != cudaSuccess || g.n_splits == 1) return e;
    return attn_combine_launch(p.part_ml, p.part_o, c.sink, c.o, n_tokens, c.h, kD, g.n_splits,
                               c.stream);
}

}  // namespace sa
