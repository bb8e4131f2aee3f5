// Internal declarations shared by the library's CUDA translation units (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_attn.h"

namespace sa {

// The kernels size their grids from the device's SM count, taken at most this large; workspace
// sizes assume this many SMs, so that they depend on the shape only (GB300: 152).
constexpr int kMaxSmCount = 160;

// SMs of the current device, at most kMaxSmCount (cached per device; sa_helpers.cu).
int device_sm_count();

// Status word bits (first 32-bit word of the workspace status block).
constexpr uint32_t kStatusBadIndex = 1u;
constexpr uint32_t kStatusTimeout = 2u;

// Everything a sparse_attn kernel family needs for one call, already validated.
struct AttnCall {
    const void* q;
    const void* kv;
    const uint8_t* kv_scale;
    int kv_format;
    const float* sink;
    const int32_t* idx;
    float softmax_scale;
    int64_t b, s;
    int h, d;
    int64_t rows;
    int topk;
    void* o;
    uint32_t* status;   // device status word
    void* scratch;      // workspace past the status block
    size_t scratch_bytes;
    cudaStream_t stream;
    // optional inverse rotation of o's last rope_dim dims (apply_rotary_emb, inverse): rope is the
    // [positions][rope_dim / 2][2] (cos, sin) f32 table, token (bi, si) at position rope_pos0 + si;
    // nullptr for none
    const float* rope = nullptr;
    int rope_dim = 0;
    int64_t rope_pos0 = 0;
};

// mma.sync family (sa_attn_mma.cu)
size_t attn_mma_scratch_bytes(int64_t b, int64_t s, int h, int d, int topk);
cudaError_t attn_mma_launch(const AttnCall& c);
// merge of split partials: part_ml [tokens][splits][h][2] (max in log2 units, sum),
// part_o [tokens][splits][h][d] f32 -> o bf16 (sa_attn_mma.cu)
cudaError_t attn_combine_launch(const float* part_ml, const float* part_o, const float* sink,
                                void* o, int64_t n_tokens, int h, int d, int n_splits,
                                cudaStream_t stream);

// tcgen05 family (sa_attn_tc.cu)
// d = 512 with bf16 kv
bool attn_tc_supports(int h, int d, int kv_format, int64_t b, int64_t rows);
size_t attn_tc_scratch_bytes(int64_t b, int64_t s, int h, int topk);
cudaError_t attn_tc_launch(const AttnCall& c);

// helpers (sa_helpers.cu)
cudaError_t window_idxs_launch(int64_t start_pos, int64_t seqlen, int window, int32_t* idx,
                               int64_t ld, int64_t nbatch, int64_t batch_stride,
                               cudaStream_t stream);
cudaError_t window_write_launch(const void* x, int64_t nbatch, int64_t seqlen, int d,
                                int64_t x_stride, int64_t start_pos, int window, void* ring_rt,
                                int64_t rt_stride, int64_t rt_batch_stride, uint8_t* codes,
                                int64_t codes_stride, int64_t codes_batch_stride, uint8_t* scales,
                                int64_t scales_stride, int64_t scales_batch_stride,
                                cudaStream_t stream);
cudaError_t act_quant_launch(const void* x, int64_t n, int d, int64_t x_stride, void* x_rt,
                             int64_t rt_stride, uint8_t* codes, int64_t codes_stride,
                             uint8_t* scales, int64_t scales_stride, cudaStream_t stream);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Programmatic dependent launches.  The kernels of one sparse_attn step (window table, act_quant
// or ring write, attention, split merge) are launched so that each may be scheduled while the
// work queued before it on the stream drains.  A kernel so launched may do set-up that touches
// no global memory (barriers, TMEM, shared memory), must call pdl_wait() before its first global
// read or write (it returns once every earlier grid on the stream has completed and its writes
// are visible; with no such grid it returns at once), and calls pdl_trigger() to let the launch
// after it be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <class Kernel, class... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Routing (sa_api.cu): the family a call runs in (SA_FAMILY_AUTO resolved; -1 = that family
// cannot run the shape), and the workspace bytes that family needs for the shape.
int routed_family(int family, int h, int d, int kv_format, int64_t b, int64_t rows);
size_t routed_workspace_bytes(int family, int64_t b, int64_t s, int h, int d, int64_t rows,
                              int topk);

}  // namespace sa
