// sa_sparse_attn_static_scratch: sparse_attn for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin loaded into a host runtime that owns
// every device allocation and hands the plugin none, or a latency-critical serving loop that
// must not call cudaMalloc / cudaFree on the request path (both can synchronise the device).
// This entry point gives them sparse_attn with the workspace taken from a fixed array in the
// library's own device memory instead.
//
// The array is a file-scope __device__ variable of SA_STATIC_SCRATCH_BYTES; every GPU that loads
// the library keeps it until the process exits.  Host code cannot use the array's name as a
// device address (on the host it names a shadow variable), so the first call on each device
// looks the address up with cudaGetSymbolAddress while that device is current and caches it;
// make that first call before any stream capture.  All calls share the one array and it keeps
// the previous call's contents: the status word is cleared on the stream at the start of every
// call, and two calls whose work overlaps on the GPU (different streams, no ordering) race on
// the array.  Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library call.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "sa_internal.cuh"
#include "sparse_attn.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchTable {
    std::mutex mu;
    void* ptr[kMaxDevices] = {};
};

ScratchTable& table() {
    static ScratchTable t;
    return t;
}

// Device address of the array on the current device, looked up once per device.
sa_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
    ScratchTable& t = table();
    std::lock_guard<std::mutex> lock(t.mu);
    if (!t.ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) return SA_ERR_CUDA;
        t.ptr[dev] = p;
    }
    *out = t.ptr[dev];
    return SA_OK;
}

}  // namespace

extern "C" sa_status sa_sparse_attn_static_scratch(
    const void* q, const void* kv, const uint8_t* kv_scale, int kv_format, const float* sink,
    const int32_t* idx, float softmax_scale, int64_t b, int64_t s, int h, int d, int64_t rows,
    int topk, void* o, uint32_t* status_out, void* stream) {
    if (kv_format != SA_KV_BF16 && kv_format != SA_KV_FP8_E4M3) return SA_ERR_INVALID_ARG;
    if (b < 0 || s < 0 || h < 1 || d < 1 || rows < 0 || topk < 0) return SA_ERR_INVALID_ARG;
    if (sa_sparse_attn_workspace_size(b, s, h, d, rows, topk, kv_format) == 0) return SA_ERR_UNSUPPORTED;
    // the scratch of the family sa_sparse_attn routes this call to
    const int fam = sa::routed_family(SA_FAMILY_AUTO, h, d, kv_format, b, rows);
    if (fam < 0) return SA_ERR_UNSUPPORTED;
    const size_t need = sa::routed_workspace_bytes(fam, b, s, h, d, rows, topk);
    if (need > (size_t)SA_STATIC_SCRATCH_BYTES) return SA_ERR_WORKSPACE;  // beyond the array
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // sa_sparse_attn checks every other argument before it looks at the workspace, so a call
    // without one validates the arguments and enqueues nothing
    const sa_status pre = sa_sparse_attn(q, kv, kv_scale, kv_format, sink, idx, softmax_scale, b, s,
                                         h, d, rows, topk, o, nullptr, 0, stream);
    if (pre == SA_OK) {  // b * s == 0: nothing to compute, but the status word is still reported
        if (status_out && cudaMemsetAsync(status_out, 0, sizeof(uint32_t), cs) != cudaSuccess)
            return SA_ERR_CUDA;
        return SA_OK;
    }
    if (pre != SA_ERR_WORKSPACE) return pre;  // an argument error
    void* scratch = nullptr;
    const sa_status st = scratch_address(&scratch);
    if (st != SA_OK) return st;
    if (cudaMemsetAsync(scratch, 0, SA_STATUS_BYTES, cs) != cudaSuccess) return SA_ERR_CUDA;
    const sa_status run = sa_sparse_attn(q, kv, kv_scale, kv_format, sink, idx, softmax_scale, b,
                                         s, h, d, rows, topk, o, scratch,
                                         (size_t)SA_STATIC_SCRATCH_BYTES, stream);
    if (run != SA_OK) return run;
    if (status_out &&
        cudaMemcpyAsync(status_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, cs) !=
            cudaSuccess)
        return SA_ERR_CUDA;
    return SA_OK;
}
