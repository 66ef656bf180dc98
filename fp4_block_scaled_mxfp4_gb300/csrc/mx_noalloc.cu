// mx_noalloc.cu -- moe_mxfp4_forward for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and are not allowed to
// allocate: a custom-op or plugin interface whose host framework owns every device
// allocation and passes no workspace, code that must not trigger cudaMalloc's implicit
// device-wide synchronisation, or a process whose device memory is already fully reserved
// by another allocator. For them the MoE forward runs on a fixed scratch area that lives
// in the library itself: a file-scope static __device__ array, created on every device
// that loads the library and held until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mxfp4moe.h"

namespace {

// The scratch area (one per device). Host code may not use this symbol as a pointer: its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MXFP4MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch area on the current device, looked up once per device.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MX_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MX_OK;
}

}  // namespace

extern "C" int moe_mxfp4_forward_noalloc(const void* x, const int32_t* topk_ids, const float* topk_w,
                                         const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                                         const uint8_t* s2, void* out, int64_t T, int64_t H, int64_t I,
                                         int64_t E, int64_t K, mx_stream_t stream) {
    const int routed = topk_ids != nullptr ? 1 : 0;
    // argument rules first, in moe_mxfp4_forward's order and with no CUDA call, so both
    // entry points return the same status: routing ids and weights come together, then
    // the size rules, then the scratch limit
    if ((topk_ids != nullptr) != (topk_w != nullptr)) return MX_ERR_INVALID_ARG;
    int64_t layout[8];
    if (int st = moe_mxfp4_workspace_layout(T, H, I, E, K, routed, layout)) return st;
    if (moe_mxfp4_workspace_size(T, H, I, E, K, routed) > MXFP4MOE_NOALLOC_SCRATCH_BYTES) return MX_ERR_WORKSPACE;
    if (T == 0) return MX_OK;
    void* scratch = nullptr;
    if (int st = scratch_address(&scratch)) return st;
    // The forward's results never depend on scratch bytes it did not write in the same call
    // (rows it reads without writing only feed rows that are never stored), so whatever the
    // previous call left there needs no clearing.
    return moe_mxfp4_forward(x, topk_ids, topk_w, w13, s13, w2, s2, out, T, H, I, E, K, scratch,
                             MXFP4MOE_NOALLOC_SCRATCH_BYTES, stream);
}
