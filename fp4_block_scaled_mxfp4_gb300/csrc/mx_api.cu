// mx_api.cu -- the C ABI (include/mxfp4moe.h): argument validation, workspace layout,
// TMA tensor-map encoding and the launch sequence of each call. No device memory is
// allocated here; every launch goes to the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <nvtx3/nvToolsExt.h>

#include <cstring>
#include <mutex>

#include "../../include/mxfp4moe.h"
#include "mx_internal.h"

namespace mx {

// Device status word (one per device): bounded device-side waits OR an error code in.
__device__ uint32_t g_mx_status;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int num_sms = 0;
    uint32_t* status = nullptr;
    bool ready = false;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MX_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mx_status) != cudaSuccess) return MX_ERR_CUDA;
        d.status = static_cast<uint32_t*>(p);
        if (g_encode == nullptr) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return MX_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return MX_OK;
}

// NVTX ranges (domain "mxfp4moe") around each call's launch sequence and each phase of a
// forward, so a timeline profiler shows which launches belong to which step. They mark the
// host side only; without a profiler attached a range costs a null-pointer check.
nvtxDomainHandle_t nvtx_domain() {
    static nvtxDomainHandle_t d = nvtxDomainCreateA("mxfp4moe");
    return d;
}

struct NvtxRange {
    explicit NvtxRange(const char* name) {
        nvtxEventAttributes_t a;
        std::memset(&a, 0, sizeof(a));
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(nvtx_domain(), &a);
    }
    ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D uint8 tensor [rows, inner_bytes] read in boxes of [box_rows, 128 bytes], 128-byte swizzle.
int make_tmap(CUtensorMap* m, const void* base, int64_t inner_bytes, int64_t rows, uint32_t box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)inner_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)inner_bytes};
    cuuint32_t box[2] = {128u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// Stacked gate/up weights w13 [E][2I][H/2] viewed as [E][2][I][H/2] (4-D, innermost first
// in the map): one box of 128 bytes x box_rows rows x both halves brings the gate rows of an
// N tile and the matching up rows in a single TMA load, 128-byte swizzle.
int make_tmap_w13(CUtensorMap* m, const void* base, int64_t H, int64_t I, int64_t E, uint32_t box_rows) {
    const cuuint64_t row = (cuuint64_t)(H / 2);
    cuuint64_t dims[4] = {row, (cuuint64_t)I, 2, (cuuint64_t)E};
    cuuint64_t strides[3] = {row, row * (cuuint64_t)I, row * (cuuint64_t)I * 2};
    cuuint32_t box[4] = {128u, box_rows, 2u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// E2M1 codes [rows, K/2 bytes] read as K 4-bit elements per row through the type that spreads
// each 8 bytes of 16 codes over 16 bytes of shared memory (the layout kind::mxf8f6f4 reads):
// boxes of 128 elements (128 bytes in shared memory) x box_rows, 128-byte swizzle. The base
// must be 32-byte aligned and K a multiple of 128.
int make_tmap_fp4s(CUtensorMap* m, const void* base, int64_t K, int64_t rows, uint32_t box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// The stacked w13 of make_tmap_w13 in that spread form: [E][2][I][H] elements.
int make_tmap_w13_fp4s(CUtensorMap* m, const void* base, int64_t H, int64_t I, int64_t E, uint32_t box_rows) {
    const cuuint64_t row = (cuuint64_t)(H / 2);
    cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)E};
    cuuint64_t strides[3] = {row, row * (cuuint64_t)I, row * (cuuint64_t)I * 2};
    cuuint32_t box[4] = {128u, box_rows, 2u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// 2-D output [rows, cols] written in boxes of 32 rows x box_bytes (32: 16 BF16 or 32 code
// bytes; 16: 16 code bytes). BF16 boxes use the 32-byte swizzle: in shared memory the two
// 16-byte halves of box row r trade places when bit 2 of r is set, so that the 32 lanes of
// a warp, each writing one row, spread over all banks (the GEMM epilogue writes them so).
int make_tmap_out(CUtensorMap* m, void* base, int64_t cols, int64_t rows, bool bf16 = true, uint32_t box_bytes = 32) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * (bf16 ? 2 : 1)};
    cuuint32_t box[2] = {bf16 ? box_bytes / 2 : box_bytes, 32u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          bf16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Bytes of a scale tensor [rows, kb] in the tile layout (128-row groups x 4-byte K-words).
size_t tiled_bytes(int64_t rows, int64_t kb) { return (size_t)((rows + 127) / 128) * (size_t)(kb / 4) * 512; }

// Workspace layout shared by moe_mxfp4_forward (and its persistent form), moe_nvfp4_forward
// (sf_div 16: one scale per 16 columns) and moe_mxfp4_route. The status word comes first, at
// offset 0, where mx_check_workspace finds it; the persistent forward's grid-barrier counter
// follows at 256.
constexpr size_t kWsStatusOff = 0;
constexpr size_t kWsSyncOff = 256;
struct WsLayout {
    int64_t R = 0, nchunks = 0, max_mtiles = 0;
    size_t status = 0, sync = 0, num_mtiles = 0, counts = 0, offsets = 0, chunk_counts = 0, chunk_base = 0, local_rank = 0,
           row_of = 0, tile_expert = 0, tile_row0 = 0, tile_rows = 0, tile_base = 0, xq = 0, xs = 0, hq = 0, hs = 0,
           y = 0, total = 0;
};

// code_div: activation elements per code byte (2 for E2M1, 1 for the MXFP8 path's E4M3).
WsLayout ws_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, bool routed, int sf_div = 32,
                   int code_div = 2) {
    WsLayout L;
    L.R = routed ? T * K : T;
    L.nchunks = routed ? (L.R + kRouteChunk - 1) / kRouteChunk : 0;
    L.max_mtiles = (L.R + kBM - 1) / kBM + (routed ? E : 0);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    L.status = take(16);
    L.sync = take(16);
    L.num_mtiles = take(16);
    if (routed) {
        L.counts = take(4 * (size_t)E);
        L.offsets = take(4 * (size_t)(E + 1));
        L.chunk_counts = take(4 * (size_t)(L.nchunks * E));
        L.chunk_base = take(4 * (size_t)(L.nchunks * E));
        L.local_rank = take(4 * (size_t)L.R);
        L.row_of = take(4 * (size_t)L.R);
        L.tile_expert = take(4 * (size_t)L.max_mtiles);
        L.tile_row0 = take(4 * (size_t)L.max_mtiles);
        L.tile_rows = take(4 * (size_t)L.max_mtiles);
        L.tile_base = take(4 * (size_t)(E + 1));
    }
    // The routed MXFP4 and NVFP4 forwards (code_div 2) keep xs and hs stage-major: whole M
    // tiles x K stages x 2 (MXFP4) or 4 (NVFP4) 512-byte words, which also holds them row-major
    const bool stage_major = routed && code_div == 2;
    const size_t words = sf_div == 16 ? 4 : 2;
    auto scale_bytes = [&](int64_t cols) {
        return stage_major ? (size_t)L.max_mtiles * (size_t)((cols + kBK - 1) / kBK) * words * 512
                           : (size_t)L.R * (size_t)(cols / sf_div);
    };
    L.xq = take((size_t)L.R * (size_t)(H / code_div));
    L.xs = take(scale_bytes(H));
    L.hq = take((size_t)L.R * (size_t)(I / code_div));
    L.hs = take(scale_bytes(I));
    if (routed) L.y = take((size_t)L.R * (size_t)H * 2);
    L.total = off;
    return L;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

RouteBufs route_bufs(void* ws, const WsLayout& L) {
    RouteBufs rb;
    rb.chunk_counts = at<int32_t>(ws, L.chunk_counts);
    rb.chunk_base = at<int32_t>(ws, L.chunk_base);
    rb.local_rank = at<int32_t>(ws, L.local_rank);
    rb.counts = at<int32_t>(ws, L.counts);
    rb.offsets = at<int32_t>(ws, L.offsets);
    rb.row_of = at<int32_t>(ws, L.row_of);
    rb.tile_expert = at<int32_t>(ws, L.tile_expert);
    rb.tile_row0 = at<int32_t>(ws, L.tile_row0);
    rb.tile_rows = at<int32_t>(ws, L.tile_rows);
    rb.num_mtiles = at<int32_t>(ws, L.num_mtiles);
    rb.tile_base = at<int32_t>(ws, L.tile_base);
    rb.nchunks = L.nchunks;
    return rb;
}

int check_moe_dims(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, bool routed) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0) return MX_ERR_INVALID_ARG;
    if (routed && K <= 0) return MX_ERR_INVALID_ARG;
    if (H % 128 || I % 128) return MX_ERR_UNSUPPORTED;
    if (E > kMaxExperts || (routed && K > kMaxTopK)) return MX_ERR_UNSUPPORTED;
    if (!routed && E != 1) return MX_ERR_INVALID_ARG;
    if (H >= (int64_t)1 << 24 || I >= (int64_t)1 << 24) return MX_ERR_UNSUPPORTED;
    const int64_t R = routed ? T * K : T;
    if (R >= ((int64_t)1 << 31) - (int64_t)kBM * (E + 1)) return MX_ERR_UNSUPPORTED;
    if (E * 2 * I >= ((int64_t)1 << 31) || E * H >= ((int64_t)1 << 31)) return MX_ERR_UNSUPPORTED;
    return MX_OK;
}

// Fill the GEMM arguments shared by L1 and L2; waits that run out report to the device-wide
// word (a forward adds its workspace word).
GemmArgs base_args(const uint8_t* sfa, const uint8_t* sfb, int64_t K, int64_t a_rows, int64_t b_rows,
                   uint32_t* dev_status) {
    GemmArgs g;
    std::memset(&g, 0, sizeof(g));
    g.sfa = sfa;
    g.sfb = sfb;
    g.ld_sf = K / 32;
    g.a_rows = a_rows;
    g.b_rows = b_rows;
    g.b_groups = (b_rows + 127) / 128;
    g.kw = K / 128;
    g.k_tiles = (int32_t)((K + kBK - 1) / kBK);
    g.k_tail_half = (K % kBK) != 0 ? 1 : 0;
    g.status = StatusWords{nullptr, dev_status};
    return g;
}

// A float32 global scale the NVFP4 quantiser accepts: finite and in [2^-117, 2^100], so that
// 1 / (6 g), e4m3(scale) * g and its reciprocal are normal floats.
bool nv_global_ok(float g) { return g >= 0x1p-117f && g <= 0x1p100f; }

int grid_for(int64_t work, int num_sms) {
    int64_t g = work < num_sms ? work : num_sms;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace mx

using namespace mx;

extern "C" {

const char* mx_status_string(int s) {
    switch (s) {
        case MX_OK: return "MX_OK";
        case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
        case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
        case MX_ERR_MISALIGNED: return "MX_ERR_MISALIGNED";
        case MX_ERR_WORKSPACE: return "MX_ERR_WORKSPACE";
        case MX_ERR_CUDA: return "MX_ERR_CUDA";
        case MX_ERR_DEVICE_TIMEOUT: return "MX_ERR_DEVICE_TIMEOUT";
        default: return "MX_ERR_UNKNOWN";
    }
}

int mx_version(void) { return 100; }

int mx_selftest_wait_timeout(mx_stream_t stream) {
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_wait_probe(StatusWords{nullptr, d->status}, static_cast<cudaStream_t>(stream)));
}

int mx_selftest_wait_timeout_ws(void* workspace, mx_stream_t stream) {
    if (!workspace) return MX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_wait_probe(StatusWords{static_cast<uint32_t*>(workspace), d->status},
                                         static_cast<cudaStream_t>(stream)));
}

int mx_selftest_grid_barrier_timeout(void* workspace, mx_stream_t stream) {
    if (!workspace) return MX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* counter = at<uint32_t>(workspace, kWsSyncOff);
    if (cudaMemsetAsync(counter, 0, sizeof(uint32_t), s) != cudaSuccess) return MX_ERR_CUDA;
    return cuda_status(
        launch_grid_sync_probe(counter, StatusWords{at<uint32_t>(workspace, kWsStatusOff), d->status}, s));
}

int mx_check_workspace(const void* workspace, int clear, mx_stream_t stream) {
    if (!workspace) return MX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MX_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    // ordered after the stream's work; the wait covers this stream only
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MX_ERR_CUDA;
    if (clear && v != 0 && cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(v), s) != cudaSuccess)
        return MX_ERR_CUDA;
    return v ? MX_ERR_DEVICE_TIMEOUT : MX_OK;
}

int mx_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return MX_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_mx_status, sizeof(v)) != cudaSuccess) return MX_ERR_CUDA;
    if (clear) {
        const uint32_t z = 0;
        if (cudaMemcpyToSymbol(g_mx_status, &z, sizeof(z)) != cudaSuccess) return MX_ERR_CUDA;
    }
    return v ? MX_ERR_DEVICE_TIMEOUT : MX_OK;
}

int mxfp4_dequant(const uint8_t* codes, const uint8_t* sf, void* out_bf16, int64_t rows, int64_t cols,
                  mx_stream_t stream) {
    if (rows < 0 || cols <= 0) return MX_ERR_INVALID_ARG;
    if (cols % 32) return MX_ERR_UNSUPPORTED;
    if (rows == 0) return MX_OK;
    if (!codes || !sf || !out_bf16) return MX_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(out_bf16)) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_mxfp4_dequant(codes, sf, static_cast<uint16_t*>(out_bf16), rows, cols, d->num_sms,
                                            static_cast<cudaStream_t>(stream)));
}

int nvfp4_dequant(const uint8_t* codes, const uint8_t* sf_e4m3, float global_scale, void* out_bf16, int64_t rows,
                  int64_t cols, mx_stream_t stream) {
    if (rows < 0 || cols <= 0) return MX_ERR_INVALID_ARG;
    if (cols % 16) return MX_ERR_UNSUPPORTED;
    if (rows == 0) return MX_OK;
    if (!codes || !sf_e4m3 || !out_bf16) return MX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(codes) & 7u) != 0 || !aligned16(out_bf16)) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_nvfp4_dequant(codes, sf_e4m3, global_scale, static_cast<uint16_t*>(out_bf16), rows,
                                            cols, d->num_sms, static_cast<cudaStream_t>(stream)));
}

int fp8_block_dequant_128x128(const uint8_t* q, const uint8_t* sf, void* out_bf16, int64_t rows, int64_t cols,
                              mx_stream_t stream) {
    if (rows < 0 || cols <= 0) return MX_ERR_INVALID_ARG;
    if (cols % 16) return MX_ERR_UNSUPPORTED;
    if (rows == 0) return MX_OK;
    if (!q || !sf || !out_bf16) return MX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out_bf16)) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_fp8_dequant(q, sf, static_cast<uint16_t*>(out_bf16), rows, cols, d->num_sms,
                                          static_cast<cudaStream_t>(stream)));
}

int act_quant_nvfp4(const void* x_bf16, float global_scale, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K,
                    mx_stream_t stream) {
    if (M < 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (!nv_global_ok(global_scale)) return MX_ERR_INVALID_ARG;
    if (K % 16) return MX_ERR_UNSUPPORTED;
    if (M == 0) return MX_OK;
    if (!x_bf16 || !codes || !sf) return MX_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || (reinterpret_cast<uintptr_t>(codes) & 7u) != 0) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_act_quant_nvfp4(static_cast<const uint16_t*>(x_bf16), global_scale, codes, sf, M, K,
                                              d->num_sms, static_cast<cudaStream_t>(stream)));
}

int nvfp4_calibrate_global(const void* x_bf16, int64_t M, int64_t K, float* amax, float* global_scale,
                           mx_stream_t stream) {
    if (M < 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (!amax || !global_scale || (M > 0 && !x_bf16)) return MX_ERR_INVALID_ARG;
    if ((M > 0 && !aligned16(x_bf16)) || (reinterpret_cast<uintptr_t>(amax) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(global_scale) & 3u) != 0)
        return MX_ERR_MISALIGNED;
    if (M > ((int64_t)1 << 40) / K) return MX_ERR_UNSUPPORTED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_nv_calibrate(static_cast<const uint16_t*>(x_bf16), M * K, amax, global_scale,
                                           d->num_sms, static_cast<cudaStream_t>(stream)));
}

int act_quant_mxfp4(const void* x_bf16, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K, mx_stream_t stream) {
    if (M < 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (K % 32) return MX_ERR_UNSUPPORTED;
    if (M == 0) return MX_OK;
    if (!x_bf16 || !codes || !sf) return MX_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(codes)) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_act_quant(static_cast<const uint16_t*>(x_bf16), codes, sf, M, K, d->num_sms,
                                        static_cast<cudaStream_t>(stream)));
}

int act_quant_mxfp8(const void* x_bf16, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K, mx_stream_t stream) {
    if (M < 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (K % 32) return MX_ERR_UNSUPPORTED;
    if (M == 0) return MX_OK;
    if (!x_bf16 || !codes || !sf) return MX_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(codes)) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    return cuda_status(launch_act_quant_mxfp8(static_cast<const uint16_t*>(x_bf16), codes, sf, M, K, d->num_sms,
                                              static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_tiled_scales_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols <= 0 || cols % 128) return 0;
    return tiled_bytes(rows, cols / 32);
}

int mxfp4_scales_to_tiled(const uint8_t* sf, uint8_t* out, int64_t rows, int64_t cols, mx_stream_t stream) {
    if (rows < 0 || cols <= 0) return MX_ERR_INVALID_ARG;
    if (cols % 128) return MX_ERR_UNSUPPORTED;
    if (rows == 0) return MX_OK;
    if (!sf || !out) return MX_ERR_INVALID_ARG;
    if (!aligned16(sf) || !aligned16(out)) return MX_ERR_MISALIGNED;
    if ((cols / 128 + 31) / 32 > 65535) return MX_ERR_UNSUPPORTED;
    return cuda_status(launch_sf_tile(sf, out, rows, cols / 32, static_cast<cudaStream_t>(stream)));
}

size_t nvfp4_tiled_scales_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols <= 0 || cols % 64) return 0;
    return tiled_bytes(rows, cols / 16);
}

int nvfp4_scales_to_tiled(const uint8_t* sf, uint8_t* out, int64_t rows, int64_t cols, mx_stream_t stream) {
    if (rows < 0 || cols <= 0) return MX_ERR_INVALID_ARG;
    if (cols % 64) return MX_ERR_UNSUPPORTED;
    if (rows == 0) return MX_OK;
    if (!sf || !out) return MX_ERR_INVALID_ARG;
    if (!aligned16(sf) || !aligned16(out)) return MX_ERR_MISALIGNED;
    if ((cols / 64 + 31) / 32 > 65535) return MX_ERR_UNSUPPORTED;
    return cuda_status(launch_sf_tile(sf, out, rows, cols / 16, static_cast<cudaStream_t>(stream)));
}

int nvfp4_gemm_bf16(const uint8_t* a, const uint8_t* sa, float a_global, const uint8_t* b, const uint8_t* sb_tiled,
                    float b_global, void* d_bf16, int64_t M, int64_t N, int64_t K, mx_stream_t stream) {
    return nvfp4_gemm_bf16_multi(a, sa, a_global, b, sb_tiled, &b_global, &N, 1, d_bf16, M, K, stream);
}

int nvfp4_gemm_bf16_multi(const uint8_t* a, const uint8_t* sa, float a_global, const uint8_t* b,
                          const uint8_t* sb_tiled, const float* b_globals, const int64_t* seg_rows, int nseg,
                          void* d_bf16, int64_t M, int64_t K, mx_stream_t stream) {
    if (!b_globals || !seg_rows || nseg < 1) return MX_ERR_INVALID_ARG;
    if (nseg > kMaxSegments) return MX_ERR_UNSUPPORTED;
    int64_t N = 0;
    for (int i = 0; i < nseg; ++i) {
        if (seg_rows[i] <= 0) return MX_ERR_INVALID_ARG;
        if (seg_rows[i] % 16) return MX_ERR_UNSUPPORTED;
        if (seg_rows[i] >= ((int64_t)1 << 31)) return MX_ERR_UNSUPPORTED;
        N += seg_rows[i];
    }
    if (M < 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (K % 128) return MX_ERR_UNSUPPORTED;
    if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 24)) return MX_ERR_UNSUPPORTED;
    if (M == 0) return MX_OK;
    if (!a || !sa || !b || !sb_tiled || !d_bf16) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(sa) || !aligned16(sb_tiled) || !aligned16(d_bf16))
        return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    CUtensorMap ta, tb, ty;
    if (make_tmap(&ta, a, K / 2, M, 128) || make_tmap(&tb, b, K / 2, N, 256) || make_tmap_out(&ty, d_bf16, N, M))
        return MX_ERR_CUDA;
    GemmArgs g = base_args(sa, sb_tiled, K, M, N, d->status);
    g.ld_sf = K / 16;                  // one E4M3 scale per 16 elements
    g.kw = K / 64;                     // scale words (4 scales) per row
    g.alpha = a_global * b_globals[0];
    if (nseg > 1) {                    // a fused projection: one scale per segment of columns
        int64_t end = 0;
        g.nseg = nseg;
        for (int i = 0; i < nseg; ++i) {
            end += seg_rows[i];
            g.seg_end[i] = (int32_t)end;
            g.seg_alpha[i] = a_global * b_globals[i];
        }
    }
    g.num_mtiles_host = (int32_t)((M + kBM - 1) / kBM);
    g.m_total = M;
    g.n_tiles = (int32_t)((N + kBN - 1) / kBN);
    g.b_rows_per_expert = N;
    g.n_valid = N;
    g.y = static_cast<uint16_t*>(d_bf16);
    g.ld_y = N;
    return cuda_status(launch_gemm_nvfp4(ta, tb, ty, g, grid_for((int64_t)g.num_mtiles_host * g.n_tiles, d->num_sms),
                                         static_cast<cudaStream_t>(stream)));
}

// N tile width for a GEMM whose 256-wide tiling has units256 work units: 128 when those
// would leave SMs idle.
int tile_cols(int64_t units256, int num_sms) { return units256 < num_sms ? 128 : kBN; }

int mxfp4_gemm_bf16(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb, void* d_bf16,
                    int64_t M, int64_t N, int64_t K, mx_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (K % 128 || N % 16) return MX_ERR_UNSUPPORTED;
    if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 24)) return MX_ERR_UNSUPPORTED;
    if (M == 0) return MX_OK;
    if (!a || !sa || !b || !sb || !d_bf16) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(sa) || !aligned16(sb) || !aligned16(d_bf16))
        return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    const int64_t mtiles = (M + kBM - 1) / kBM;
    const int nw = tile_cols(mtiles * ((N + kBN - 1) / kBN), d->num_sms);
    CUtensorMap ta, tb, ty;
    if (make_tmap(&ta, a, K / 2, M, 128) || make_tmap(&tb, b, K / 2, N, (uint32_t)nw) || make_tmap_out(&ty, d_bf16, N, M))
        return MX_ERR_CUDA;
    GemmArgs g = base_args(sa, sb, K, M, N, d->status);
    g.num_mtiles_host = (int32_t)mtiles;
    g.m_total = M;
    g.n_tiles = (int32_t)((N + nw - 1) / nw);
    g.b_rows_per_expert = N;
    g.n_valid = N;
    g.y = static_cast<uint16_t*>(d_bf16);
    g.ld_y = N;
    return cuda_status(launch_gemm_l2(ta, tb, ty, g, grid_for((int64_t)g.num_mtiles_host * g.n_tiles, d->num_sms), true,
                                      nw, static_cast<cudaStream_t>(stream)));
}

int mxfp8_mxfp4_gemm_bf16(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb_tiled,
                          void* d_bf16, int64_t M, int64_t N, int64_t K, mx_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0) return MX_ERR_INVALID_ARG;
    if (K % 128 || N % 16) return MX_ERR_UNSUPPORTED;
    if (M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 24)) return MX_ERR_UNSUPPORTED;
    if (M == 0) return MX_OK;
    if (!a || !sa || !b || !sb_tiled || !d_bf16) return MX_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned32(b) || !aligned16(sa) || !aligned16(sb_tiled) || !aligned16(d_bf16))
        return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    CUtensorMap ta, tb, ty;
    if (make_tmap(&ta, a, K, M, 128) || make_tmap_fp4s(&tb, b, K, N, 256) || make_tmap_out(&ty, d_bf16, N, M))
        return MX_ERR_CUDA;
    GemmArgs g = base_args(sa, sb_tiled, K, M, N, d->status);
    g.k_tiles = (int32_t)(K / 128);
    g.k_tail_half = 0;
    g.num_mtiles_host = (int32_t)((M + kBM - 1) / kBM);
    g.m_total = M;
    g.n_tiles = (int32_t)((N + kBN - 1) / kBN);
    g.b_rows_per_expert = N;
    g.n_valid = N;
    g.y = static_cast<uint16_t*>(d_bf16);
    g.ld_y = N;
    return cuda_status(launch_gemm_a8(ta, tb, ty, g, grid_for((int64_t)g.num_mtiles_host * g.n_tiles, d->num_sms),
                                      false, static_cast<cudaStream_t>(stream)));
}

size_t moe_mxfp4_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed) {
    if (check_moe_dims(T, H, I, E, K, routed != 0) != MX_OK) return 0;
    return ws_layout(T, H, I, E, K, routed != 0).total;
}

int moe_mxfp4_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed, int64_t* out) {
    if (!out) return MX_ERR_INVALID_ARG;
    if (int e = check_moe_dims(T, H, I, E, K, routed != 0)) return e;
    const WsLayout L = ws_layout(T, H, I, E, K, routed != 0);
    out[0] = (int64_t)L.xq;
    out[1] = (int64_t)L.xs;
    out[2] = (int64_t)L.hq;
    out[3] = (int64_t)L.hs;
    out[4] = routed ? (int64_t)L.y : -1;
    out[5] = routed ? (int64_t)L.row_of : -1;
    out[6] = routed ? (int64_t)L.counts : -1;
    out[7] = routed ? (int64_t)L.offsets : -1;
    return MX_OK;
}

int moe_mxfp4_route(const int32_t* topk_ids, int64_t T, int64_t K, int64_t E, int32_t* counts, int32_t* offsets,
                    int32_t* row_of, void* workspace, size_t ws_bytes, mx_stream_t stream) {
    if (T < 0 || K <= 0 || E <= 0) return MX_ERR_INVALID_ARG;
    if (E > kMaxExperts || K > kMaxTopK) return MX_ERR_UNSUPPORTED;
    if (T * K >= ((int64_t)1 << 31) - (int64_t)kBM * (E + 1)) return MX_ERR_UNSUPPORTED;
    if (!counts || !offsets || !row_of) return MX_ERR_INVALID_ARG;
    if (T > 0 && !topk_ids) return MX_ERR_INVALID_ARG;
    // the routing part of the forward's workspace; H = I = 128 keeps the size check simple
    const WsLayout L = ws_layout(T, 128, 128, E, K, true);
    if (!workspace || ws_bytes < L.total) return MX_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MX_ERR_MISALIGNED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    RouteBufs rb = route_bufs(workspace, L);
    rb.counts = counts;
    rb.offsets = offsets;
    rb.row_of = row_of;
    if (T == 0) {
        if (cudaMemsetAsync(counts, 0, 4 * (size_t)E, s) != cudaSuccess) return MX_ERR_CUDA;
        return cuda_status(cudaMemsetAsync(offsets, 0, 4 * (size_t)(E + 1), s));
    }
    if (cudaError_t e = launch_route(topk_ids, T, K, E, rb, s)) return MX_ERR_CUDA;
    // row_of needs the gather pass; run it without writing activations (H = 0 columns)
    return cuda_status(launch_quant_gather(nullptr, topk_ids, T, K, E, 0, rb, nullptr, nullptr, s));
}

}  // extern "C"

namespace {

// The NVFP4 forward's extra inputs: per-expert weight globals (g13 [E][2] gate, up; g2 [E],
// device float32) and the two activation globals.
struct NvGlobals {
    const float* g13;
    const float* g2;
    float x_global;
    float h_global;
};

int forward_impl(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                 const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, void* out, int64_t T, int64_t H,
                 int64_t I, int64_t E, int64_t K, void* workspace, size_t ws_bytes, mx_stream_t stream,
                 void* const* events, bool scales_tiled, const NvGlobals* nv = nullptr, bool fused = false,
                 bool a8 = false) {
    const bool routed = topk_ids != nullptr;
    if (routed != (topk_w != nullptr)) return MX_ERR_INVALID_ARG;
    if (int e = check_moe_dims(T, H, I, E, K, routed)) return e;
    if (nv && (!nv_global_ok(nv->x_global) || !nv_global_ok(nv->h_global))) return MX_ERR_INVALID_ARG;
    if (T == 0) return MX_OK;
    if (!x || !w13 || !s13 || !w2 || !s2 || !out) return MX_ERR_INVALID_ARG;
    if (nv && (!nv->g13 || !nv->g2)) return MX_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w13) || !aligned16(s13) || !aligned16(w2) || !aligned16(s2) ||
        !aligned16(out))
        return MX_ERR_MISALIGNED;
    if (a8 && (!aligned32(w13) || !aligned32(w2))) return MX_ERR_MISALIGNED;
    const int sf_div = nv ? 16 : 32;
    const int code_div = a8 ? 1 : 2;
    const WsLayout L = ws_layout(T, H, I, E, K, routed, sf_div, code_div);
    if (!workspace || ws_bytes < L.total) return MX_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MX_ERR_MISALIGNED;
    DeviceInfo* d;
    if (int e = device_info(&d)) return e;
    const NvtxRange range(fused ? "moe_mxfp4_forward_fused"
                          : nv  ? "moe_nvfp4_forward"
                          : a8  ? "moe_mxfp4w_mxfp8a_forward"
                                : "moe_mxfp4_forward");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto mark = [&](int i) -> bool {
        return !(events && events[i]) || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
    };
    uint8_t* xq = at<uint8_t>(workspace, L.xq);
    uint8_t* xs = at<uint8_t>(workspace, L.xs);
    uint8_t* hq = at<uint8_t>(workspace, L.hq);
    uint8_t* hs = at<uint8_t>(workspace, L.hs);
    // The forward's status word: its first kernel clears it, its GEMMs' waits set it.
    uint32_t* ws_status = at<uint32_t>(workspace, L.status);
    const int64_t R = L.R;

    GemmArgs g1 = base_args(xs, s13, H, R, E * 2 * I, d->status);
    GemmArgs g2 = base_args(hs, s2, I, R, E * H, d->status);
    g1.status.ws = g2.status.ws = ws_status;
    if (nv) {
        // one E4M3 scale per 16 elements: four per 4-byte word
        g1.ld_sf = H / 16;
        g1.kw = H / 64;
        g1.alpha = nv->x_global;
        g1.w_global = nv->g13;
        g1.q_global = nv->h_global;
        g2.ld_sf = I / 16;
        g2.kw = I / 64;
        g2.alpha = nv->h_global;
        g2.w_global = nv->g2;
    }
    RouteBufs rb{};
    if (routed) {
        rb = route_bufs(workspace, L);
        for (GemmArgs* g : {&g1, &g2}) {
            g->tile_expert = rb.tile_expert;
            g->tile_row0 = rb.tile_row0;
            g->tile_rows = rb.tile_rows;
            g->num_mtiles_dev = rb.num_mtiles;
        }
    } else {
        for (GemmArgs* g : {&g1, &g2}) {
            g->num_mtiles_host = (int32_t)((T + kBM - 1) / kBM);
            g->m_total = T;
        }
    }
    const int64_t max_mtiles = L.max_mtiles;

    // Tile widths: 256 columns, or 128 where 256-wide tiles would leave SMs idle. Only with
    // uniform tiling: the routed tile count is known on the device alone, and its bound
    // max_mtiles counts an extra tile per expert. NVFP4 runs 256-column tiles only. The
    // persistent forward runs both GEMMs through one pipeline, so one width for both.
    int n1 = routed || nv || a8 ? kBN : tile_cols(max_mtiles * (I / 128), d->num_sms);
    int n2 = routed || nv || a8 ? kBN : tile_cols(max_mtiles * ((H + kBN - 1) / kBN), d->num_sms);
    if (fused && (n1 == 128 || n2 == 128)) n1 = n2 = 128;

    // L1: [R, H] x [2I, H]^T per expert, fused SiLU(gate) * up and MX re-quant.
    CUtensorMap ta1, tb1, ty1, ta2, tb2, ty2;
    if (a8) {
        // E4M3 activations (one byte per element), E2M1 weights spread for kind::mxf8f6f4
        if (make_tmap(&ta1, xq, H, R, 128) || make_tmap_w13_fp4s(&tb1, w13, H, I, E, (uint32_t)(n1 / 2)) ||
            make_tmap_out(&ty1, hq, I, R, false, 32u))
            return MX_ERR_CUDA;
        g1.k_tiles = (int32_t)(H / 128);
        g1.k_tail_half = 0;
        g2.k_tiles = (int32_t)(I / 128);
        g2.k_tail_half = 0;
    } else if (make_tmap(&ta1, xq, H / 2, R, 128) || make_tmap_w13(&tb1, w13, H, I, E, (uint32_t)(n1 / 2)) ||
               make_tmap_out(&ty1, hq, I / 2, R, false, n1 == 128 ? 16u : 32u)) {
        return MX_ERR_CUDA;
    }
    g1.n_tiles = (int32_t)(I / (n1 / 2));
    g1.b_rows_per_expert = 2 * I;
    g1.n_half = I;
    g1.n_valid = I;
    g1.hq = hq;
    g1.hs = hs;
    g1.ld_hq = I / code_div;
    g1.ld_hs = I / sf_div;
    // L2: [R, I] x [H, I]^T per expert, BF16 out (to `out` directly without routing).
    if (a8 ? (make_tmap(&ta2, hq, I, R, 128) || make_tmap_fp4s(&tb2, w2, I, E * H, (uint32_t)n2))
           : (make_tmap(&ta2, hq, I / 2, R, 128) || make_tmap(&tb2, w2, I / 2, E * H, (uint32_t)n2)))
        return MX_ERR_CUDA;
    g2.n_tiles = (int32_t)((H + n2 - 1) / n2);
    g2.b_rows_per_expert = H;
    g2.n_valid = H;
    g2.y = routed ? at<uint16_t>(workspace, L.y) : static_cast<uint16_t*>(out);
    g2.ld_y = H;
    if (make_tmap_out(&ty2, g2.y, H, R)) return MX_ERR_CUDA;

    if (fused) {
        if (nv || a8) return MX_ERR_UNSUPPORTED;
        FusedArgs fa;
        std::memset(&fa, 0, sizeof(fa));
        fa.g1 = g1;
        fa.g2 = g2;
        fa.x = static_cast<const uint16_t*>(x);
        fa.ids = topk_ids;
        fa.topk_w = topk_w;
        fa.out = static_cast<uint16_t*>(out);
        fa.y = g2.y;
        fa.xq = xq;
        fa.xs = xs;
        fa.rb = rb;
        fa.T = T;
        fa.H = H;
        fa.K = (int32_t)(routed ? K : 1);
        fa.E = (int32_t)E;
        fa.sync = at<uint32_t>(workspace, L.sync);
        fa.clear_word = ws_status;
        fa.status = g1.status;
        if (cudaMemsetAsync(fa.sync, 0, sizeof(uint32_t), s) != cudaSuccess) return MX_ERR_CUDA;
        return cuda_status(launch_moe_fused(ta1, tb1, ty1, ta2, tb2, ty2, fa, n1, d->num_sms, s));
    }

    // Routed MXFP4 and NVFP4: x's and h's scales stage-major, in the order the GEMMs' scale
    // loaders read them. (Without routing the stage-major writes cost the short quantiser more
    // than the GEMMs gain.)
    const bool stage_major = routed && !a8;
    const int64_t sm_k_tiles = stage_major ? g1.k_tiles : 0;
    g1.a_sm = g2.a_sm = stage_major ? 1 : 0;
    g1.hs_k_tiles = stage_major ? g2.k_tiles : 0;
    if (!mark(0)) return MX_ERR_CUDA;
    if (routed) {
        const NvtxRange r("route + quantise");
        if (launch_route(topk_ids, T, K, E, rb, s, ws_status) != cudaSuccess || !mark(1)) return MX_ERR_CUDA;
        if (launch_quant_gather(static_cast<const uint16_t*>(x), topk_ids, T, K, E, H, rb, xq, xs, s,
                                nv ? 1 : (a8 ? 2 : 0), nv ? nv->x_global : 0.0f, sm_k_tiles) != cudaSuccess)
            return MX_ERR_CUDA;
    } else {
        const NvtxRange r("quantise");
        if (!mark(1)) return MX_ERR_CUDA;
        const uint16_t* xb = static_cast<const uint16_t*>(x);
        const cudaError_t qe = nv ? launch_act_quant_nvfp4(xb, nv->x_global, xq, xs, T, H, d->num_sms, s, ws_status)
                               : a8 ? launch_act_quant_mxfp8(xb, xq, xs, T, H, d->num_sms, s, ws_status)
                                    : launch_act_quant(xb, xq, xs, T, H, d->num_sms, s, ws_status, sm_k_tiles);
        if (qe != cudaSuccess) return MX_ERR_CUDA;
    }
    if (!mark(2)) return MX_ERR_CUDA;
    const NvtxRange r_gemm("L1 + L2 + combine");
    const int grid1 = grid_for(max_mtiles * g1.n_tiles, d->num_sms);
    if ((nv   ? launch_gemm_nvfp4_l1(ta1, tb1, ty1, g1, grid1, s)
         : a8 ? launch_gemm_a8(ta1, tb1, ty1, g1, grid1, true, s)
              : launch_gemm_l1(ta1, tb1, ty1, g1, grid1, scales_tiled, n1, s)) != cudaSuccess ||
        !mark(3))
        return MX_ERR_CUDA;
    const int grid2 = grid_for(max_mtiles * g2.n_tiles, d->num_sms);
    if ((nv   ? launch_gemm_nvfp4(ta2, tb2, ty2, g2, grid2, s)
         : a8 ? launch_gemm_a8(ta2, tb2, ty2, g2, grid2, false, s)
              : launch_gemm_l2(ta2, tb2, ty2, g2, grid2, scales_tiled, n2, s)) != cudaSuccess ||
        !mark(4))
        return MX_ERR_CUDA;
    if (routed) {
        if (launch_combine(at<uint16_t>(workspace, L.y), rb.row_of, topk_w, static_cast<uint16_t*>(out), T, K, H,
                           d->num_sms, s) != cudaSuccess)
            return MX_ERR_CUDA;
    }
    return mark(5) ? MX_OK : MX_ERR_CUDA;
}

}  // namespace

extern "C" {

int moe_mxfp4_forward(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                      const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, void* out, int64_t T, int64_t H,
                      int64_t I, int64_t E, int64_t K, void* workspace, size_t ws_bytes, mx_stream_t stream) {
    return forward_impl(x, topk_ids, topk_w, w13, s13, w2, s2, out, T, H, I, E, K, workspace, ws_bytes, stream,
                        nullptr, false);
}

int moe_mxfp4_forward_tiled(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                            const uint8_t* s13_tiled, const uint8_t* w2, const uint8_t* s2_tiled, void* out,
                            int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, void* workspace,
                            size_t ws_bytes, mx_stream_t stream) {
    return forward_impl(x, topk_ids, topk_w, w13, s13_tiled, w2, s2_tiled, out, T, H, I, E, K, workspace, ws_bytes,
                        stream, nullptr, true);
}

int moe_mxfp4_forward_timed(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                            const uint8_t* s13, const uint8_t* w2, const uint8_t* s2, void* out, int64_t T,
                            int64_t H, int64_t I, int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                            mx_stream_t stream, void* const* events, int scales_tiled) {
    return forward_impl(x, topk_ids, topk_w, w13, s13, w2, s2, out, T, H, I, E, K, workspace, ws_bytes, stream,
                        events, scales_tiled != 0);
}

int moe_mxfp4_forward_fused(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                            const uint8_t* s13_tiled, const uint8_t* w2, const uint8_t* s2_tiled, void* out,
                            int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, void* workspace,
                            size_t ws_bytes, mx_stream_t stream) {
    return forward_impl(x, topk_ids, topk_w, w13, s13_tiled, w2, s2_tiled, out, T, H, I, E, K, workspace, ws_bytes,
                        stream, nullptr, true, nullptr, true);
}

size_t moe_mxfp4w_mxfp8a_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed) {
    if (check_moe_dims(T, H, I, E, K, routed != 0) != MX_OK) return 0;
    return ws_layout(T, H, I, E, K, routed != 0, 32, 1).total;
}

int moe_mxfp4w_mxfp8a_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed,
                                       int64_t* out) {
    if (!out) return MX_ERR_INVALID_ARG;
    if (int e = check_moe_dims(T, H, I, E, K, routed != 0)) return e;
    const WsLayout L = ws_layout(T, H, I, E, K, routed != 0, 32, 1);
    out[0] = (int64_t)L.xq;
    out[1] = (int64_t)L.xs;
    out[2] = (int64_t)L.hq;
    out[3] = (int64_t)L.hs;
    out[4] = routed ? (int64_t)L.y : -1;
    out[5] = routed ? (int64_t)L.row_of : -1;
    out[6] = routed ? (int64_t)L.counts : -1;
    out[7] = routed ? (int64_t)L.offsets : -1;
    return MX_OK;
}

int moe_mxfp4w_mxfp8a_forward_timed(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                                    const uint8_t* s13_tiled, const uint8_t* w2, const uint8_t* s2_tiled, void* out,
                                    int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, void* workspace,
                                    size_t ws_bytes, mx_stream_t stream, void* const* events) {
    return forward_impl(x, topk_ids, topk_w, w13, s13_tiled, w2, s2_tiled, out, T, H, I, E, K, workspace, ws_bytes,
                        stream, events, true, nullptr, false, true);
}

int moe_mxfp4w_mxfp8a_forward(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                              const uint8_t* s13_tiled, const uint8_t* w2, const uint8_t* s2_tiled, void* out,
                              int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, void* workspace,
                              size_t ws_bytes, mx_stream_t stream) {
    return moe_mxfp4w_mxfp8a_forward_timed(x, topk_ids, topk_w, w13, s13_tiled, w2, s2_tiled, out, T, H, I, E, K,
                                           workspace, ws_bytes, stream, nullptr);
}

size_t moe_nvfp4_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed) {
    if (check_moe_dims(T, H, I, E, K, routed != 0) != MX_OK) return 0;
    return ws_layout(T, H, I, E, K, routed != 0, 16).total;
}

int moe_nvfp4_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed, int64_t* out) {
    if (!out) return MX_ERR_INVALID_ARG;
    if (int e = check_moe_dims(T, H, I, E, K, routed != 0)) return e;
    const WsLayout L = ws_layout(T, H, I, E, K, routed != 0, 16);
    out[0] = (int64_t)L.xq;
    out[1] = (int64_t)L.xs;
    out[2] = (int64_t)L.hq;
    out[3] = (int64_t)L.hs;
    out[4] = routed ? (int64_t)L.y : -1;
    out[5] = routed ? (int64_t)L.row_of : -1;
    out[6] = routed ? (int64_t)L.counts : -1;
    out[7] = routed ? (int64_t)L.offsets : -1;
    return MX_OK;
}

int moe_nvfp4_forward_timed(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                            const uint8_t* s13_tiled, const float* g13, const uint8_t* w2, const uint8_t* s2_tiled,
                            const float* g2, float x_global, float h_global, void* out, int64_t T, int64_t H,
                            int64_t I, int64_t E, int64_t K, void* workspace, size_t ws_bytes, mx_stream_t stream,
                            void* const* events) {
    const NvGlobals nv{g13, g2, x_global, h_global};
    return forward_impl(x, topk_ids, topk_w, w13, s13_tiled, w2, s2_tiled, out, T, H, I, E, K, workspace, ws_bytes,
                        stream, events, true, &nv);
}

int moe_nvfp4_forward(const void* x, const int32_t* topk_ids, const float* topk_w, const uint8_t* w13,
                      const uint8_t* s13_tiled, const float* g13, const uint8_t* w2, const uint8_t* s2_tiled,
                      const float* g2, float x_global, float h_global, void* out, int64_t T, int64_t H, int64_t I,
                      int64_t E, int64_t K, void* workspace, size_t ws_bytes, mx_stream_t stream) {
    return moe_nvfp4_forward_timed(x, topk_ids, topk_w, w13, s13_tiled, g13, w2, s2_tiled, g2, x_global, h_global,
                                   out, T, H, I, E, K, workspace, ws_bytes, stream, nullptr);
}

}  // extern "C"
