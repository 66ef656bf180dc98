// mx_elementwise.cu -- HBM-bound kernels: MXFP4 -> BF16 and FP8 E4M3 x E8M0 128x128 -> BF16
// dequantisation, the standalone MX activation quantiser, and the top-k weighted combine.
//
// Weight format per "2026-05-08 DeepSeek V4 Pro NVFP4 Quantization", "Script update:
// dequant_fp8_to_bf16.py now handles ALL compressed types" (item 2: two E2M1 values per
// byte, lower nibble first, LUT x E8M0 per row per 32 columns; item 1: FP8 x E8M0 per
// 128x128 block). Combine per "Current Bug: vLLM produces empty/garbage output", "Phase 1"
// (routing, top-k, scatter) and "Phase 3: Clean up" (the final scatter is BF16).
#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {

namespace {

constexpr int kThreads = 256;

int grid_for(int64_t work_items, int num_sms, int per_sm = 8) {
    int64_t blocks = (work_items + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)num_sms * per_sm;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) { return lo | (hi << 16); }

// One group = 8 logical columns = 4 code bytes; groups are contiguous over the whole tensor
// because cols % 32 == 0, so group g reads codes32[g], scale sf[g / 4] and writes out[g].
__global__ void __launch_bounds__(kThreads) mxfp4_dequant_kernel(const uint32_t* __restrict__ codes32,
                                                                 const uint8_t* __restrict__ sf,
                                                                 uint4* __restrict__ out, int64_t groups) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < groups; g += stride) {
        const uint32_t c = __ldg(codes32 + g);
        const uint32_t s = __ldg(sf + (g >> 2));
        uint32_t o[8];
        if (s == 255u) {
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = (((c >> (4 * i)) & 8u) << 12) | 0x7FC0u;
        } else {
            const float scale = e8m0_value(s);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = f32_to_bf16(e2m1_value((c >> (4 * i)) & 15u) * scale);
        }
        out[g] = make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
    }
}

// E4M3 ("fn") byte -> float32, exact. S.1111.111 is NaN.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float mag;
    if (e == 0) {
        mag = (float)m * 0.001953125f;                        // m * 2^-9
    } else {
        mag = __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) 2^(e-7)
    }
    return (b & 0x80u) ? -mag : mag;
}

// One group = 16 consecutive columns of one row (cols % 16 == 0).
__global__ void __launch_bounds__(kThreads) fp8_dequant_kernel(const uint4* __restrict__ q16,
                                                               const uint8_t* __restrict__ sf,
                                                               uint4* __restrict__ out, int64_t groups,
                                                               int64_t groups_per_row, int64_t sf_cols) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < groups; g += stride) {
        const int64_t row = g / groups_per_row;
        const int64_t col = (g - row * groups_per_row) * 16;
        const uint32_t s = __ldg(sf + (row >> 7) * sf_cols + (col >> 7));
        const uint4 qv = __ldg(q16 + g);
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
        const float scale = (s == 255u) ? 0.0f : e8m0_value(s);
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t b = (w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
            if ((b & 0x7Fu) == 0x7Fu || s == 255u) {
                o[i] = ((b & 0x80u) << 8) | 0x7FC0u;
            } else {
                o[i] = f32_to_bf16(e4m3_value(b) * scale);
            }
        }
        out[2 * g] = make_uint4(pack2(o[0], o[1]), pack2(o[2], o[3]), pack2(o[4], o[5]), pack2(o[6], o[7]));
        out[2 * g + 1] =
            make_uint4(pack2(o[8], o[9]), pack2(o[10], o[11]), pack2(o[12], o[13]), pack2(o[14], o[15]));
    }
}

// One group = 8 elements (16 bytes of BF16); four consecutive lanes form one 32-element
// block. The loop runs in whole warps so the quad shuffles always have all lanes.
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint4* __restrict__ x8,
                                                             uint32_t* __restrict__ codes32,
                                                             uint8_t* __restrict__ sf, int64_t groups) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_stride = (int64_t)gridDim.x * kThreads;
    for (int64_t g0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31); g0 < groups; g0 += warp_stride) {
        const int64_t g = g0 + lane;
        const bool ok = g < groups;
        const uint4 xv = ok ? __ldg(x8 + g) : make_uint4(0, 0, 0, 0);
        uint32_t E;
        const uint32_t packed = mx_quant8_quad(xv, E);
        if (ok) {
            codes32[g] = packed;
            if ((g & 3) == 0) sf[g >> 2] = (uint8_t)E;
        }
    }
}

// out[t, c] = bf16( sum_k w[t,k] * y[row_of[t,k], c] ), float32, slot order, no FMA.
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint4* __restrict__ y8,
                                                           const int32_t* __restrict__ row_of,
                                                           const float* __restrict__ w,
                                                           uint4* __restrict__ out8, int64_t groups,
                                                           int64_t groups_per_row, int K) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t g = (int64_t)blockIdx.x * kThreads + threadIdx.x; g < groups; g += stride) {
        const int64_t t = g / groups_per_row;
        const int64_t c = g - t * groups_per_row;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int k = 0; k < K; ++k) {
            const int32_t r = __ldg(row_of + t * K + k);
            if (r < 0) continue;
            const float wk = __ldg(w + t * K + k);
            const uint4 yv = __ldg(y8 + (int64_t)r * groups_per_row + c);
            const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wk, bf16_to_f32(yw[i] & 0xFFFFu)));
                acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wk, bf16_to_f32(yw[i] >> 16)));
            }
        }
        out8[g] = make_uint4(pack2(f32_to_bf16(acc[0]), f32_to_bf16(acc[1])),
                             pack2(f32_to_bf16(acc[2]), f32_to_bf16(acc[3])),
                             pack2(f32_to_bf16(acc[4]), f32_to_bf16(acc[5])),
                             pack2(f32_to_bf16(acc[6]), f32_to_bf16(acc[7])));
    }
}

// Scale tensor [rows, kb] (kb = K/32 bytes per row) -> tile layout: for row group g of 128
// rows and K-word w (4 consecutive scale bytes), 512 bytes at ((g * kw) + w) * 512 holding,
// at byte l * 16 + j * 4 + b, the scale of row g * 128 + 32 j + l and K block 4 w + b. That
// is the 32-lane x 16-byte block tcgen05.cp copies into tensor memory. One CTA converts 128
// rows x 32 K-words through shared memory; rows past the end read as 0.
constexpr int kTileThreads = 128;
__global__ void __launch_bounds__(kTileThreads) sf_tile_kernel(const uint8_t* __restrict__ sf,
                                                               uint8_t* __restrict__ out, int64_t rows,
                                                               int64_t kb) {
    __shared__ uint32_t s_rows[128][33];             // 128 rows x 32 words (+1 against conflicts)
    const int64_t g = blockIdx.x;                    // row group
    const int64_t wc = (int64_t)blockIdx.y * 32;     // first K-word of this chunk
    const int64_t kw = kb / 4;
    const int nw = (int)(kw - wc < 32 ? kw - wc : 32);
    const int t = threadIdx.x;
    const int64_t row = g * 128 + t;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(sf + row * kb) + wc;
    for (int w = 0; w < nw; ++w) s_rows[t][w] = row < rows ? __ldg(src + w) : 0u;
    __syncthreads();
    uint4* o = reinterpret_cast<uint4*>(out + ((g * kw) + wc) * 512);
    for (int u = t; u < nw * 32; u += kTileThreads) {
        const int w = u >> 5, l = u & 31;
        o[u] = make_uint4(s_rows[l][w], s_rows[l + 32][w], s_rows[l + 64][w], s_rows[l + 96][w]);
    }
}

}  // namespace

cudaError_t launch_sf_tile(const uint8_t* sf, uint8_t* out, int64_t rows, int64_t kb, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const dim3 grid((unsigned)((rows + 127) / 128), (unsigned)((kb / 4 + 31) / 32));
    sf_tile_kernel<<<grid, kTileThreads, 0, s>>>(sf, out, rows, kb);
    return cudaGetLastError();
}

cudaError_t launch_mxfp4_dequant(const uint8_t* codes, const uint8_t* sf, uint16_t* out, int64_t rows,
                                 int64_t cols, int num_sms, cudaStream_t s) {
    const int64_t groups = rows * (cols / 8);
    if (groups == 0) return cudaSuccess;
    mxfp4_dequant_kernel<<<grid_for(groups, num_sms), kThreads, 0, s>>>(
        reinterpret_cast<const uint32_t*>(codes), sf, reinterpret_cast<uint4*>(out), groups);
    return cudaGetLastError();
}

cudaError_t launch_fp8_dequant(const uint8_t* q, const uint8_t* sf, uint16_t* out, int64_t rows,
                               int64_t cols, int num_sms, cudaStream_t s) {
    const int64_t gpr = cols / 16;
    const int64_t groups = rows * gpr;
    if (groups == 0) return cudaSuccess;
    fp8_dequant_kernel<<<grid_for(groups, num_sms), kThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(q), sf, reinterpret_cast<uint4*>(out), groups, gpr, (cols + 127) / 128);
    return cudaGetLastError();
}

cudaError_t launch_act_quant(const uint16_t* x, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K,
                             int num_sms, cudaStream_t s) {
    const int64_t groups = M * (K / 8);
    if (groups == 0) return cudaSuccess;
    act_quant_kernel<<<grid_for(groups, num_sms), kThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(x), reinterpret_cast<uint32_t*>(codes), sf, groups);
    return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* y, const int32_t* row_of, const float* w, uint16_t* out,
                           int64_t T, int64_t K, int64_t H, int num_sms, cudaStream_t s) {
    const int64_t gpr = H / 8;
    const int64_t groups = T * gpr;
    if (groups == 0) return cudaSuccess;
    combine_kernel<<<grid_for(groups, num_sms), kThreads, 0, s>>>(reinterpret_cast<const uint4*>(y), row_of,
                                                                  w, reinterpret_cast<uint4*>(out), groups,
                                                                  gpr, (int)K);
    return cudaGetLastError();
}

}  // namespace mx
