// mx_elementwise.cu -- HBM-bound kernels: MXFP4 -> BF16 and FP8 E4M3 x E8M0 128x128 -> BF16
// dequantisation, the standalone MX activation quantiser, and the top-k weighted combine.
//
// Weight format per "2026-05-08 DeepSeek V4 Pro NVFP4 Quantization", "Script update:
// dequant_fp8_to_bf16.py now handles ALL compressed types" (item 2: two E2M1 values per
// byte, lower nibble first, LUT x E8M0 per row per 32 columns; item 1: FP8 x E8M0 per
// 128x128 block). Combine per "Current Bug: vLLM produces empty/garbage output", "Phase 1"
// (routing, top-k, scatter) and "Phase 3: Clean up" (the final scatter is BF16).
#include "mx_phases.cuh"

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

// Four E2M1 codes (16 bits, element 0 lowest) -> four BF16 values (two words, element 0
// in the low half) times 2^(E-127), for a scale byte E in [2, 252]: every nonzero product is
// then a normal BF16 whose bits are the code's BF16 bits at scale 1 (a byte table looked up
// with prmt) with E - 127 added to the exponent field. Exact, like the arithmetic path.
__device__ __forceinline__ void e2m1x4_to_bf16(uint32_t c16, uint32_t off2, uint32_t& o0, uint32_t& o1) {
    const uint32_t sel = c16 & 0x7777u;                          // magnitudes 0..7 select table bytes
    const uint32_t hi = __byte_perm(0x3F3F3F00u, 0x40404040u, sel);   // high bytes of 0, .5, 1, .. 6
    const uint32_t lo = __byte_perm(0xC0800000u, 0xC0804000u, sel);   // low bytes
    uint32_t a = __byte_perm(lo, hi, 0x5140u);                   // elements 0, 1
    uint32_t b = __byte_perm(lo, hi, 0x7362u);                   // elements 2, 3
    a = __vadd2(a, off2 & __vcmpne2(a, 0u));                     // scale the nonzero halves
    b = __vadd2(b, off2 & __vcmpne2(b, 0u));
    o0 = a | ((c16 & 0x8u) << 12) | ((c16 & 0x80u) << 24);       // signs (bit 3 of each code)
    o1 = b | ((c16 & 0x800u) << 4) | ((c16 & 0x8000u) << 16);
}

// Eight codes of one word with scale byte s, any s (255: NaN with the code's sign).
__device__ __forceinline__ void e2m1x8_to_bf16_any(uint32_t c, uint32_t s, uint32_t (&o)[4]) {
    if (s >= 2u && s <= 252u) {
        const uint32_t off2 = (((s - 127u) << 7) & 0xFFFFu) * 0x10001u;
        e2m1x4_to_bf16(c & 0xFFFFu, off2, o[0], o[1]);
        e2m1x4_to_bf16(c >> 16, off2, o[2], o[3]);
    } else if (s == 255u) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack2((((c >> (8 * i)) & 8u) << 12) | 0x7FC0u, (((c >> (8 * i + 4)) & 8u) << 12) | 0x7FC0u);
    } else {
        const float scale = e8m0_value(s);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack2(f32_to_bf16(e2m1_value((c >> (8 * i)) & 15u) * scale),
                         f32_to_bf16(e2m1_value((c >> (8 * i + 4)) & 15u) * scale));
    }
}

// One unit = one 32-element scale block = 16 code bytes (four words) -> 64 output bytes;
// units are contiguous over the whole tensor because cols % 32 == 0, so unit u reads code
// words 4u..4u+3 and scale sf[u] and writes output vectors 4u..4u+3. A warp takes 64 units
// per pass, lane l handling word l % 4 of units 8i + l / 4 (i = 0..7): each load
// instruction reads 128 contiguous bytes and each store writes 512 contiguous bytes, with
// eight loads in flight per lane.
constexpr int kDeqUnitsPerWarp = 64;
__global__ void __launch_bounds__(kThreads) mxfp4_dequant_kernel(const uint32_t* __restrict__ codes32,
                                                                 const uint8_t* __restrict__ sf,
                                                                 uint4* __restrict__ out, int64_t units) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t base = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * kDeqUnitsPerWarp;
         base < units; base += nwarps * kDeqUnitsPerWarp) {
        uint32_t c[8], sc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t u = base + 8 * i + (lane >> 2);
            const bool ok = u < units;
            c[i] = ok ? __ldg(codes32 + 4 * u + (lane & 3)) : 0u;
            sc[i] = ok ? __ldg(sf + u) : 127u;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t u = base + 8 * i + (lane >> 2);
            if (u < units) {
                uint32_t o[4];
                e2m1x8_to_bf16_any(c[i], sc[i], o);
                out[4 * u + (lane & 3)] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// E4M3 ("fn") byte -> float32, exact, for every byte but the NaN ones (S.1111.111), which
// the callers handle first.
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

// NVFP4 -> BF16 ("Current Bug: vLLM produces empty/garbage output", "What we know":
// NVFP4 weights dequantised to BF16; the per-tensor global scale of "Phase 2: CuTeDSL
// Attention Kernel"): out = bf16(float32(LUT[code] * e4m3(scale) * global)). LUT[code] *
// e4m3(scale) is exact in float32, so the multiply by the global scale is the one float32
// rounding, then one BF16 rounding (both to nearest even). A NaN result is 0x7FC0 with the
// XOR of the code's, the scale's and the global's sign bits.
//
// Both roundings are symmetric, so a value is its magnitude's BF16 with the XOR of the
// three sign bits. A 16-element block has one scale, hence eight possible magnitudes,
// rounded once per block with the same float32 operations in the same order. Each thread
// takes one block (8 code bytes in, 32 bytes out): it splits the eight BF16 magnitudes
// into a high-byte and a low-byte table (two registers each), selects four elements' bytes
// at once by byte-permute on their 3-bit magnitude codes, puts each element's sign into its
// high byte and interleaves the bytes into BF16.
__device__ __forceinline__ uint32_t nv_sel(uint32_t x) {   // bytes' low 3 bits -> 4 selector nibbles
    x &= 0x07070707u;
    x = (x | (x >> 4)) & 0x00770077u;
    return (x | (x >> 8)) & 0x00007777u;
}

// Eight elements (one code word, lower nibble first) from the block's byte tables.
__device__ __forceinline__ uint4 nv_lookup8(uint32_t c, uint32_t hi0, uint32_t hi1, uint32_t lo0, uint32_t lo1,
                                            uint32_t sneg) {
    // even elements: low nibble of each code byte; odd: high nibble
    const uint32_t se = nv_sel(c), so = nv_sel(c >> 4);
    const uint32_t he = __byte_perm(hi0, hi1, se) ^ ((c << 4) & 0x80808080u) ^ sneg;
    const uint32_t le = __byte_perm(lo0, lo1, se);
    const uint32_t ho = __byte_perm(hi0, hi1, so) ^ (c & 0x80808080u) ^ sneg;
    const uint32_t lo = __byte_perm(lo0, lo1, so);
    // BF16 of elements 0, 2 (ea) / 4, 6 (eb) and 1, 3 (oa) / 5, 7 (ob)
    const uint32_t ea = __byte_perm(le, he, 0x5140u), eb = __byte_perm(le, he, 0x7362u);
    const uint32_t oa = __byte_perm(lo, ho, 0x5140u), ob = __byte_perm(lo, ho, 0x7362u);
    return make_uint4(__byte_perm(ea, oa, 0x5410u), __byte_perm(ea, oa, 0x7632u), __byte_perm(eb, ob, 0x5410u),
                      __byte_perm(eb, ob, 0x7632u));
}

// One 16-element block: 8 code bytes and its scale byte -> 32 bytes of BF16 at out[2b], out[2b + 1].
__device__ __forceinline__ void nvfp4_block_to_bf16(uint2 c, uint32_t sbyte, float ga, uint32_t gneg, uint4* out) {
    const float sa = (sbyte & 0x7Fu) == 0x7Fu ? __uint_as_float(0x7FC00000u) : fabsf(e4m3_value(sbyte));
    // t[k]: BF16 magnitudes of codes 2k (low half) and 2k + 1 (high half)
    uint32_t t[4];
    const float m[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    if (isfinite(sa) && isfinite(ga)) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            t[k] = pack_bf16x2(__fmul_rn(__fmul_rn(m[2 * k], sa), ga), __fmul_rn(__fmul_rn(m[2 * k + 1], sa), ga));
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t hh[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float v = __fmul_rn(__fmul_rn(m[2 * k + j], sa), ga);
                hh[j] = v != v ? 0x7FC0u : f32_to_bf16(v);
            }
            t[k] = hh[0] | (hh[1] << 16);
        }
    }
    const uint32_t hi0 = __byte_perm(t[0], t[1], 0x7531u), hi1 = __byte_perm(t[2], t[3], 0x7531u);
    const uint32_t lo0 = __byte_perm(t[0], t[1], 0x6420u), lo1 = __byte_perm(t[2], t[3], 0x6420u);
    const uint32_t sneg = (((sbyte >> 7) ^ gneg) & 1u) ? 0x80808080u : 0u;
    out[0] = nv_lookup8(c.x, hi0, hi1, lo0, lo1, sneg);
    out[1] = nv_lookup8(c.y, hi0, hi1, lo0, lo1, sneg);
}

// Each thread takes kNvBlocksPerThread blocks a whole grid apart per pass, loading all of
// them before converting any, so that many loads are in flight per thread: one 8-byte load
// each left the kernel latency-bound near 70 % of HBM.
constexpr int kNvBlocksPerThread = 4;
__global__ void __launch_bounds__(kThreads) nvfp4_dequant_kernel(const uint2* __restrict__ codes8,
                                                                 const uint8_t* __restrict__ sf, float g,
                                                                 uint4* __restrict__ out, int64_t blocks) {
    const uint32_t gneg = __float_as_uint(g) >> 31;
    const float ga = fabsf(g);
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    for (int64_t b0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; b0 < blocks;
         b0 += kNvBlocksPerThread * nthreads) {
        uint2 c[kNvBlocksPerThread];
        uint32_t sb[kNvBlocksPerThread];
#pragma unroll
        for (int i = 0; i < kNvBlocksPerThread; ++i) {
            const int64_t b = b0 + i * nthreads;
            const bool ok = b < blocks;
            c[i] = ok ? __ldg(codes8 + b) : make_uint2(0u, 0u);
            sb[i] = ok ? (uint32_t)__ldg(sf + b) : 0u;
        }
#pragma unroll
        for (int i = 0; i < kNvBlocksPerThread; ++i) {
            const int64_t b = b0 + i * nthreads;
            if (b < blocks) nvfp4_block_to_bf16(c[i], sb[i], ga, gneg, out + 2 * b);
        }
    }
}

// Two E4M3 bytes (first in the low half) -> two BF16 values times 2^(s-127), for s in
// [10, 246] and no NaN byte: the hardware conversion to FP16 is exact, every value is then
// a normal FP16 of exponent 6..23, and with the scale a normal BF16 whose exponent is the
// FP16 exponent + s - 15 and whose mantissa is the FP16's top 7 bits (E4M3 has 3).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16(uint32_t b16, uint32_t off2) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)b16));
    const uint32_t mag = ((h & 0x7FFF7FFFu) >> 3) & 0x0FFF0FFFu;   // FP16 exponent+mantissa at BF16 places
    return __vadd2(mag, off2 & __vcmpne2(mag, 0u)) | (h & 0x80008000u);
}

__device__ __forceinline__ uint32_t e4m3_to_bf16_slow(uint32_t b, uint32_t s) {
    if ((b & 0x7Fu) == 0x7Fu || s == 255u) return ((b & 0x80u) << 8) | 0x7FC0u;
    return f32_to_bf16(e4m3_value(b) * e8m0_value(s));
}

// 8 E4M3 bytes of one row (one 128-column scale block) -> 16 bytes of BF16.
__device__ __forceinline__ uint4 fp8x8_to_bf16(const uint2 qv, uint32_t s) {
    const uint32_t w[2] = {qv.x, qv.y};
    uint32_t o[4];
    const uint32_t nan_bytes = __vcmpeq4(w[0] & 0x7F7F7F7Fu, 0x7F7F7F7Fu) | __vcmpeq4(w[1] & 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    if (s >= 10u && s <= 246u && nan_bytes == 0u) {
        const uint32_t off2 = (((s - 15u) << 7) & 0xFFFFu) * 0x10001u;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            o[2 * i] = e4m3x2_to_bf16(w[i] & 0xFFFFu, off2);
            o[2 * i + 1] = e4m3x2_to_bf16(w[i] >> 16, off2);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t ww = w[i >> 1] >> (16 * (i & 1));
            o[i] = pack2(e4m3_to_bf16_slow(ww & 0xFFu, s), e4m3_to_bf16_slow((ww >> 8) & 0xFFu, s));
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// One CTA per row (grid-stride over rows); lane l of a warp takes the row's 8-column chunks
// l, l + 32, ...: each load instruction reads 256 contiguous bytes and each store writes 512.
// Four chunks per thread per pass keep four loads in flight; the 128x128 block scale comes
// from the row's block row and the chunk's block column.
constexpr int kFp8ChunksPerPass = 4;
__global__ void __launch_bounds__(kThreads) fp8_dequant_kernel(const uint8_t* __restrict__ q,
                                                               const uint8_t* __restrict__ sf,
                                                               uint16_t* __restrict__ out, int64_t rows,
                                                               int64_t cols, int64_t sf_cols) {
    const int chunks = (int)(cols / 8);
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint2* qr = reinterpret_cast<const uint2*>(q + row * cols);
        uint4* orow = reinterpret_cast<uint4*>(out + row * cols);
        const uint8_t* srow = sf + (row >> 7) * sf_cols;
        for (int c0 = threadIdx.x; c0 < chunks; c0 += kFp8ChunksPerPass * kThreads) {
            uint2 qv[kFp8ChunksPerPass];
            uint32_t sv[kFp8ChunksPerPass];
#pragma unroll
            for (int i = 0; i < kFp8ChunksPerPass; ++i) {
                const int c = c0 + i * kThreads;
                qv[i] = c < chunks ? __ldg(qr + c) : make_uint2(0, 0);
                sv[i] = c < chunks ? __ldg(srow + (c >> 4)) : 127u;
            }
#pragma unroll
            for (int i = 0; i < kFp8ChunksPerPass; ++i) {
                const int c = c0 + i * kThreads;
                if (c < chunks) orow[c] = fp8x8_to_bf16(qv[i], sv[i]);
            }
        }
    }
}

// One thread per 32-element block (act_quant_blocks).
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint4* __restrict__ x8,
                                                             uint4* __restrict__ codes16,
                                                             uint8_t* __restrict__ sf, int64_t blocks,
                                                             uint32_t* clear_word, int64_t blocks_per_row,
                                                             int64_t sm_k_tiles) {
    pdl_wait();
    if (clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *clear_word = 0u;
    act_quant_blocks(x8, codes16, sf, blocks, (int64_t)blockIdx.x * kThreads + threadIdx.x,
                     (int64_t)gridDim.x * kThreads, blocks_per_row, sm_k_tiles);
    pdl_launch_dependents();
}

// One thread per 32-element block, MXFP8 (act_quant8_blocks).
__global__ void __launch_bounds__(kThreads) act_quant8_kernel(const uint4* __restrict__ x8,
                                                              uint4* __restrict__ codes16,
                                                              uint8_t* __restrict__ sf, int64_t blocks,
                                                              uint32_t* clear_word) {
    pdl_wait();
    if (clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *clear_word = 0u;
    act_quant8_blocks(x8, codes16, sf, blocks, (int64_t)blockIdx.x * kThreads + threadIdx.x,
                      (int64_t)gridDim.x * kThreads);
    pdl_launch_dependents();
}

// Self-test of the failure path: one thread waits, with the bounded wait every pipeline of
// the GEMMs uses, on a freshly initialised mbarrier that nothing arrives at. The wait runs
// out after its limit, records kErrWaitFull in the status word and the kernel returns, so
// the context stays usable. No asynchronous copy or MMA references the barrier.
__global__ void __launch_bounds__(32) wait_probe_kernel(StatusWords status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    mbar_wait(smem_u32(&bar), 0, &abort_flag, status, kErrWaitFull);
}

// NVFP4 activation quantisation (nv_quant16): one thread per 16-element block, two 16-byte
// loads, 8 bytes of codes and one E4M3 scale byte out.
__global__ void __launch_bounds__(kThreads) act_quant_nv_kernel(const uint4* __restrict__ x8,
                                                                uint2* __restrict__ codes8,
                                                                uint8_t* __restrict__ sf, int64_t blocks,
                                                                float g, uint32_t* clear_word) {
    pdl_wait();
    if (clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *clear_word = 0u;
    const float r = __frcp_rn(__fmul_rn(6.0f, g));
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x; b < blocks; b += stride) {
        float f[16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint4 v = __ldg(x8 + 2 * b + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[8 * i + 2 * j] = bf16_to_f32(w[j] & 0xFFFFu);
                f[8 * i + 2 * j + 1] = bf16_to_f32(w[j] >> 16);
            }
        }
        uint2 codes;
        sf[b] = (uint8_t)nv_quant16(f, g, r, codes);
        codes8[b] = codes;
    }
    pdl_launch_dependents();
}

// NVFP4 activation-global calibration ("Current Bug: vLLM produces empty/garbage output",
// "Phase 1: CuTeDSL Shared Expert Kernel": a warm-up-based gs). amax_kernel folds the
// largest finite |x| of a BF16 tensor into a running maximum kept as float32 bits (a
// non-negative float orders like its bit pattern, so atomicMax on the bits is the float
// maximum); NaN and infinities are skipped. Each thread reduces its 16-byte vectors (plus
// the scalar tail), then the warp and the CTA, and one atomic per CTA updates the maximum.
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint4* __restrict__ x8, int64_t n8,
                                                        const uint16_t* __restrict__ tail, int ntail,
                                                        uint32_t* __restrict__ amax_bits) {
    __shared__ uint32_t s_max[kThreads / 32];
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n8; i += stride) {
        const uint4 v = __ldg(x8 + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = w[j] & 0x7FFFu, hi = (w[j] >> 16) & 0x7FFFu;
            if (lo < 0x7F80u) m = max(m, lo);
            if (hi < 0x7F80u) m = max(m, hi);
        }
    }
    if (blockIdx.x == 0 && (int)threadIdx.x < ntail) {
        const uint32_t b = tail[threadIdx.x] & 0x7FFFu;
        if (b < 0x7F80u) m = max(m, b);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int i = 1; i < kThreads / 32; ++i) m = max(m, s_max[i]);
        atomicMax(amax_bits, m << 16);          // BF16 bits -> float32 bits
    }
}

// global = amax / (6 * 448), one float32 division rounded to nearest even, clamped into the
// range the NVFP4 quantiser accepts ([2^-117, 2^100]).
__global__ void nv_global_kernel(const uint32_t* __restrict__ amax_bits, float* __restrict__ global_scale) {
    const float g = __fdiv_rn(__uint_as_float(*amax_bits), 2688.0f);
    *global_scale = fminf(fmaxf(g, 0x1p-117f), 0x1p100f);
}

// The top-k weighted combine (combine_groups).
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint4* __restrict__ y8,
                                                           const int32_t* __restrict__ row_of,
                                                           const float* __restrict__ w,
                                                           uint4* __restrict__ out8, int64_t groups,
                                                           int64_t groups_per_row, int K) {
    pdl_wait();
    combine_groups<false>(y8, row_of, w, out8, groups, groups_per_row, K,
                          (int64_t)blockIdx.x * kThreads + threadIdx.x, (int64_t)gridDim.x * kThreads);
    pdl_launch_dependents();
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
    const int64_t units = rows * (cols / 32);
    if (units == 0) return cudaSuccess;
    const int64_t warps = (units + kDeqUnitsPerWarp - 1) / kDeqUnitsPerWarp;
    mxfp4_dequant_kernel<<<grid_for(warps * 32, num_sms), kThreads, 0, s>>>(
        reinterpret_cast<const uint32_t*>(codes), sf, reinterpret_cast<uint4*>(out), units);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* sf, float global_scale, uint16_t* out,
                                 int64_t rows, int64_t cols, int num_sms, cudaStream_t s) {
    const int64_t blocks = rows * (cols / 16);
    if (blocks == 0) return cudaSuccess;
    nvfp4_dequant_kernel<<<grid_for(blocks, num_sms), kThreads, 0, s>>>(
        reinterpret_cast<const uint2*>(codes), sf, global_scale, reinterpret_cast<uint4*>(out), blocks);
    return cudaGetLastError();
}

cudaError_t launch_fp8_dequant(const uint8_t* q, const uint8_t* sf, uint16_t* out, int64_t rows,
                               int64_t cols, int num_sms, cudaStream_t s) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int64_t grid = rows < (int64_t)num_sms * 8 ? rows : (int64_t)num_sms * 8;
    fp8_dequant_kernel<<<(unsigned)grid, kThreads, 0, s>>>(q, sf, out, rows, cols, (cols + 127) / 128);
    return cudaGetLastError();
}

cudaError_t launch_act_quant(const uint16_t* x, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K,
                             int num_sms, cudaStream_t s, uint32_t* clear_word, int64_t sm_k_tiles) {
    const int64_t blocks = M * (K / 32);
    if (blocks == 0) return cudaSuccess;
    return launch_pdl(act_quant_kernel, dim3(grid_for(blocks, num_sms)), dim3(kThreads), 0, s,
                      reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(codes), sf, blocks, clear_word,
                      K / 32, sm_k_tiles);
}

cudaError_t launch_act_quant_mxfp8(const uint16_t* x, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K,
                                   int num_sms, cudaStream_t s, uint32_t* clear_word) {
    const int64_t blocks = M * (K / 32);
    if (blocks == 0) return cudaSuccess;
    return launch_pdl(act_quant8_kernel, dim3(grid_for(blocks, num_sms)), dim3(kThreads), 0, s,
                      reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(codes), sf, blocks, clear_word);
}

cudaError_t launch_wait_probe(StatusWords status, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_act_quant_nvfp4(const uint16_t* x, float global_scale, uint8_t* codes, uint8_t* sf, int64_t M,
                                   int64_t K, int num_sms, cudaStream_t s, uint32_t* clear_word) {
    const int64_t blocks = M * (K / 16);
    if (blocks == 0) return cudaSuccess;
    return launch_pdl(act_quant_nv_kernel, dim3(grid_for(blocks, num_sms)), dim3(kThreads), 0, s,
                      reinterpret_cast<const uint4*>(x), reinterpret_cast<uint2*>(codes), sf, blocks, global_scale,
                      clear_word);
}

cudaError_t launch_nv_calibrate(const uint16_t* x, int64_t n, float* amax, float* global_scale, int num_sms,
                                cudaStream_t s) {
    const int64_t n8 = n / 8;
    const int ntail = (int)(n - 8 * n8);
    if (n > 0) {
        amax_kernel<<<grid_for(n8 > 0 ? n8 : 1, num_sms, 4), kThreads, 0, s>>>(
            reinterpret_cast<const uint4*>(x), n8, x + 8 * n8, ntail, reinterpret_cast<uint32_t*>(amax));
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    nv_global_kernel<<<1, 1, 0, s>>>(reinterpret_cast<const uint32_t*>(amax), global_scale);
    return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* y, const int32_t* row_of, const float* w, uint16_t* out,
                           int64_t T, int64_t K, int64_t H, int num_sms, cudaStream_t s) {
    const int64_t gpr = H / 8;
    const int64_t groups = T * gpr;
    if (groups == 0) return cudaSuccess;
    return launch_pdl(combine_kernel, dim3(grid_for(groups, num_sms)), dim3(kThreads), 0, s,
                      reinterpret_cast<const uint4*>(y), row_of, w, reinterpret_cast<uint4*>(out), groups, gpr, (int)K);
}

}  // namespace mx
