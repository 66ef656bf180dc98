// mx_device.cuh -- device-side building blocks for the sm_103a kernels: BF16 and MXFP4
// element helpers, the MX quantiser, mbarrier / TMA / cp.async / tcgen05 wrappers written
// as inline PTX, and bounded waits that report through a device status word.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mx_internal.h"

namespace mx {

// ------------------------------------------------------------------------------------
// Status words. A bounded wait that runs out ORs a code into the caller's workspace word
// (the forward's own, which its first kernel clears and mx_check_workspace reads) and into
// the device-wide word (read by mx_device_status), then gives up.
// ------------------------------------------------------------------------------------
enum : uint32_t {
    kErrWaitFull = 1u << 0,
    kErrWaitEmpty = 1u << 1,
    kErrWaitTmemFull = 1u << 2,
    kErrWaitTmemEmpty = 1u << 3,
    kErrWaitDrain = 1u << 4,
    kErrWaitGrid = 1u << 5,
};

// Upper bound on one wait, in globaltimer nanoseconds. Every legitimate wait in these
// kernels resolves in microseconds; two seconds only fires when a pipeline is broken.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(const StatusWords& st, uint32_t code) {
    if (st.ws != nullptr) atomicOr(st.ws, code);
    if (st.dev != nullptr) atomicOr(st.dev, code);
}

// ------------------------------------------------------------------------------------
// BF16 helpers (bit patterns as uint16)
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Round to BF16, nearest-even; NaN -> 0x7FC0 with its sign.
__device__ __forceinline__ uint32_t f32_to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return ((u >> 16) & 0x8000u) | 0x7FC0u;
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two values to packed BF16 (lo in the low half), round to nearest even by the hardware
// conversion; a NaN becomes the positive 0x7FFF.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two values to packed BF16 (a in the low half), round to nearest even; the hardware
// conversion, with NaN written as sign | 0x7FC0 like f32_to_bf16.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    if (__builtin_expect(a != a || b != b, 0)) r = f32_to_bf16(a) | (f32_to_bf16(b) << 16);
    return r;
}

// ------------------------------------------------------------------------------------
// MX quantiser: shared exponent and E2M1 code (round to nearest even, saturating at 6)
// ------------------------------------------------------------------------------------
// Scale byte for a finite amax >= 0: floor(log2 amax) - 2 + 127, clamped at 0. For a normal
// float amax this is its biased exponent minus 2; zero and subnormals give 0.
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
    int be = (int)(__float_as_uint(amax) >> 23);
    return (uint32_t)max(be - 2, 0);
}

// 2^(127 - E) as a float for E in [0, 252] (always a normal float).
__device__ __forceinline__ float mx_inv_scale(uint32_t E) { return __uint_as_float((254u - E) << 23); }

// E2M1 codes of eight scaled values, element 0 in the lowest nibble: the hardware
// conversion rounds to the nearest point of the grid {0, .5, 1, 1.5, 2, 3, 4, 6} (even code
// at a midpoint), saturates at +-6 and keeps the sign of a value that rounds to zero.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Quantise one 32-element block held entirely by this thread (float values that are
// already BF16 numbers). Writes 16 bytes of codes and returns the scale byte.
__device__ __forceinline__ uint32_t mx_quant32(const float (&f)[32], uint4& codes) {
    float amax = 0.0f;
    uint32_t bad = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        bad |= (uint32_t)((__float_as_uint(f[i]) & 0x7F800000u) == 0x7F800000u);
        amax = fmaxf(amax, fabsf(f[i]));
    }
    uint32_t w[4] = {0, 0, 0, 0};
    uint32_t E;
    if (bad) {
        E = 255u;
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i >> 3] |= (((__float_as_uint(f[i]) >> 28) & 8u) | 7u) << (4 * (i & 7));
    } else {
        E = mx_scale_byte(amax);
        const float inv = mx_inv_scale(E);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float sv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) sv[i] = f[8 * k + i] * inv;   // exact: inv is a power of two
            w[k] = e2m1x8(sv);
        }
    }
    codes = make_uint4(w[0], w[1], w[2], w[3]);
    return E;
}

// MXFP8 quantiser (E4M3 elements, one E8M0 scale per 32): the OCP MX rule with E4M3's
// largest exponent 8. Scale byte floor(log2 amax) - 8 + 127, clamped at 0 (the biased
// exponent of a normal float amax, minus 8); elements E4M3 nearest-even of x * 2^(127 - E)
// (exact: a power-of-two scaling), saturating at +-448, sign kept (-0 -> 0x80); a block
// holding a NaN or an infinity gets scale 255 and elements sign|0x7F. Quantises one block
// held by this thread (floats that are BF16 numbers) into 32 code bytes (element 0 in the
// lowest byte of codes[0].x); returns the scale byte.
__device__ __forceinline__ uint32_t mx8_quant32(const float (&f)[32], uint4 (&codes)[2]) {
    float amax = 0.0f;
    uint32_t bad = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        bad |= (uint32_t)((__float_as_uint(f[i]) & 0x7F800000u) == 0x7F800000u);
        amax = fmaxf(amax, fabsf(f[i]));
    }
    uint32_t w[8];
    uint32_t E;
    if (bad) {
        E = 255u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            w[k] = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) w[k] |= (((__float_as_uint(f[4 * k + i]) >> 24) & 0x80u) | 0x7Fu) << (8 * i);
        }
    } else {
        E = (uint32_t)max((int)(__float_as_uint(amax) >> 23) - 8, 0);
        const float inv = mx_inv_scale(E);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            uint32_t lo, hi;   // the second source of each conversion lands in the low byte
            asm("{\n\t.reg .b16 a, b;\n\t"
                "cvt.rn.satfinite.e4m3x2.f32 a, %3, %2;\n\t"
                "cvt.rn.satfinite.e4m3x2.f32 b, %5, %4;\n\t"
                "cvt.u32.u16 %0, a;\n\t"
                "cvt.u32.u16 %1, b;\n\t}"
                : "=r"(lo), "=r"(hi)
                : "f"(f[4 * k] * inv), "f"(f[4 * k + 1] * inv), "f"(f[4 * k + 2] * inv), "f"(f[4 * k + 3] * inv));
            w[k] = lo | (hi << 16);
        }
    }
    codes[0] = make_uint4(w[0], w[1], w[2], w[3]);
    codes[1] = make_uint4(w[4], w[5], w[6], w[7]);
    return E;
}

// E4M3 byte of a float 0 <= t <= 448: round to nearest, ties to even (the second source
// of the x2 conversion lands in the low byte).
__device__ __forceinline__ uint32_t e4m3_rn(float t) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
    return (uint32_t)r & 0xFFu;
}

// Value of a non-negative finite E4M3 byte (0x00..0x7E), exact in float32.
__device__ __forceinline__ float e4m3_pos_value(uint32_t s) {
    const uint32_t e = s >> 3, m = s & 7u;
    return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// NVFP4 quantisation of one 16-element block held by this thread (float values that are
// BF16 numbers) against the float32 global g, with r = 1 / (6 g): the scale byte is the
// E4M3 value nearest min(amax * r, 448), and each element's code the E2M1 value nearest
// x * (1 / (e4m3(scale) * g)), saturating at 6 and keeping the sign; every step one float32
// operation rounded to nearest even. A zero scale gives the codes +-0; a block holding a NaN
// or an infinity gets the NaN scale 0x7F and codes sign|7. Writes 8 bytes of codes and
// returns the scale byte.
__device__ __forceinline__ uint32_t nv_quant16(const float* f, float g, float r, uint2& codes) {
    float amax = 0.0f;
    uint32_t bad = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        bad |= (uint32_t)((__float_as_uint(f[i]) & 0x7F800000u) == 0x7F800000u);
        amax = fmaxf(amax, fabsf(f[i]));
    }
    uint32_t w[2] = {0, 0};
    uint32_t S;
    if (bad) {
        S = 0x7Fu;
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i >> 3] |= (((__float_as_uint(f[i]) >> 28) & 8u) | 7u) << (4 * (i & 7));
    } else {
        S = e4m3_rn(fminf(__fmul_rn(amax, r), 448.0f));
        if (S == 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i >> 3] |= ((__float_as_uint(f[i]) >> 28) & 8u) << (4 * (i & 7));
        } else {
            const float rd = __frcp_rn(__fmul_rn(e4m3_pos_value(S), g));
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float sv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) sv[i] = fminf(fmaxf(__fmul_rn(f[8 * k + i], rd), -6.0f), 6.0f);
                w[k] = e2m1x8(sv);
            }
        }
    }
    codes = make_uint2(w[0], w[1]);
    return S;
}

// E2M1 magnitude values by code (device constant table used by the dequant kernels).
__device__ __forceinline__ float e2m1_value(uint32_t code) {
    // magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 built from the bit fields
    uint32_t e = (code >> 1) & 3u, m = code & 1u;
    float mag = (e == 0) ? 0.5f * (float)m : __uint_as_float(((126u + e) << 23) | (m << 22));
    return (code & 8u) ? -mag : mag;
}

// 2^(b - 127) for an E8M0 byte b < 255 (b = 0 gives the float32 subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t b) {
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// ------------------------------------------------------------------------------------
// Shared-memory addresses and mbarriers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false when the CTA-wide abort
// flag is raised or the time limit passes (then it raises the flag and sets `code`).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const StatusWords& status, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = 0;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            uint64_t t = globaltimer();
            if (t0 == 0) {
                t0 = t;
            } else if (t - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                set_status(status, code);
                return false;
            }
        }
    }
}

// Grid-wide barrier of a cooperative launch (every CTA resident at once). Each CTA makes its
// earlier global writes visible to the other CTAs, including to their TMA (async-proxy)
// reads; thread 0 adds the CTA's arrival to `counter` and waits until it reaches `target`
// (the barrier's cumulative arrival count: gridDim.x per barrier passed). The wait is
// bounded like an mbarrier wait: past the limit it raises the CTA's abort flag, records
// kErrWaitGrid and lets the CTA go on. Every thread of the CTA calls it.
__device__ __forceinline__ void grid_sync(uint32_t* counter, uint32_t target, volatile int* abort_flag,
                                          const StatusWords& status) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        uint64_t t0 = 0;
        for (uint32_t i = 0;; ++i) {
            uint32_t v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            if (v >= target) break;
            if ((i & 63u) == 63u) {
                const uint64_t t = globaltimer();
                if (t0 == 0) {
                    t0 = t;
                } else if (t - t0 > kWaitLimitNs) {
                    *abort_flag = 1;
                    set_status(status, kErrWaitGrid);
                    break;
                }
            }
            __nanosleep(32);
        }
        __threadfence();
    }
    __syncthreads();
}

// ------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) and cp.async
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 4-D TMA load (coordinates innermost first) completing on the mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            int32_t w, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// 2-D TMA store shared -> global of one box; the shared source is read asynchronously
// (bulk_wait_read before it is overwritten). Coordinates: x innermost, in elements.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap), "r"(x),
                 "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// This thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bulk copy global -> shared (async proxy) completing `bytes` on the mbarrier; both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Programmatic dependent launch. A kernel of the forward launched with programmatic stream
// serialisation may start while the kernel before it in the stream is still finishing: it
// does its setup, then pdl_wait() until that kernel (and, transitively, every earlier one)
// has completed and its memory is visible, before touching global memory. Each kernel
// calls pdl_launch_dependents() once the next kernel may be scheduled. Without the launch
// attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 4-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
// 8 bytes (both addresses 8-byte aligned); bytes past src_bytes (0, 4 or 8) are zero-filled.
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
// Arrive on `bar` once every cp.async this thread issued before has completed; the
// arrival counts toward the barrier's expected count (which must include it).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// tcgen05: tensor memory, block-scaled MMA, copies and loads
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand tile written by TMA with 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024u >> 4) << 32;      // stride byte offset: one 8 x 128 B swizzle atom
    d |= (uint64_t)1 << 46;                 // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                 // 128-byte swizzle
    return d;
}

// Descriptor of a 32-row x 16-byte scale-factor block (no swizzle, rows 16 bytes apart,
// 8-row groups 128 bytes apart), the source of a 32x128b tcgen05.cp.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor of kind::mxf4 block-scaled MMA: E2M1 A and B (K-major), E8M0
// scales, FP32 accumulation implied by the kind, M x N tile.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor of kind::mxf8f6f4 block-scaled MMA with E4M3 A (type 0) and E2M1 B
// (type 5), both K-major, E8M0 scales, FP32 accumulation implied by the kind, M x N tile.
__host__ __device__ constexpr uint32_t idesc_mxf8_e2m1(int M, int N) {
    return (0u << 7) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_with_sf_ids(uint32_t idesc, uint32_t a_id, uint32_t b_id) {
    return idesc | (b_id << 4) | (a_id << 29);
}

__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// MXFP8 x MXFP4 block-scaled MMA (K = 32): E4M3 A, E2M1 B (held in shared memory as 16
// values per 16 bytes, the second 8 bytes of each 16 unused), one E8M0 scale per 32 elements
// of K: each MMA reads one byte of the rows' scale words, chosen by the idesc scale ids.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// NVFP4 block-scaled MMA: E2M1 A and B with one E4M3 scale per 16 elements of K; the
// instruction descriptor's scale-format bit (23) must be clear (E4M3). Each MMA (K = 64)
// reads one 32-bit scale word per row (four scales).
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Copy a 32-row x 128-bit block from shared memory into tensor memory, replicated into
// all four 32-lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Copy 128 rows x 256 bits from shared memory into 128 lanes x 8 columns of tensor memory
// (row r -> lane r, its eight 32-bit words -> eight columns); no replication.
__device__ __forceinline__ void tc_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive 32-bit columns of this warp's 32 lanes.
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace mx
