// mx_phases.cuh -- the element-wise phases of the MoE forward as device functions: the
// routing permutation ("Current Bug: vLLM produces empty/garbage output", "Phase 1: CuTeDSL
// Shared Expert Kernel": the MoE is the shared-expert pipeline plus routing, top-k and
// scatter), the MX quantisation of x (routed: gathered into the grouped rows) and the
// top-k weighted combine ("Phase 3: Clean up": the final scatter is BF16).
//
// Each function does the work of one CTA of a grid: `cta` / `ncta` place it in the grid and
// the caller's `nthreads` threads all call it (the functions synchronise the CTA). The
// standalone kernels (mx_route.cu, mx_elementwise.cu) call them with their own grids; the
// persistent forward (mx_gemm.cu) calls them between grid-wide barriers with one CTA per SM.
// Shared-memory scratch comes from the caller, so the persistent kernel can reuse the GEMM
// ring's memory for it.
#pragma once

#include <type_traits>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {

constexpr int kCountThreads = 256;                 // threads that count one chunk
constexpr int kCountWarps = kCountThreads / 32;

// Stage-major layout of an activation's block scales, the order the GEMM's scale loader reads
// them in: for M tile mt (128 rows), K stage kt (256 columns) and scale word w of the stage (4
// scale bytes), the 128 rows' words lie in row order, 512 bytes. kWords = words per stage: 2 for
// MXFP4 (blocks of 32 columns), 4 for NVFP4 (blocks of 16). Block b of tile row r is at this
// byte offset; k_tiles = ceil(K / 256). It holds as many bytes per row as the row-major
// [rows, K / block] layout, rounded up to whole tiles and stages.
template <int kWords = 2>
__host__ __device__ __forceinline__ int64_t sm_scale_off(int64_t mt, int64_t r, int64_t b, int64_t k_tiles) {
    return (((mt * k_tiles + b / (4 * kWords)) * kWords + (b >> 2) % kWords) * 128 + r) * 4 + (b & 3);
}

// Shared-memory scratch of route_count_chunk: s_run [E] and s_warp [kCountWarps][E].
__host__ __device__ constexpr size_t route_count_smem(int E) { return (size_t)(1 + kCountWarps) * E * 4; }

// 1. Per chunk of kRouteChunk pairs: per-expert counts and each pair's rank among the earlier
// pairs of its expert inside the chunk (warp match + a per-warp scan). Threads 0..255 count;
// the others only take part in the barriers.
__device__ __forceinline__ void route_count_chunk(const int32_t* __restrict__ ids, int64_t n_pairs, int E,
                                                  int64_t chunk, int32_t* __restrict__ chunk_counts,
                                                  int32_t* __restrict__ local_rank, int32_t* s_run,
                                                  int32_t* s_warp, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    const bool counter = tid < kCountThreads;
    if (counter)
        for (int e = tid; e < E; e += kCountThreads) s_run[e] = 0;
    const int64_t base = chunk * kRouteChunk;
    for (int round = 0; round < kRouteChunk / kCountThreads; ++round) {
        if (counter)
            for (int i = tid; i < kCountWarps * E; i += kCountThreads) s_warp[i] = 0;
        __syncthreads();
        int rank_in_warp = 0, e = -1;
        bool valid = false;
        int64_t p = 0;
        if (counter) {
            p = base + (int64_t)round * kCountThreads + tid;
            e = (p < n_pairs) ? __ldg(ids + p) : -1;
            valid = (e >= 0) && (e < E);
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
            rank_in_warp = __popc(peers & ((1u << lane) - 1u));
            if (valid && rank_in_warp == 0) s_warp[warp * E + e] = __popc(peers);
        }
        __syncthreads();
        if (counter)
            for (int x = tid; x < E; x += kCountThreads) {
                int32_t run = s_run[x];
#pragma unroll
                for (int w = 0; w < kCountWarps; ++w) {
                    const int32_t c = s_warp[w * E + x];
                    s_warp[w * E + x] = run;
                    run += c;
                }
                s_run[x] = run;
            }
        __syncthreads();
        if (counter && valid) local_rank[p] = s_warp[warp * E + e] + rank_in_warp;
        __syncthreads();
    }
    if (counter)
        for (int e = tid; e < E; e += kCountThreads) chunk_counts[chunk * E + e] = s_run[e];
}

// Shared-memory scratch of route_scan: s_cnt [E], s_off [E + 1], s_toff [E + 1].
__host__ __device__ constexpr size_t route_scan_smem(int E) { return (size_t)(3 * E + 2) * 4; }

// 2. One CTA: per-expert prefix over chunks, expert offsets and the list of 128-row M tiles
// (expert, first row, valid rows) that the grouped GEMMs walk.
__device__ __forceinline__ void route_scan(const int32_t* __restrict__ chunk_counts, int64_t nchunks, int E,
                                           const RouteBufs& rb, int32_t* s_cnt, int32_t* s_off, int32_t* s_toff,
                                           int tid, int nthreads) {
    for (int e = tid; e < E; e += nthreads) {
        int32_t run = 0;
        for (int64_t c = 0; c < nchunks; ++c) {
            const int32_t v = chunk_counts[c * E + e];
            rb.chunk_base[c * E + e] = run;
            run += v;
        }
        s_cnt[e] = run;
    }
    __syncthreads();
    if (tid == 0) {
        int32_t off = 0, toff = 0;
        for (int e = 0; e < E; ++e) {
            s_off[e] = off;
            s_toff[e] = toff;
            off += s_cnt[e];
            toff += (s_cnt[e] + kBM - 1) / kBM;
        }
        s_off[E] = off;
        s_toff[E] = toff;
        rb.offsets[E] = off;
        rb.tile_base[E] = toff;
        *rb.num_mtiles = toff;
    }
    __syncthreads();
    for (int e = tid; e < E; e += nthreads) {
        rb.counts[e] = s_cnt[e];
        rb.offsets[e] = s_off[e];
        rb.tile_base[e] = s_toff[e];
        const int32_t nt = (s_cnt[e] + kBM - 1) / kBM;
        for (int32_t m = 0; m < nt; ++m) {
            const int32_t idx = s_toff[e] + m;
            rb.tile_expert[idx] = e;
            rb.tile_row0[idx] = s_off[e] + m * kBM;
            rb.tile_rows[idx] = min(kBM, s_cnt[e] - m * kBM);
        }
    }
}

// One block of a BF16 row as floats: MXFP4 32 elements (four 16-byte loads), NVFP4 16 (two).
template <int kLoads>
__device__ __forceinline__ void load_bf16_block(const uint4* __restrict__ src, float (&f)[8 * kLoads]) {
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
        const uint4 v = __ldg(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[8 * i + 2 * j] = bf16_to_f32(w[j] & 0xFFFFu);
            f[8 * i + 2 * j + 1] = bf16_to_f32(w[j] >> 16);
        }
    }
}

// Activation formats of the quantisers: MXFP4 (E2M1 codes, E8M0 per 32), NVFP4 (E2M1, E4M3
// per 16 against a float32 global) and MXFP8 (E4M3 codes, E8M0 per 32).
enum QFmt : int { kQMx4 = 0, kQNv4 = 1, kQMx8 = 2 };

// 3. Token t: row_of for its K pairs and the quantisation of its row in format kFmt (NVFP4
// against the global g), written to the rows of all its routed pairs. One thread per block
// of the row (32 elements; 16 for NVFP4): its codes (16, 8 or 32 bytes) and a scale byte per
// destination row, so a warp writes contiguous codes and scales per row. s_rows: kMaxTopK
// ints of shared memory.
template <int kFmt>
__device__ __forceinline__ void quant_gather_token(const uint4* __restrict__ x8, const int32_t* __restrict__ ids,
                                                   int K, int E, int64_t blocks_per_row, const RouteBufs& rb,
                                                   uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, float g,
                                                   int64_t t, int32_t* s_rows, int tid, int nthreads,
                                                   int64_t sm_k_tiles = 0) {
    constexpr int kLoads = kFmt == kQNv4 ? 2 : 4;
    // s_rows[k]: routed row of slot k (-1: dropped); s_rows[kMaxTopK + k]: with stage-major
    // scales, that row's M tile * 128 + row in the tile
    if (tid < K) {
        const int64_t p = t * K + tid;
        const int32_t e = __ldg(ids + p);
        int32_t row = -1, tile_pos = 0;
        if (e >= 0 && e < E) {
            const int32_t local = rb.chunk_base[(p / kRouteChunk) * E + e] + rb.local_rank[p];
            row = rb.offsets[e] + local;
            tile_pos = (rb.tile_base[e] + local / kBM) * kBM + local % kBM;
        }
        s_rows[tid] = row;
        s_rows[kMaxTopK + tid] = tile_pos;
        rb.row_of[p] = row;
    }
    __syncthreads();
    if (x8 != nullptr) {
        const uint4* xrow = x8 + t * blocks_per_row * kLoads;
        const float r = kFmt == kQNv4 ? __frcp_rn(__fmul_rn(6.0f, g)) : 0.0f;
        for (int64_t b = tid; b < blocks_per_row; b += nthreads) {
            float f[8 * kLoads];
            load_bf16_block<kLoads>(xrow + kLoads * b, f);
            if constexpr (kFmt == kQNv4) {
                uint2 codes;
                const uint32_t sb = nv_quant16(f, g, r, codes);
                for (int k = 0; k < K; ++k) {
                    const int32_t row = s_rows[k];
                    if (row < 0) continue;
                    reinterpret_cast<uint2*>(xq)[(int64_t)row * blocks_per_row + b] = codes;
                    const int32_t pos = s_rows[kMaxTopK + k];
                    const int64_t at = sm_k_tiles ? sm_scale_off<4>(pos / kBM, pos % kBM, b, sm_k_tiles)
                                                  : (int64_t)row * blocks_per_row + b;
                    xs[at] = (uint8_t)sb;
                }
            } else if constexpr (kFmt == kQMx8) {
                uint4 codes[2];
                const uint32_t sb = mx8_quant32(f, codes);
                for (int k = 0; k < K; ++k) {
                    const int32_t row = s_rows[k];
                    if (row < 0) continue;
                    uint4* dst = reinterpret_cast<uint4*>(xq) + 2 * ((int64_t)row * blocks_per_row + b);
                    dst[0] = codes[0];
                    dst[1] = codes[1];
                    xs[(int64_t)row * blocks_per_row + b] = (uint8_t)sb;
                }
            } else {
                uint4 codes;
                const uint32_t sb = mx_quant32(f, codes);
                for (int k = 0; k < K; ++k) {
                    const int32_t row = s_rows[k];
                    if (row < 0) continue;
                    reinterpret_cast<uint4*>(xq)[(int64_t)row * blocks_per_row + b] = codes;
                    const int32_t pos = s_rows[kMaxTopK + k];
                    const int64_t at = sm_k_tiles ? sm_scale_off(pos / kBM, pos % kBM, b, sm_k_tiles)
                                                  : (int64_t)row * blocks_per_row + b;
                    xs[at] = (uint8_t)sb;
                }
            }
        }
    }
    __syncthreads();   // s_rows is reused by the caller's next token
}

// MX quantisation of 32-element blocks [first, blocks) with stride `stride` (one block per
// thread and step: four 16-byte loads, a 16-byte code store and a scale byte).
// With sm_k_tiles > 0 the scales go to the stage-major layout (rows of blocks_per_row blocks).
__device__ __forceinline__ void act_quant_blocks(const uint4* __restrict__ x8, uint4* __restrict__ codes16,
                                                 uint8_t* __restrict__ sf, int64_t blocks, int64_t first,
                                                 int64_t stride, int64_t blocks_per_row = 0,
                                                 int64_t sm_k_tiles = 0) {
    for (int64_t b = first; b < blocks; b += stride) {
        float f[32];
        load_bf16_block<4>(x8 + 4 * b, f);
        uint4 codes;
        const uint8_t e = (uint8_t)mx_quant32(f, codes);
        if (sm_k_tiles) {
            const int64_t row = b / blocks_per_row, blk = b - row * blocks_per_row;
            sf[sm_scale_off(row / kBM, row % kBM, blk, sm_k_tiles)] = e;
        } else {
            sf[b] = e;
        }
        codes16[b] = codes;
    }
}

// MXFP8 quantisation of 32-element blocks [first, blocks) with stride `stride`: four 16-byte
// loads, two 16-byte code stores and a scale byte per block.
__device__ __forceinline__ void act_quant8_blocks(const uint4* __restrict__ x8, uint4* __restrict__ codes16,
                                                  uint8_t* __restrict__ sf, int64_t blocks, int64_t first,
                                                  int64_t stride) {
    for (int64_t b = first; b < blocks; b += stride) {
        float f[32];
        load_bf16_block<4>(x8 + 4 * b, f);
        uint4 codes[2];
        sf[b] = (uint8_t)mx8_quant32(f, codes);
        codes16[2 * b] = codes[0];
        codes16[2 * b + 1] = codes[1];
    }
}

// out[t, c] = bf16( sum_k w[t,k] * y[row_of[t,k], c] ), float32, slot order, no FMA, for
// 8-column groups [first, groups) with stride `stride`. kFresh: y and row_of were written
// earlier in the same kernel, so they are read through L2 (ld.global.cg), not the read-only
// path.
template <bool kFresh>
__device__ __forceinline__ void combine_groups(const uint4* __restrict__ y8, const int32_t* __restrict__ row_of,
                                               const float* __restrict__ w, uint4* __restrict__ out8, int64_t groups,
                                               int64_t groups_per_row, int K, int64_t first, int64_t stride) {
    for (int64_t g = first; g < groups; g += stride) {
        const int64_t t = g / groups_per_row;
        const int64_t c = g - t * groups_per_row;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        // eight slots at a time: every row index, then every y load, are issued before the
        // first sum, so the slots' DRAM reads overlap; the sums still run in slot order
        for (int k0 = 0; k0 < K; k0 += 8) {
            int32_t r[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                r[j] = k0 + j < K ? (kFresh ? __ldcg(row_of + t * K + k0 + j) : __ldg(row_of + t * K + k0 + j)) : -1;
            uint4 yv[8];
            float wk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                yv[j] = make_uint4(0u, 0u, 0u, 0u);
                wk[j] = 0.0f;
                if (r[j] >= 0) {
                    wk[j] = __ldg(w + t * K + k0 + j);
                    yv[j] = kFresh ? __ldcg(y8 + (int64_t)r[j] * groups_per_row + c)
                                   : __ldg(y8 + (int64_t)r[j] * groups_per_row + c);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (r[j] < 0) continue;
                const uint32_t yw[4] = {yv[j].x, yv[j].y, yv[j].z, yv[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wk[j], bf16_to_f32(yw[i] & 0xFFFFu)));
                    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wk[j], bf16_to_f32(yw[i] >> 16)));
                }
            }
        }
        out8[g] = make_uint4(f32_to_bf16(acc[0]) | (f32_to_bf16(acc[1]) << 16),
                             f32_to_bf16(acc[2]) | (f32_to_bf16(acc[3]) << 16),
                             f32_to_bf16(acc[4]) | (f32_to_bf16(acc[5]) << 16),
                             f32_to_bf16(acc[6]) | (f32_to_bf16(acc[7]) << 16));
    }
}

}  // namespace mx
