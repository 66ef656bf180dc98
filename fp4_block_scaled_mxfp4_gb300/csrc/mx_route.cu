// mx_route.cu -- routing permutation for the MoE ("Current Bug: vLLM produces empty/garbage
// output", "Phase 1: CuTeDSL Shared Expert Kernel": the MoE pipeline is the shared-expert
// pipeline plus routing, top-k and scatter).
//
// The routed (token, slot) pairs are grouped by expert in a stable order: expert, then
// token, then slot. Three launches, no host synchronisation (graph-capturable):
//   1. route_count: per chunk of 2048 pairs, per-expert counts and each pair's rank among
//      the earlier pairs of its expert inside the chunk (warp match + a per-warp scan);
//   2. route_scan (one CTA): per-expert prefix over chunks, expert offsets, and the list of
//      128-row M tiles (expert, first row, valid rows) that the grouped GEMMs walk;
//   3. quant_gather: row_of[t, k] = offsets[e] + chunk_base[chunk, e] + rank, and the
//      quantisation of each token row (MXFP4, or NVFP4 against the activation's global scale)
//      written once per routed pair into the grouped rows.
#include <type_traits>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {

namespace {

constexpr int kCountThreads = 256;
constexpr int kCountWarps = kCountThreads / 32;

__global__ void __launch_bounds__(kCountThreads) route_count_kernel(const int32_t* __restrict__ ids,
                                                                    int64_t n_pairs, int E,
                                                                    int32_t* __restrict__ chunk_counts,
                                                                    int32_t* __restrict__ local_rank,
                                                                    uint32_t* clear_word) {
    __shared__ int32_t s_run[kMaxExperts];
    __shared__ int32_t s_warp[kCountWarps][kMaxExperts];
    pdl_wait();
    // the forward's first kernel: its workspace status word starts at zero
    if (clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *clear_word = 0u;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kCountThreads) s_run[e] = 0;
    const int64_t base = (int64_t)blockIdx.x * kRouteChunk;
    for (int round = 0; round < kRouteChunk / kCountThreads; ++round) {
        for (int i = tid; i < kCountWarps * E; i += kCountThreads) s_warp[i / E][i % E] = 0;
        __syncthreads();
        const int64_t p = base + (int64_t)round * kCountThreads + tid;
        const int32_t e = (p < n_pairs) ? __ldg(ids + p) : -1;
        const bool valid = (e >= 0) && (e < E);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1);
        const uint32_t below = peers & ((1u << lane) - 1u);
        const int rank_in_warp = __popc(below);
        if (valid && rank_in_warp == 0) s_warp[warp][e] = __popc(peers);
        __syncthreads();
        for (int x = tid; x < E; x += kCountThreads) {
            int32_t run = s_run[x];
#pragma unroll
            for (int w = 0; w < kCountWarps; ++w) {
                const int32_t c = s_warp[w][x];
                s_warp[w][x] = run;
                run += c;
            }
            s_run[x] = run;
        }
        __syncthreads();
        if (valid) local_rank[p] = s_warp[warp][e] + rank_in_warp;
        __syncthreads();
    }
    for (int e = tid; e < E; e += kCountThreads) chunk_counts[(int64_t)blockIdx.x * E + e] = s_run[e];
    pdl_launch_dependents();
}

__global__ void __launch_bounds__(1024) route_scan_kernel(const int32_t* __restrict__ chunk_counts,
                                                          int64_t nchunks, int E, RouteBufs rb) {
    __shared__ int32_t s_cnt[kMaxExperts];
    __shared__ int32_t s_off[kMaxExperts + 1];
    __shared__ int32_t s_toff[kMaxExperts + 1];
    pdl_wait();
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) {
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
        *rb.num_mtiles = toff;
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        rb.counts[e] = s_cnt[e];
        rb.offsets[e] = s_off[e];
        const int32_t nt = (s_cnt[e] + kBM - 1) / kBM;
        for (int32_t m = 0; m < nt; ++m) {
            const int32_t idx = s_toff[e] + m;
            rb.tile_expert[idx] = e;
            rb.tile_row0[idx] = s_off[e] + m * kBM;
            rb.tile_rows[idx] = min(kBM, s_cnt[e] - m * kBM);
        }
    }
    pdl_launch_dependents();
}

constexpr int kGatherThreads = 256;

// One thread per block of the token's row -- MXFP4: 32 elements, four 16-byte loads, a
// 16-byte code store; NVFP4 (kNv, global g): 16 elements, two loads, an 8-byte store --
// then per routed copy of the row the codes and a scale byte, so a warp writes 512 (256)
// contiguous code bytes and 32 contiguous scale bytes per destination row.
template <bool kNv>
__global__ void __launch_bounds__(kGatherThreads) quant_gather_kernel(
    const uint4* __restrict__ x8, const int32_t* __restrict__ ids, int K, int E, int64_t blocks_per_row,
    RouteBufs rb, uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, float g) {
    using Codes = typename std::conditional<kNv, uint2, uint4>::type;
    constexpr int kLoads = kNv ? 2 : 4;
    __shared__ int32_t s_rows[kMaxTopK];
    pdl_wait();
    const int64_t t = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid < K) {
        const int64_t p = t * K + tid;
        const int32_t e = __ldg(ids + p);
        int32_t row = -1;
        if (e >= 0 && e < E)
            row = rb.offsets[e] + rb.chunk_base[(p / kRouteChunk) * E + e] + rb.local_rank[p];
        s_rows[tid] = row;
        rb.row_of[p] = row;
    }
    __syncthreads();
    const uint4* xrow = x8 + t * blocks_per_row * kLoads;
    Codes* xqc = reinterpret_cast<Codes*>(xq);
    const float r = kNv ? __frcp_rn(__fmul_rn(6.0f, g)) : 0.0f;
    for (int64_t b = tid; b < blocks_per_row; b += kGatherThreads) {
        float f[8 * kLoads];
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const uint4 v = __ldg(xrow + kLoads * b + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[8 * i + 2 * j] = bf16_to_f32(w[j] & 0xFFFFu);
                f[8 * i + 2 * j + 1] = bf16_to_f32(w[j] >> 16);
            }
        }
        Codes codes;
        uint32_t sb;
        if constexpr (kNv)
            sb = nv_quant16(f, g, r, codes);
        else
            sb = mx_quant32(f, codes);
        for (int k = 0; k < K; ++k) {
            const int32_t row = s_rows[k];
            if (row < 0) continue;
            xqc[(int64_t)row * blocks_per_row + b] = codes;
            xs[(int64_t)row * blocks_per_row + b] = (uint8_t)sb;
        }
    }
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_route(const int32_t* ids, int64_t T, int64_t K, int64_t E, const RouteBufs& rb,
                         cudaStream_t s, uint32_t* clear_word) {
    const int64_t n = T * K;
    if (n == 0) return cudaSuccess;
    const cudaError_t err = launch_pdl(route_count_kernel, dim3((unsigned)rb.nchunks), dim3(kCountThreads), 0, s, ids,
                                       n, (int)E, rb.chunk_counts, rb.local_rank, clear_word);
    if (err != cudaSuccess) return err;
    return launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, s, rb.chunk_counts, rb.nchunks, (int)E, rb);
}

cudaError_t launch_quant_gather(const uint16_t* x, const int32_t* ids, int64_t T, int64_t K, int64_t E,
                                int64_t H, const RouteBufs& rb, uint8_t* xq, uint8_t* xs, cudaStream_t s,
                                bool nvfp4, float global_scale) {
    if (T == 0) return cudaSuccess;
    if (nvfp4)
        return launch_pdl(quant_gather_kernel<true>, dim3((unsigned)T), dim3(kGatherThreads), 0, s,
                          reinterpret_cast<const uint4*>(x), ids, (int)K, (int)E, (int64_t)(H / 16), rb, xq, xs,
                          global_scale);
    return launch_pdl(quant_gather_kernel<false>, dim3((unsigned)T), dim3(kGatherThreads), 0, s,
                      reinterpret_cast<const uint4*>(x), ids, (int)K, (int)E, (int64_t)(H / 32), rb, xq, xs, 0.0f);
}

}  // namespace mx
