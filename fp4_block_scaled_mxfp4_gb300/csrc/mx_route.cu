// mx_route.cu -- routing permutation for the MoE ("Current Bug: vLLM produces empty/garbage
// output", "Phase 1: CuTeDSL Shared Expert Kernel": the MoE pipeline is the shared-expert
// pipeline plus routing, top-k and scatter).
//
// The routed (token, slot) pairs are grouped by expert in a stable order: expert, then
// token, then slot. Three launches (two when all pairs fit in one chunk, whose count and
// scan then share one CTA), no host synchronisation (graph-capturable):
//   1. route_count: per chunk of 2048 pairs, per-expert counts and each pair's rank among
//      the earlier pairs of its expert inside the chunk (warp match + a per-warp scan);
//   2. route_scan (one CTA): per-expert prefix over chunks, expert offsets, and the list of
//      128-row M tiles (expert, first row, valid rows) that the grouped GEMMs walk;
//   3. quant_gather: row_of[t, k] = offsets[e] + chunk_base[chunk, e] + rank, and the
//      quantisation of each token row (MXFP4, or NVFP4 against the activation's global scale)
//      written once per routed pair into the grouped rows.
#include "mx_phases.cuh"

namespace mx {

namespace {

__global__ void __launch_bounds__(kCountThreads) route_count_kernel(const int32_t* __restrict__ ids,
                                                                    int64_t n_pairs, int E,
                                                                    int32_t* __restrict__ chunk_counts,
                                                                    int32_t* __restrict__ local_rank,
                                                                    uint32_t* clear_word) {
    __shared__ int32_t s_buf[(1 + kCountWarps) * kMaxExperts];
    pdl_wait();
    // the forward's first kernel: its workspace status word starts at zero
    if (clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *clear_word = 0u;
    route_count_chunk(ids, n_pairs, E, blockIdx.x, chunk_counts, local_rank, s_buf, s_buf + E, threadIdx.x);
    pdl_launch_dependents();
}

__global__ void __launch_bounds__(1024) route_scan_kernel(const int32_t* __restrict__ chunk_counts,
                                                          int64_t nchunks, int E, RouteBufs rb) {
    __shared__ int32_t s_buf[3 * kMaxExperts + 2];
    pdl_wait();
    route_scan(chunk_counts, nchunks, E, rb, s_buf, s_buf + E, s_buf + 2 * E + 1, threadIdx.x, blockDim.x);
    pdl_launch_dependents();
}

// All pairs in one chunk (decode-sized batches): both routing steps in one CTA, one launch
// fewer. The count's scratch is reused by the scan once the count is done.
constexpr int kSmallRouteThreads = 1024;
constexpr int kSmallRouteSmemInts = (1 + kCountWarps) * kMaxExperts > 3 * kMaxExperts + 2
                                        ? (1 + kCountWarps) * kMaxExperts
                                        : 3 * kMaxExperts + 2;
__global__ void __launch_bounds__(kSmallRouteThreads) route_small_kernel(const int32_t* __restrict__ ids,
                                                                         int64_t n_pairs, int E, RouteBufs rb,
                                                                         uint32_t* clear_word) {
    __shared__ int32_t s_buf[kSmallRouteSmemInts];
    pdl_wait();
    if (clear_word != nullptr && threadIdx.x == 0) *clear_word = 0u;
    route_count_chunk(ids, n_pairs, E, 0, rb.chunk_counts, rb.local_rank, s_buf, s_buf + E, threadIdx.x);
    __syncthreads();   // the chunk's counts (global) are read by other threads of the CTA below
    route_scan(rb.chunk_counts, 1, E, rb, s_buf, s_buf + E, s_buf + 2 * E + 1, threadIdx.x, blockDim.x);
    pdl_launch_dependents();
}

constexpr int kGatherThreads = 256;

// One CTA per token (quant_gather_token).
template <int kFmt>
__global__ void __launch_bounds__(kGatherThreads) quant_gather_kernel(
    const uint4* __restrict__ x8, const int32_t* __restrict__ ids, int K, int E, int64_t blocks_per_row,
    RouteBufs rb, uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, float g, int64_t sm_k_tiles) {
    __shared__ int32_t s_rows[2 * kMaxTopK];
    pdl_wait();
    quant_gather_token<kFmt>(x8, ids, K, E, blocks_per_row, rb, xq, xs, g, blockIdx.x, s_rows, threadIdx.x,
                             kGatherThreads, sm_k_tiles);
    pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_route(const int32_t* ids, int64_t T, int64_t K, int64_t E, const RouteBufs& rb,
                         cudaStream_t s, uint32_t* clear_word) {
    const int64_t n = T * K;
    if (n == 0) return cudaSuccess;
    if (rb.nchunks == 1)
        return launch_pdl(route_small_kernel, dim3(1), dim3(kSmallRouteThreads), 0, s, ids, n, (int)E, rb,
                          clear_word);
    const cudaError_t err = launch_pdl(route_count_kernel, dim3((unsigned)rb.nchunks), dim3(kCountThreads), 0, s, ids,
                                       n, (int)E, rb.chunk_counts, rb.local_rank, clear_word);
    if (err != cudaSuccess) return err;
    return launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, s, rb.chunk_counts, rb.nchunks, (int)E, rb);
}

cudaError_t launch_quant_gather(const uint16_t* x, const int32_t* ids, int64_t T, int64_t K, int64_t E,
                                int64_t H, const RouteBufs& rb, uint8_t* xq, uint8_t* xs, cudaStream_t s,
                                int fmt, float global_scale, int64_t sm_k_tiles) {
    if (T == 0) return cudaSuccess;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    if (fmt == kQNv4)
        return launch_pdl(quant_gather_kernel<kQNv4>, dim3((unsigned)T), dim3(kGatherThreads), 0, s, x8, ids, (int)K,
                          (int)E, (int64_t)(H / 16), rb, xq, xs, global_scale, sm_k_tiles);
    if (fmt == kQMx8)
        return launch_pdl(quant_gather_kernel<kQMx8>, dim3((unsigned)T), dim3(kGatherThreads), 0, s, x8, ids, (int)K,
                          (int)E, (int64_t)(H / 32), rb, xq, xs, 0.0f, (int64_t)0);
    return launch_pdl(quant_gather_kernel<kQMx4>, dim3((unsigned)T), dim3(kGatherThreads), 0, s, x8, ids, (int)K,
                      (int)E, (int64_t)(H / 32), rb, xq, xs, 0.0f, sm_k_tiles);
}

}  // namespace mx
