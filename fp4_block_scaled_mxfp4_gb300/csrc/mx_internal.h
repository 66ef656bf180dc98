// mx_internal.h -- launcher interfaces between the C-ABI layer (mx_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mx {

// Where a bounded device wait that runs out reports (either may be null): the caller's
// workspace word, which the forward's first kernel clears and mx_check_workspace reads,
// and the device-wide word that mx_device_status reads.
struct StatusWords {
    uint32_t* ws;
    uint32_t* dev;
};

// Launch a kernel of the forward with programmatic stream serialisation (see pdl_wait in
// mx_device.cuh): it may be scheduled before the previous kernel in the stream completes and
// waits for it on the device.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- GEMM tile geometry (tcgen05 block-scaled MMA; persistent CTAs walk 128-row x kBN tiles;
// each configuration's stage count is in mx_gemm.cu) ----
constexpr int kBM = 128;           // rows of A per tile (TMEM lanes)
constexpr int kBN = 256;           // columns of the accumulator (L1: 128 gate + 128 up); 128 for small M
constexpr int kBK = 256;           // E2M1 elements of K per pipeline stage (128 bytes)
constexpr int kGemmThreads = 384;  // 4 control warps + 8 epilogue warps

// Routing: pairs per counting block.
constexpr int kRouteChunk = 2048;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 64;
// Stacked weight matrices of one fused NVFP4 projection.
constexpr int kMaxSegments = 8;

// Arguments of the expert GEMM kernels (plain data, copied into the kernel parameters).
struct GemmArgs {
    const uint8_t* sfa;          // A scales [a_rows, K/32]
    const uint8_t* sfb;          // B scales: row-major [b_rows, K/32], or tile layout
                                 // [b_rows/128][K/128][512 B] (b_tiled launches)
    int64_t ld_sf;               // K/32: scale bytes per row (A and B share K)
    int64_t a_rows;              // rows of A (bound for scale loads; TMA zero-fills beyond)
    int64_t b_rows;              // rows of the stacked B tensor
    int64_t b_groups;            // 128-row groups of B's tiled scales
    int64_t kw;                  // scale words (4 bytes) per row: K/128 (MXFP4), K/64 (NVFP4)
    int32_t k_tiles;             // ceil(K / 256)
    int32_t k_tail_half;         // 1 when the last stage holds only 128 of K
    // M tiles: from the routing tables (device) or uniform over m_total rows.
    const int32_t* tile_expert;  // nullptr -> uniform tiling
    const int32_t* tile_row0;
    const int32_t* tile_rows;
    const int32_t* num_mtiles_dev;
    int32_t num_mtiles_host;
    int64_t m_total;
    int32_t n_tiles;             // tiles along N per M tile
    int64_t b_rows_per_expert;   // L1: 2I, L2: N
    int64_t n_half;              // L1: I (first up row); L2: 0
    int64_t n_valid;             // L1: I; L2: N (columns that exist)
    // outputs
    uint8_t* hq;                 // L1: requantised activation codes [rows, I/2]
    uint8_t* hs;                 // L1: its scales [rows, I/32] (NVFP4: [rows, I/16])
    int64_t ld_hq, ld_hs;
    uint16_t* y;                 // L2: BF16 output [rows, ld_y]
    int64_t ld_y;
    StatusWords status;          // where a wait that runs out reports
    // NVFP4 only. Without w_global the output is scaled by alpha (the product of the two
    // operands' globals). With it, alpha is the activation's global and each expert's
    // weight global(s) multiply it in the kernel: L1 w_global[2e] (gate), [2e + 1] (up);
    // L2 w_global[e]. q_global is the global of L1's NVFP4 re-quantisation of h.
    float alpha;
    const float* w_global;
    float q_global;
    // NVFP4 L2 with nseg > 0: B is nseg weight matrices stacked along N (a fused projection);
    // output columns below seg_end[s] (and at or above seg_end[s - 1]) are scaled by
    // seg_alpha[s] instead of alpha. Boundaries are multiples of 16.
    int32_t nseg;
    int32_t seg_end[kMaxSegments];
    float seg_alpha[kMaxSegments];
    // MXFP4 forward: A's scales in the stage-major layout (sm_scale_off) instead of row-major
    // [a_rows, K/32]; with hs_k_tiles > 0, L1 writes h's scales that way too (hs_k_tiles =
    // ceil(I / 256), the K stages of L2).
    int32_t a_sm;
    int32_t hs_k_tiles;
};

size_t gemm_smem_bytes();
// n_cols: the tile's width, 256 (L1: 128 gate + 128 up columns) or 128 (64 + 64), used where
// 256-wide tiles would leave SMs idle. tb: B in boxes of 128 bytes x n_cols rows (L1: the 4-D
// w13 view with n_cols / 2 rows of each half). ty: the output as a 2-D tensor map, no swizzle,
// boxes of 32 rows x 32 bytes (L2 BF16; L1 codes with n_cols = 256) or 32 rows x 16 bytes
// (L1 codes with n_cols = 128): L1 the codes hq [rows, ld_hq], L2 the BF16 y [rows, ld_y].
cudaError_t launch_gemm_l1(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                           int grid, bool b_tiled, int n_cols, cudaStream_t s);
cudaError_t launch_gemm_l2(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                           int grid, bool b_tiled, int n_cols, cudaStream_t s);

// NVFP4 GEMMs (256-column tiles): A codes with row-major E4M3 scales per 16 (a.sfa,
// ld_sf = K/16), B codes with E4M3 scales in the tile layout (a.sfb, kw = K/64); tb in
// boxes of 256 rows (L1: the 4-D w13 view, 128 rows of each half); K % 128 == 0. L2: BF16
// out; L1: SiLU(gate) * up re-quantised to NVFP4 with a.q_global (scales [rows, I/16]).
cudaError_t launch_gemm_nvfp4(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                              int grid, cudaStream_t s);
cudaError_t launch_gemm_nvfp4_l1(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty,
                                 const GemmArgs& a, int grid, cudaStream_t s);

// The whole routed (or shared-expert) MXFP4 forward as one persistent cooperative launch:
// routing, quantisation of x, L1, L2 and the combine, separated by grid-wide barriers.
// Weight scales in the tile layout; both GEMMs run tiles of kN = n_cols columns.
struct RouteBufs;
struct FusedArgs;
cudaError_t launch_moe_fused(const CUtensorMap& ta1, const CUtensorMap& tb1, const CUtensorMap& ty1,
                             const CUtensorMap& ta2, const CUtensorMap& tb2, const CUtensorMap& ty2,
                             const FusedArgs& fa, int n_cols, int num_sms, cudaStream_t s);
// Failure-path self-test of the grid-wide barrier: a cooperative launch of two CTAs waits on a
// barrier count no arrival reaches (counter must be zero, in device memory).
cudaError_t launch_grid_sync_probe(uint32_t* counter, StatusWords status, cudaStream_t s);

// MXFP8 activations over MXFP4 weights (kind::mxf8f6f4, 256-column tiles, tile-layout weight
// scales; K % 128 == 0, k_tiles = K / 128): ta E4M3 codes [rows, K] in boxes of 128 rows x
// 128 bytes; tb the E2M1 weights through a 16U4_ALIGN16B map (boxes of 128 elements, L1 the
// 4-D w13 view); L1 re-quantises h to MXFP8 (codes [rows, I], ty in boxes of 32 rows x 32
// bytes), L2 writes BF16.
cudaError_t launch_gemm_a8(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                           int grid, bool l1, cudaStream_t s);

// ---- element-wise kernels ----
// Scale tensor [rows, kb] -> tile layout [ceil(rows/128)][kb/4][512 B] (kb % 4 == 0).
cudaError_t launch_sf_tile(const uint8_t* sf, uint8_t* out, int64_t rows, int64_t kb, cudaStream_t s);
cudaError_t launch_mxfp4_dequant(const uint8_t* codes, const uint8_t* sf, uint16_t* out, int64_t rows,
                                 int64_t cols, int num_sms, cudaStream_t s);
// NVFP4 codes [rows, cols/2] + E4M3 scales [rows, cols/16] + float32 global -> BF16.
cudaError_t launch_nvfp4_dequant(const uint8_t* codes, const uint8_t* sf, float global_scale, uint16_t* out,
                                 int64_t rows, int64_t cols, int num_sms, cudaStream_t s);
cudaError_t launch_fp8_dequant(const uint8_t* q, const uint8_t* sf, uint16_t* out, int64_t rows,
                               int64_t cols, int num_sms, cudaStream_t s);
// The activation quantisers; clear_word (optional): a forward's workspace status word, set
// to zero once this kernel may touch global memory (the forward's first kernel does this).
// sm_k_tiles > 0 (launch_act_quant only): sf in the stage-major layout with that many K stages.
cudaError_t launch_act_quant(const uint16_t* x, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K,
                             int num_sms, cudaStream_t s, uint32_t* clear_word = nullptr, int64_t sm_k_tiles = 0);
// MXFP8 activation quantisation (E4M3 codes [M, K], E8M0 sf [M, K/32]).
cudaError_t launch_act_quant_mxfp8(const uint16_t* x, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K,
                                   int num_sms, cudaStream_t s, uint32_t* clear_word = nullptr);
// NVFP4 activation quantisation with the float32 global (codes [M, K/2], E4M3 sf [M, K/16]).
cudaError_t launch_act_quant_nvfp4(const uint16_t* x, float global_scale, uint8_t* codes, uint8_t* sf, int64_t M,
                                   int64_t K, int num_sms, cudaStream_t s, uint32_t* clear_word = nullptr);
// NVFP4 activation-global calibration over n BF16 values (x 16-byte aligned): *amax (float32,
// device) becomes the running maximum of the finite |x|, *global_scale = amax / (6 * 448).
cudaError_t launch_nv_calibrate(const uint16_t* x, int64_t n, float* amax, float* global_scale, int num_sms,
                                cudaStream_t s);
// Failure-path self-test: a bounded wait on a barrier nothing arrives at (see mx_elementwise.cu).
cudaError_t launch_wait_probe(StatusWords status, cudaStream_t s);
cudaError_t launch_combine(const uint16_t* y, const int32_t* row_of, const float* w, uint16_t* out,
                           int64_t T, int64_t K, int64_t H, int num_sms, cudaStream_t s);

// ---- routing ----
struct RouteBufs {
    int32_t* chunk_counts;   // [nchunks, E]
    int32_t* chunk_base;     // [nchunks, E]
    int32_t* local_rank;     // [T*K]
    int32_t* counts;         // [E]
    int32_t* offsets;        // [E+1]
    int32_t* row_of;         // [T*K]
    int32_t* tile_expert;    // [max_mtiles]
    int32_t* tile_row0;
    int32_t* tile_rows;
    int32_t* num_mtiles;     // [1]
    int32_t* tile_base;      // [E+1]: index of each expert's first M tile
    int64_t nchunks;
};
// clear_word: as for launch_act_quant.
cudaError_t launch_route(const int32_t* ids, int64_t T, int64_t K, int64_t E, const RouteBufs& rb,
                         cudaStream_t s, uint32_t* clear_word = nullptr);
// Arguments of the persistent forward (launch_moe_fused).
struct FusedArgs {
    GemmArgs g1, g2;             // L1 and L2, as the multi-kernel forward fills them
    const uint16_t* x;           // BF16 [T, H]
    const int32_t* ids;          // [T, K], or null: shared expert (uniform tiling)
    const float* topk_w;         // [T, K]
    uint16_t* out;               // BF16 [T, H]
    uint16_t* y;                 // L2's BF16 rows [R, H] (routed)
    uint8_t* xq;
    uint8_t* xs;
    RouteBufs rb;
    int64_t T, H;
    int32_t K, E;
    uint32_t* sync;              // grid-barrier arrival counter, zero at launch
    uint32_t* clear_word;        // the workspace status word, cleared first
    StatusWords status;
};

// Quantise each token row once (MXFP4, or NVFP4 with the float32 global) and write it to the
// rows of all its routed pairs; also writes row_of (needs launch_route first).
// fmt: 0 MXFP4, 1 NVFP4 (with the global), 2 MXFP8 (E4M3 codes [rows, H]).
// sm_k_tiles > 0 (MXFP4): xs in the stage-major layout with that many K stages.
cudaError_t launch_quant_gather(const uint16_t* x, const int32_t* ids, int64_t T, int64_t K, int64_t E,
                                int64_t H, const RouteBufs& rb, uint8_t* xq, uint8_t* xs,
                                cudaStream_t s, int fmt = 0, float global_scale = 0.0f, int64_t sm_k_tiles = 0);

}  // namespace mx
