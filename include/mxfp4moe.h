/*
 * mxfp4moe.h -- C ABI of the GB300 (sm_103a) MXFP4 mixture-of-experts expert FFN library.
 *
 * The operations follow three pages of developer notes (cited by page title and section):
 *   [FMT]  "2026-05-08 DeepSeek V4 Pro NVFP4 Quantization" -- "FP4 (E2M1) expert weight
 *          format confirmed" (w1/w3 int8 [3072, 3584] + E8M0 [3072, 224] -> [3072, 7168];
 *          w2 int8 [7168, 1536] + E8M0 [7168, 96] -> [7168, 3072]; code 0 = +0, code 8 = -0).
 *   [DQ]   same page -- "Script update: dequant_fp8_to_bf16.py now handles ALL compressed
 *          types", item 1 (FP8 E4M3 x E8M0 per 128x128 block -> BF16) and item 2 (two E2M1
 *          values per byte, lower nibble first, LUT x E8M0 scale per row per 32 columns).
 *   [PIPE] "Current Bug: vLLM produces empty/garbage output" -- "Phase 1: CuTeDSL Shared
 *          Expert Kernel" (L1 GEMM -> SiLU -> re-quant -> L2 GEMM; MoE = that plus routing,
 *          top-k and scatter; gate/up stacked; shared expert = one group, no routing;
 *          cudagraph-safe with pre-allocated buffers).
 *   [BF16] same page -- "Phase 3: Clean up" (BF16 only for the SiLU activation and the
 *          final scatter).
 *   [GS]   same page -- "Phase 1: CuTeDSL Shared Expert Kernel" (warm-up-based activation
 *          global scale "gs") and "Phase 2: CuTeDSL Attention Kernel" (a per-tensor weight
 *          global scale; the MoE's gate and up carry different ones).
 *
 * Conventions for every call below:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library allocates no
 *     device memory, never synchronises the stream (except mx_device_status) and launches
 *     its kernels asynchronously on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream). Calls are safe to capture in a CUDA graph.
 *   - Layouts are row-major. MXFP4 tensors are a code tensor uint8 [rows, cols/2] (byte j
 *     holds logical column 2j in its low nibble, 2j+1 in its high nibble) plus a scale
 *     tensor uint8 [rows, cols/32] of E8M0 bytes (value 2^(b-127), b = 255 is NaN). The
 *     checkpoint's int8 code dtype is read as raw bytes. BF16 tensors are uint16 bit
 *     patterns. Weights are in the nn.Linear [out, in] layout (K contiguous).
 *   - Base pointers must be 16-byte aligned (MX_ERR_MISALIGNED otherwise).
 *   - Arguments are validated before anything is launched; on any error nothing is launched.
 *     A CUDA launch error maps to MX_ERR_CUDA.
 *   - Kernels never trap. Every device-side wait is bounded; a wait that runs out records a
 *     code and the kernel returns early. A call with a workspace records it in the
 *     workspace's status word (its first 16 bytes; the call's first kernel clears it), read
 *     for one stream by mx_check_workspace(); every call also records it in a device-wide
 *     word that mx_device_status() reads (and optionally clears).
 *   - NaN results are written as 0x7FC0 with the element's sign bit.
 */
#ifndef MXFP4MOE_H
#define MXFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MX_OK = 0,
    MX_ERR_INVALID_ARG = 1,     /* null pointer, negative or inconsistent size           */
    MX_ERR_UNSUPPORTED = 2,     /* size outside what the kernels support (see each call) */
    MX_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned                      */
    MX_ERR_WORKSPACE = 4,       /* workspace missing or smaller than the size query      */
    MX_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed                  */
    MX_ERR_DEVICE_TIMEOUT = 6   /* a bounded device-side wait ran out (mx_device_status) */
} mx_status;

typedef void* mx_stream_t;      /* cudaStream_t */

/* Human-readable name of a status code. Never returns NULL. */
const char* mx_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int mx_version(void);

/* Synchronises the current device, then returns MX_OK or MX_ERR_DEVICE_TIMEOUT from the
 * device status word that bounded waits set; clears the word when `clear` is non-zero.
 * Returns MX_ERR_CUDA if the synchronisation itself reports an error. */
int mx_device_status(int clear);

/*
 * mx_check_workspace -- the device status of the last forward (moe_mxfp4_forward and its
 * variants, moe_nvfp4_forward) launched on `stream` with this workspace ("Current Bug: vLLM
 * produces empty/garbage output", "Phase 1: CuTeDSL Shared Expert Kernel": the experts
 * runner owns pre-allocated buffers; this is their error channel). Waits for `stream` only
 * (other streams keep running), then returns MX_OK, or MX_ERR_DEVICE_TIMEOUT when one of
 * that forward's bounded waits ran out (its output is then incomplete). `clear` != 0 zeroes
 * the word afterwards (the next forward on the workspace zeroes it too, so check before
 * reusing the workspace). Returns MX_ERR_INVALID_ARG for a null workspace,
 * MX_ERR_MISALIGNED unless it is 256-byte aligned, MX_ERR_CUDA if a CUDA call fails.
 */
int mx_check_workspace(const void* workspace, int clear, mx_stream_t stream);

/*
 * mx_selftest_wait_timeout -- exercises the failure path of the bounded device waits: launches
 * a one-thread kernel on `stream` that waits, with the same bounded wait the GEMM pipelines use
 * (about 2 s), on a barrier nothing arrives at. When the wait runs out the kernel records a
 * timeout in the device status word and returns; nothing traps and the context stays usable.
 * mx_device_status() then reports MX_ERR_DEVICE_TIMEOUT. For tests only. Returns MX_OK once
 * launched, MX_ERR_CUDA if the launch fails.
 */
int mx_selftest_wait_timeout(mx_stream_t stream);

/*
 * mx_selftest_wait_timeout_ws -- mx_selftest_wait_timeout whose timeout is also recorded in
 * the status word of `workspace` (256-byte aligned device memory of at least 16 bytes), as a
 * forward's would be: mx_check_workspace(workspace, ., stream) then reports
 * MX_ERR_DEVICE_TIMEOUT. For tests only.
 */
int mx_selftest_wait_timeout_ws(void* workspace, mx_stream_t stream);

/*
 * mx_selftest_grid_barrier_timeout -- exercises the failure path of the persistent
 * forward's grid-wide barrier: zeroes the barrier counter of `workspace` (256-byte aligned
 * device memory of at least 512 bytes) on `stream`, then launches two CTAs cooperatively
 * that wait, with that barrier's bounded wait (about 2 s), for one arrival more than there
 * are CTAs. The waits run out, the kernel records MX_ERR_DEVICE_TIMEOUT in the workspace's
 * status word and the device-wide word, and returns. For tests only.
 */
int mx_selftest_grid_barrier_timeout(void* workspace, mx_stream_t stream);

/*
 * mxfp4_dequant -- MXFP4 -> BF16 ([DQ] item 2, [FMT]).
 *   out[r, c] = bf16( E2M1(nibble(codes[r, c/2], c%2)) * 2^(sf[r, c/32] - 127) )
 *   codes uint8 [rows, cols/2], sf uint8 [rows, cols/32], out uint16 [rows, cols].
 *   cols must be a positive multiple of 32 (MX_ERR_UNSUPPORTED otherwise); rows >= 0
 *   (rows == 0 launches nothing). The result is exact whenever it is finite. Stacked
 *   expert tensors [E, R, C/2] are passed as rows = E * R.
 */
int mxfp4_dequant(const uint8_t* codes, const uint8_t* sf, void* out_bf16,
                  int64_t rows, int64_t cols, mx_stream_t stream);

/*
 * nvfp4_dequant -- NVFP4 -> BF16 ("Current Bug: vLLM produces empty/garbage output",
 * "What we know": the NVFP4 weights dequantised to BF16; "Phase 2: CuTeDSL Attention
 * Kernel": one float32 global scale per tensor, weight_scale_2).
 *   out[r, c] = bf16( float32( E2M1(nibble(codes[r, c/2], c%2)) * e4m3(sf[r, c/16]) * global ) )
 *   codes uint8 [rows, cols/2] (two E2M1 per byte, lower nibble first), sf uint8
 *   [rows, cols/16] (E4M3 "fn" bytes), global_scale float32, out uint16 [rows, cols].
 *   E2M1 * E4M3 is exact in float32; the product with the global scale is rounded once to
 *   float32 and then to BF16, both to nearest even. A NaN result (NaN scale byte, NaN
 *   global, or zero times an infinite global) is 0x7FC0 with the XOR of the three sign
 *   bits. cols must be a positive multiple of 16 (MX_ERR_UNSUPPORTED otherwise); codes
 *   8-byte and out 16-byte aligned (MX_ERR_MISALIGNED); rows == 0 launches nothing.
 */
int nvfp4_dequant(const uint8_t* codes, const uint8_t* sf_e4m3, float global_scale, void* out_bf16,
                  int64_t rows, int64_t cols, mx_stream_t stream);

/*
 * nvfp4_tiled_scales_bytes / nvfp4_scales_to_tiled -- the tile layout above for an NVFP4
 * scale tensor sf uint8 [rows, cols/16] (E4M3 bytes, one per 16 columns): its 4-byte
 * words (four scales, 64 columns) take the place of the MXFP4 K-words. cols % 64 == 0.
 */
size_t nvfp4_tiled_scales_bytes(int64_t rows, int64_t cols);
int nvfp4_scales_to_tiled(const uint8_t* sf, uint8_t* out, int64_t rows, int64_t cols,
                          mx_stream_t stream);

/*
 * nvfp4_gemm_bf16 -- D = bf16(a_global * b_global * A . B^T) with NVFP4 operands on the
 * tcgen05 tensor cores (kind::mxf4nvf4, scale_vec::4X): the standard NVFP4 GEMM the pages
 * plan for their attention projections ("Current Bug: vLLM produces empty/garbage
 * output", "Phase 2: CuTeDSL Attention Kernel", one global scale per operand).
 *   A codes uint8 [M, K/2] + sa uint8 [M, K/16] (E4M3, row-major); B codes uint8 [N, K/2]
 *   + its E4M3 scales in the tile layout (nvfp4_scales_to_tiled of [N, K/16]);
 *   D uint16 [M, N]. The block-scaled products accumulate in float32; the sum is
 *   multiplied by the float32 product of the globals and rounded once to BF16.
 *   The tensor cores read the scale bytes as unsigned E4M3: every scale byte of A and B
 *   must lie in 0x00..0x7E (sign bit clear, not NaN). The library cannot check device
 *   data; a byte outside that range gives a result other than the signed-E4M3 reading.
 *   K must be a positive multiple of 128, N a positive multiple of 16; M >= 0.
 */
int nvfp4_gemm_bf16(const uint8_t* a, const uint8_t* sa, float a_global, const uint8_t* b,
                    const uint8_t* sb_tiled, float b_global, void* d_bf16, int64_t M, int64_t N,
                    int64_t K, mx_stream_t stream);

/*
 * nvfp4_gemm_bf16_multi -- a fused NVFP4 projection: B is nseg weight matrices stacked along
 * N, each with its own global scale ([GS]: the fused q_a + kv projection carries two
 * weight_scale_2 values). Output columns of segment s are
 *   D[:, seg s] = bf16(a_global * b_globals[s] * A . B_s^T),
 * i.e. nvfp4_gemm_bf16 of each segment, computed as one GEMM over the stacked B.
 *   b_globals float32 [nseg] and seg_rows int64 [nseg] are HOST arrays, read during the
 *   call; seg_rows[s] > 0 rows of B each, a multiple of 16; N = sum(seg_rows);
 *   1 <= nseg <= 8 (MX_ERR_UNSUPPORTED above). B's scales: nvfp4_scales_to_tiled of the
 *   stacked [N, K/16] E4M3 scales. Other arguments, layouts and rules as nvfp4_gemm_bf16;
 *   D uint16 [M, N].
 */
int nvfp4_gemm_bf16_multi(const uint8_t* a, const uint8_t* sa, float a_global, const uint8_t* b,
                          const uint8_t* sb_tiled, const float* b_globals, const int64_t* seg_rows,
                          int nseg, void* d_bf16, int64_t M, int64_t K, mx_stream_t stream);

/*
 * fp8_block_dequant_128x128 -- FP8 E4M3 x E8M0 128x128 block scale -> BF16 ([DQ] item 1).
 *   out[i, j] = bf16( e4m3(q[i, j]) * 2^(sf[i/128, j/128] - 127) )
 *   q uint8 [rows, cols] (E4M3 "fn" bytes), sf uint8 [ceil(rows/128), ceil(cols/128)],
 *   out uint16 [rows, cols]. Partial edge blocks use the scale of the block they fall in.
 *   cols must be a positive multiple of 16 (MX_ERR_UNSUPPORTED otherwise).
 */
int fp8_block_dequant_128x128(const uint8_t* q_e4m3, const uint8_t* sf, void* out_bf16,
                              int64_t rows, int64_t cols, mx_stream_t stream);

/*
 * act_quant_mxfp4 -- BF16 -> MXFP4 activation quantisation (the "re-quant" of [PIPE],
 * with the OCP MX rule, which the pages leave open):
 *   per row and per 32-column block: E = clamp(floor(log2 amax) - 2 + 127, 0, 254)
 *   (E = 0 when amax = 0); code = E2M1 round-to-nearest-even of x * 2^(127 - E),
 *   saturating at +-6, sign kept (-0 -> code 8). A block holding NaN/Inf gets E = 255 and
 *   codes sign|7. x uint16 [M, K], codes uint8 [M, K/2], sf uint8 [M, K/32].
 *   K must be a positive multiple of 32.
 */
int act_quant_mxfp4(const void* x_bf16, uint8_t* codes, uint8_t* sf,
                    int64_t M, int64_t K, mx_stream_t stream);

/*
 * act_quant_nvfp4 -- BF16 -> NVFP4 activation quantisation against a float32 global scale g
 * fixed by the caller (calibrated at warm-up, [GS]); the published NVFP4 encoder, which the
 * pages name but do not print. Per row and 16-column block, each step one float32 operation
 * rounded to nearest even:
 *   r = 1 / (6 g); S = the E4M3 byte nearest min(amax * r, 448) (ties to even);
 *   code = E2M1 nearest x * (1 / (e4m3(S) * g)), saturating at +-6, sign kept.
 *   S = 0 gives the codes +-0; a block holding NaN/Inf gets S = 0x7F and codes sign|7.
 *   x uint16 [M, K] (16-byte aligned), codes uint8 [M, K/2] (8-byte aligned), sf uint8
 *   [M, K/16]. The dequantised value is LUT[code] * e4m3(S) * g (nvfp4_dequant).
 *   K must be a positive multiple of 16; g must lie in [2^-117, 2^100] (MX_ERR_INVALID_ARG
 *   otherwise), which keeps every intermediate a normal float.
 */
int act_quant_nvfp4(const void* x_bf16, float global_scale, uint8_t* codes, uint8_t* sf,
                    int64_t M, int64_t K, mx_stream_t stream);

/*
 * act_quant_mxfp8 -- BF16 -> MXFP8 activation quantisation, for the MXFP8-activation variant
 * of the expert FFN (the FP8 reading of the "re-quant" of [PIPE]; the pages leave the format
 * open): the OCP MX rule with E4M3 elements. Per row and 32-column block:
 *   E = clamp(floor(log2 amax) - 8 + 127, 0, 254) (E = 0 when amax = 0);
 *   code = E4M3 ("fn") nearest-even of x * 2^(127 - E), saturating at +-448, sign kept
 *   (-0 -> 0x80). A block holding NaN/Inf gets E = 255 and codes sign|0x7F.
 *   x uint16 [M, K], codes uint8 [M, K] (one E4M3 byte per element), sf uint8 [M, K/32].
 *   K must be a positive multiple of 32; x and codes 16-byte aligned.
 */
int act_quant_mxfp8(const void* x_bf16, uint8_t* codes, uint8_t* sf, int64_t M, int64_t K,
                    mx_stream_t stream);

/*
 * mxfp8_mxfp4_gemm_bf16 -- D = bf16(A . B^T) with MXFP8 A (act_quant_mxfp8's codes and
 * scales) and MXFP4 B on the tcgen05 tensor cores (kind::mxf8f6f4, scale_vec::1X: E4M3 x E2M1
 * products, one E8M0 scale per 32 elements of K on each side, float32 accumulation, one BF16
 * rounding): the GEMM of the MXFP8-activation expert FFN.
 *   A codes uint8 [M, K] + sa uint8 [M, K/32] (row-major); B codes uint8 [N, K/2] (two E2M1
 *   per byte, lower nibble first) + its scales in the tile layout (mxfp4_scales_to_tiled of
 *   [N, K/32]); D uint16 [M, N]. K must be a positive multiple of 128, N of 16; M >= 0.
 *   B must be 32-byte aligned (the tensor-memory-access unit reads it through its 4-bit
 *   type, which needs that), the other pointers 16-byte aligned (MX_ERR_MISALIGNED).
 */
int mxfp8_mxfp4_gemm_bf16(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb_tiled,
                          void* d_bf16, int64_t M, int64_t N, int64_t K, mx_stream_t stream);

/*
 * nvfp4_calibrate_global -- the warm-up calibration of an NVFP4 activation global scale
 * ("Current Bug: vLLM produces empty/garbage output", "Phase 1: CuTeDSL Shared Expert
 * Kernel": a warm-up-based gs), on the GPU. For a calibration batch x uint16 [M, K] (BF16):
 *   *amax         = max(*amax, largest finite |x|)      (NaN and infinities are skipped)
 *   *global_scale = *amax / (6 * 448), one float32 division rounded to nearest even,
 *                   clamped to [2^-117, 2^100] (the range act_quant_nvfp4 accepts)
 * so that the largest magnitude seen quantises to the largest NVFP4 value (E2M1 6 times
 * E4M3 448) without clipping. amax and global_scale are float32 DEVICE pointers (4-byte
 * aligned); *amax is a running maximum over the warm-up batches: set it to 0 before the
 * first call, call once per batch (M = 0 just recomputes the global), then read the global
 * back once and pass it to act_quant_nvfp4 / moe_nvfp4_forward, where it stays a fixed
 * value (the forward remains graph-capturable). x 16-byte aligned; any K > 0.
 */
int nvfp4_calibrate_global(const void* x_bf16, int64_t M, int64_t K, float* amax, float* global_scale,
                           mx_stream_t stream);

/*
 * Tile layout of a scale tensor (the layout the GEMM's tensor-memory copies read).
 * A scale tensor sf uint8 [rows, cols/32] (one E8M0 byte per 32 columns) becomes
 * ceil(rows/128) x (cols/128) blocks of 512 bytes; block (g, w) sits at ((g*(cols/128)) + w)*512
 * and holds at byte l*16 + j*4 + b the scale of row 128g + 32j + l, column block 4w + b
 * (rows past the end are 0). The pages keep scales row-major; this is a re-ordering only.
 *   mxfp4_tiled_scales_bytes: size of the tile layout (0 when cols is not a positive
 *   multiple of 128). mxfp4_scales_to_tiled: converts on `stream`; cols % 128 == 0.
 */
size_t mxfp4_tiled_scales_bytes(int64_t rows, int64_t cols);
int mxfp4_scales_to_tiled(const uint8_t* sf, uint8_t* out, int64_t rows, int64_t cols,
                          mx_stream_t stream);

/*
 * mxfp4_gemm_bf16 -- D = bf16(A . B^T) with MXFP4 operands on the tcgen05 tensor cores:
 * the one-group case of the expert GEMM ([PIPE]: "num_groups=1 is just a regular GEMM").
 *   A codes uint8 [M, K/2] + sa [M, K/32] (row-major scales); B codes uint8 [N, K/2] + sb,
 *   B's scales in the tile layout above (mxfp4_scales_to_tiled of [N, K/32]);
 *   D uint16 [M, N]. Accumulation is float32, the result is rounded once to BF16.
 *   K must be a positive multiple of 128, N a positive multiple of 16; M >= 0.
 */
int mxfp4_gemm_bf16(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                    void* d_bf16, int64_t M, int64_t N, int64_t K, mx_stream_t stream);

/*
 * moe_mxfp4_workspace_size -- bytes of device workspace moe_mxfp4_forward and
 * moe_mxfp4_route need for these sizes (K is ignored when routed == 0). The workspace holds
 * the routing tables, the quantised activations and the L2 output; 256-byte aligned.
 */
size_t moe_mxfp4_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K,
                                int routed);

/*
 * moe_mxfp4_workspace_layout -- byte offsets, inside that workspace, of the intermediate
 * tensors a moe_mxfp4_forward call leaves behind (for inspection and tests; the layout may
 * change between library versions). R = T*K when routed, T otherwise. Writes 8 values:
 *   out[0] xq  uint8  [R, H/2]   MX-quantised x (routed: rows in expert-grouped order)
 *   out[1] xs  uint8             its E8M0 scales, stage-major when routed (below)
 *   out[2] hq  uint8  [R, I/2]   MX-re-quantised h = bf16(silu(g) * u)
 *   out[3] hs  uint8             its E8M0 scales, stage-major when routed
 *   Stage-major, the order the GEMMs read the scales in: rows form M tiles of 128 (routed:
 *   each expert's rows from its first row on, experts in order, so expert e's rows start at
 *   tile sum_{e' < e} ceil(counts[e'] / 128)); the scale of 32-column block b of tile row r
 *   in tile mt is at byte (((mt * S + b / 8) * 2 + (b / 4) % 2) * 128 + r) * 4 + b % 4,
 *   S = ceil(cols / 256). Without routing, and in moe_mxfp4_forward_fused, they are row-major
 *   [R, cols/32].
 *   out[4] y   uint16 [R, H]     BF16 L2 output (routed mode; -1 otherwise)
 *   out[5] row_of int32 [T, K], out[6] counts int32 [E], out[7] offsets int32 [E+1]
 *          (routed mode; -1 otherwise)
 * Returns MX_OK, or the status moe_mxfp4_forward would return for these sizes.
 */
int moe_mxfp4_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed,
                               int64_t* out);

/*
 * moe_mxfp4_forward -- the MoE expert FFN over MXFP4 weights ([PIPE], [BF16]):
 *   xq = act_quant(x);
 *   for each routed pair (t, k) with e = topk_ids[t, k] in [0, E):
 *     g, u = xq[t] . w13[e][0:I]^T, xq[t] . w13[e][I:2I]^T   (gate rows first, then up)
 *     h    = bf16( silu(bf16(g)) * bf16(u) ),  hq = act_quant(h)      (fused epilogue)
 *     y    = bf16( hq . w2[e]^T )
 *   out[t] = bf16( sum_k topk_w[t, k] * y(t, k) )   (float32, slot order k = 0..K-1)
 *   An id outside [0, E) (e.g. -1) contributes nothing; a token with no valid id gets 0.
 *   A NaN in h (a NaN g or u, silu(-inf), 0 * inf) is re-quantised as a positive NaN: its
 *   block's scale byte is 255 and its code 7.
 *   Shared-expert mode: topk_ids == NULL and topk_w == NULL, E must be 1, K is ignored,
 *   out = y.
 *   x uint16 [T, H]; topk_ids int32 [T, K]; topk_w float32 [T, K];
 *   w13 uint8 [E, 2I, H/2], s13 uint8 [E, 2I, H/32]; w2 uint8 [E, H, I/2],
 *   s2 uint8 [E, H, I/32]; out uint16 [T, H] (overwritten, not accumulated).
 *   H and I must be positive multiples of 128 (MX_ERR_UNSUPPORTED otherwise); 1 <= E <= 1024,
 *   1 <= K <= 64; T >= 0 (T == 0 launches nothing). workspace: device memory of at least
 *   moe_mxfp4_workspace_size(T, H, I, E, K, topk_ids != NULL) bytes, 256-byte aligned, not
 *   used by another call that runs at the same time.
 *   Weight scales given here row-major are gathered per GEMM stage; the faster route is to
 *   convert them once at load time and call moe_mxfp4_forward_tiled.
 */
int moe_mxfp4_forward(const void* x, const int32_t* topk_ids, const float* topk_w,
                      const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                      const uint8_t* s2, void* out, int64_t T, int64_t H, int64_t I,
                      int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                      mx_stream_t stream);

/*
 * moe_mxfp4_forward_tiled -- moe_mxfp4_forward with the weight scales already in the tile
 * layout (s13_tiled = mxfp4_scales_to_tiled of s13 viewed as [E*2I, H/32]; s2_tiled of s2
 * viewed as [E*H, I/32]). A weight-format transform done once when the weights are loaded;
 * the GEMMs then fetch each stage's weight scales with two bulk copies instead of one small
 * copy per row. Same arguments, results (bit for bit) and errors otherwise.
 *   This is the fast path: convert the weight scales once at load time and call this entry
 * point. With the checkpoint's row-major scales (moe_mxfp4_forward) each GEMM stage
 * gathers its weight scales as 4-byte copies, which makes the routed prefill forward
 * (T = 8192, H = 7168, I = 3072, 48 experts, top-8) about 25 % slower on a GB300
 * (2.48 ms against 1.98 ms).
 */
int moe_mxfp4_forward_tiled(const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13, const uint8_t* s13_tiled, const uint8_t* w2,
                            const uint8_t* s2_tiled, void* out, int64_t T, int64_t H, int64_t I,
                            int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                            mx_stream_t stream);

/*
 * moe_mxfp4_forward_fused -- moe_mxfp4_forward_tiled as ONE persistent kernel launch (the
 * single-launch MoE kernel of "Current Bug: vLLM produces empty/garbage output", the
 * nvfp4-megamoe-kernel plan, "Phase 1: CuTeDSL Shared Expert Kernel"): one CTA per SM runs
 * the routing, the quantisation of x, the L1 GEMM with its fused SiLU and re-quant, the L2
 * GEMM and the weighted combine, with a grid-wide barrier where the multi-kernel forward
 * starts a new kernel. The phases run the same device code in the same order, so the output
 * is bit-identical to moe_mxfp4_forward_tiled's.
 *   Same arguments, layouts, workspace (moe_mxfp4_workspace_size) and errors as
 * moe_mxfp4_forward_tiled; the weight scales must be in the tile layout. The launch is
 * cooperative (the runtime refuses it, MX_ERR_CUDA, unless every CTA can be resident at
 * once) and is preceded on `stream` by a 4-byte memset of the workspace's barrier counter;
 * both can be captured in a CUDA graph. Each barrier wait is bounded like the pipeline
 * waits: past the limit the kernel records MX_ERR_DEVICE_TIMEOUT in the workspace's status
 * word (mx_check_workspace) and returns.
 */
int moe_mxfp4_forward_fused(const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13, const uint8_t* s13_tiled, const uint8_t* w2,
                            const uint8_t* s2_tiled, void* out, int64_t T, int64_t H, int64_t I,
                            int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                            mx_stream_t stream);

/*
 * moe_mxfp4_forward_timed -- moe_mxfp4_forward (scales_tiled == 0) or
 * moe_mxfp4_forward_tiled (scales_tiled != 0) that also records caller-created
 * cudaEvent_t handles on `stream` at its phase boundaries, for profiling:
 *   events[0] before the first launch, events[1] after the routing permutation,
 *   events[2] after the MX quantisation of x, events[3] after the L1 GEMM,
 *   events[4] after the L2 GEMM, events[5] after the weighted combine.
 * `events` may be NULL and any entry may be NULL. Same arguments and errors otherwise.
 */
int moe_mxfp4_forward_timed(const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                            const uint8_t* s2, void* out, int64_t T, int64_t H, int64_t I,
                            int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                            mx_stream_t stream, void* const* events, int scales_tiled);

/*
 * moe_mxfp4_route -- the routing permutation step of moe_mxfp4_forward on its own
 * ([PIPE]: "routing, topk, scatter"), for inspection and tests.
 *   counts int32 [E]: valid pairs per expert; offsets int32 [E+1]: exclusive prefix sum;
 *   row_of int32 [T, K]: the row of pair (t, k) in the expert-grouped order, which is
 *   sorted by (expert, token, slot); -1 for a dropped pair. Same size rules and workspace
 *   as moe_mxfp4_forward in routed mode.
 */
int moe_mxfp4_route(const int32_t* topk_ids, int64_t T, int64_t K, int64_t E,
                    int32_t* counts, int32_t* offsets, int32_t* row_of,
                    void* workspace, size_t ws_bytes, mx_stream_t stream);

/*
 * moe_nvfp4_forward -- the MoE expert FFN of moe_mxfp4_forward with NVFP4 weights and
 * activations (kind::mxf4nvf4 tensor-core MMAs, E4M3 scales per 16 elements):
 *   xq = act_quant_nvfp4(x, x_global);
 *   for each routed pair (t, k) with e = topk_ids[t, k] in [0, E):
 *     g = bf16( (xq[t] . w13[e][0:I]^T) * x_global * g13[e][0] )    (gate global)
 *     u = bf16( (xq[t] . w13[e][I:2I]^T) * x_global * g13[e][1] )   (up global, [GS])
 *     h = bf16( silu(g) * u ),  hq = act_quant_nvfp4(h, h_global)    (fused epilogue)
 *     y = bf16( (hq . w2[e]^T) * h_global * g2[e] )
 *   out[t] = bf16( sum_k topk_w[t, k] * y(t, k) )   (float32, slot order)
 *   Dot products use the codes times their E4M3 scales (globals excluded), accumulate in
 *   float32 and are scaled once by the float32 product of the two globals.
 *   Routing, shared-expert mode (topk_ids == topk_w == NULL, E == 1), sizes and workspace
 *   rules as moe_mxfp4_forward, with the workspace of moe_nvfp4_workspace_size.
 *   w13 uint8 [E, 2I, H/2] with s13_tiled = nvfp4_scales_to_tiled of its E4M3 scales viewed
 *   as [E*2I, H/16]; w2 uint8 [E, H, I/2] with s2_tiled from [E*H, I/16]; g13 float32
 *   [E, 2] (gate, up) and g2 float32 [E], device arrays; x_global, h_global as for
 *   act_quant_nvfp4 (MX_ERR_INVALID_ARG outside [2^-117, 2^100]). Weight scale bytes must
 *   lie in 0x00..0x7E (nvfp4_gemm_bf16); the library does not read device data to check.
 */
int moe_nvfp4_forward(const void* x, const int32_t* topk_ids, const float* topk_w,
                      const uint8_t* w13, const uint8_t* s13_tiled, const float* g13,
                      const uint8_t* w2, const uint8_t* s2_tiled, const float* g2,
                      float x_global, float h_global, void* out, int64_t T, int64_t H,
                      int64_t I, int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                      mx_stream_t stream);

/* moe_nvfp4_forward recording the six phase events of moe_mxfp4_forward_timed. */
int moe_nvfp4_forward_timed(const void* x, const int32_t* topk_ids, const float* topk_w,
                            const uint8_t* w13, const uint8_t* s13_tiled, const float* g13,
                            const uint8_t* w2, const uint8_t* s2_tiled, const float* g2,
                            float x_global, float h_global, void* out, int64_t T, int64_t H,
                            int64_t I, int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                            mx_stream_t stream, void* const* events);

/*
 * moe_mxfp4w_mxfp8a_forward -- the MoE expert FFN of moe_mxfp4_forward_tiled with MXFP8
 * activations over the same MXFP4 weights (the FP8 reading of [PIPE]'s "re-quant": both
 * activation quantisations use act_quant_mxfp8's rule; the GEMMs are
 * mxfp8_mxfp4_gemm_bf16's):
 *   xq = act_quant_mxfp8(x); g, u = xq[t] . w13[e]^T (gate, up);
 *   h = bf16(silu(bf16(g)) * bf16(u)), hq = act_quant_mxfp8(h) (fused epilogue);
 *   y = bf16(hq . w2[e]^T); out[t] = bf16(sum_k topk_w[t, k] * y(t, k)).
 *   Arguments, routing, shared-expert mode and errors as moe_mxfp4_forward_tiled (weight
 *   scales in the tile layout), with the workspace of moe_mxfp4w_mxfp8a_workspace_size; H
 *   and I multiples of 128; w13 and w2 32-byte aligned (MX_ERR_MISALIGNED).
 */
int moe_mxfp4w_mxfp8a_forward(const void* x, const int32_t* topk_ids, const float* topk_w,
                              const uint8_t* w13, const uint8_t* s13_tiled, const uint8_t* w2,
                              const uint8_t* s2_tiled, void* out, int64_t T, int64_t H, int64_t I,
                              int64_t E, int64_t K, void* workspace, size_t ws_bytes,
                              mx_stream_t stream);

/* moe_mxfp4w_mxfp8a_forward recording the six phase events of moe_mxfp4_forward_timed. */
int moe_mxfp4w_mxfp8a_forward_timed(const void* x, const int32_t* topk_ids, const float* topk_w,
                                    const uint8_t* w13, const uint8_t* s13_tiled, const uint8_t* w2,
                                    const uint8_t* s2_tiled, void* out, int64_t T, int64_t H,
                                    int64_t I, int64_t E, int64_t K, void* workspace,
                                    size_t ws_bytes, mx_stream_t stream, void* const* events);

/*
 * moe_mxfp4w_mxfp8a_workspace_size / _layout -- as the moe_mxfp4_ pair, for
 * moe_mxfp4w_mxfp8a_forward: xq [R, H] and hq [R, I] hold one E4M3 byte per element.
 */
size_t moe_mxfp4w_mxfp8a_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K,
                                        int routed);
int moe_mxfp4w_mxfp8a_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K,
                                       int routed, int64_t* out);

/*
 * moe_nvfp4_workspace_size / moe_nvfp4_workspace_layout -- as the moe_mxfp4_ pair, for
 * moe_nvfp4_forward: xs and hs hold E4M3 scales, one per 16 columns. Routed, they are
 * stage-major with four words per stage: the scale of 16-column block b of tile row r in
 * tile mt is at byte (((mt * S + b / 16) * 4 + (b / 4) % 4) * 128 + r) * 4 + b % 4,
 * S = ceil(cols / 256); without routing they are row-major [R, cols/16].
 */
size_t moe_nvfp4_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K,
                                int routed);
int moe_nvfp4_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t K, int routed,
                               int64_t* out);

/* Bytes of the static device scratch area moe_mxfp4_forward_noalloc runs on (per device). */
#define MXFP4MOE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * moe_mxfp4_forward_noalloc -- moe_mxfp4_forward for callers that cannot allocate device
 * memory. The pages have no counterpart of this call; it exists for callers that receive
 * only their input and output buffers and may not allocate any device memory themselves:
 * a plugin or custom-op interface whose host framework owns every allocation and offers no
 * workspace, code that must not pay cudaMalloc's implicit device-wide synchronisation, or
 * a process whose device memory is entirely reserved by another allocator.
 *   Same arguments, results and errors as moe_mxfp4_forward, minus the workspace: the
 * call runs on a scratch area of MXFP4MOE_NOALLOC_SCRATCH_BYTES (32 MiB) that is a static
 * array inside the library, present on every device that loads it until the process
 * exits. The call itself allocates nothing.
 *   Limit: when moe_mxfp4_workspace_size(T, H, I, E, K, topk_ids != NULL) exceeds
 * MXFP4MOE_NOALLOC_SCRATCH_BYTES the call returns MX_ERR_WORKSPACE and launches nothing
 * (for H = 7168, I = 3072, top-8 that is about 200 routed tokens; use moe_mxfp4_forward
 * with a caller workspace for larger batches).
 *   The first call on each device looks up the scratch area's device address
 * (cudaGetSymbolAddress) with that device current. Under CUDA's lazy module loading (the
 * default) that lookup is also what loads the library's device code and creates the
 * 32 MiB array on that device, so the first call may itself take device memory and
 * synchronise: make it once per device at initialisation (a call with T = 1 will do),
 * before other allocators reserve the device's memory and before any stream capture.
 * Later calls allocate nothing. All calls on a device share the one scratch area and it
 * keeps the last call's contents (no result depends on them): calls that may overlap on
 * the GPU (different streams, or different host threads without ordering) race on it and
 * must be serialised by the caller.
 */
int moe_mxfp4_forward_noalloc(const void* x, const int32_t* topk_ids, const float* topk_w,
                              const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                              const uint8_t* s2, void* out, int64_t T, int64_t H, int64_t I,
                              int64_t E, int64_t K, mx_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4MOE_H */
