// mx_gemm.cu -- grouped block-scaled MXFP4 GEMM on the sm_103a tensor cores (tcgen05,
// kind::mxf4, E2M1 x E2M1 with E8M0 scales per 32 elements of K, FP32 accumulation in
// tensor memory), with the two epilogues of the expert FFN:
//   L1: D = A . W13^T over a tile of kN / 2 gate + kN / 2 up columns; the epilogue rounds g
//       and u to BF16, forms h = bf16(silu(g) * u) and re-quantises h to MXFP4 (codes + E8M0),
//       or to NVFP4 in the kNv mode (kind::mxf4nvf4, E4M3 scales per 16 plus global scales).
//   L2: D = A . W2^T over kN output columns; the epilogue writes BF16.
// Tiles are 128 rows x kN columns, kN = 256, or 128 where 256-wide tiles would leave SMs
// idle (see Cfg).
// The pipeline is the one the pages describe for their CuTeDSL experts kernel ("Current
// Bug: vLLM produces empty/garbage output", "Phase 1: CuTeDSL Shared Expert Kernel":
// L1 GEMM -> SiLU -> re-quant -> L2 GEMM; the shared expert is the one-group case), with
// the weight format of "2026-05-08 DeepSeek V4 Pro NVFP4 Quantization", "FP4 (E2M1) expert
// weight format confirmed".
//
// CTA layout (384 threads, one CTA per SM, persistent over the tile list):
//   warp 0      TMA producer: A tile (128 rows x 128 B) and B tile (kN rows x 128 B) per
//               K stage of 256 elements, 128-byte swizzle, into a 4- or 5-stage ring. Two
//               TMA instructions per stage: L1's B is one box of a 4-D view of the stacked
//               gate/up weights holding both halves.
//   warp 1      allocates 512 TMEM columns; lane 0 issues the 4 MMAs (K = 64 each) of a
//               stage and commits the stage free. Nothing else runs in that thread: the
//               tensor core's instruction queue is short, and any other work between two
//               MMAs leaves the pipe idle.
//   warp 2      scale-factor loader: cp.async from the plain row-major [rows, K/32] scales
//               of A (and of B when they are not in tile layout) into the layouts
//               tcgen05.cp reads, adjacent lanes taking the K-words of one row; each lane's
//               copies arrive on the stage's scale barrier when they land
//               (cp.async.mbarrier.arrive), so it never blocks. With B's scales in tile layout
//               (kBTiled), lane 0 fetches each 128-row group's blocks with one bulk copy on the
//               same barrier, except for L1's 128-column tiles, whose gate and up halves each
//               lane takes as 8-byte pieces.
//   warp 3      scale-factor copier: lane 0 waits for a stage's operands and scale tiles,
//               moves the scales into that stage's TMEM slot (tcgen05.cp) and commits the
//               copies to the stage's ready barrier, which the MMA thread waits on.
//   warps 4-11  epilogue: two warps per 32-lane TMEM quarter, each owning half of the
//               columns; they drain the accumulator to registers, release it, then compute.
//               Outputs leave through a 1 KB shared staging block per warp and an
//               asynchronous TMA store (L2: 32 rows x 16 BF16 columns, 32-byte swizzle;
//               L1: 32 rows x 32 bytes of codes, 16 at kN = 128), so the warp never waits
//               for its stores (32 scattered 16-byte row pieces per store instruction
//               otherwise); a warp whose 32 rows are not all in the tile stores directly.
// TMEM: columns [0, kN) accumulator; [256 + 24 s, 256 + 24 s + 24) the scale factors of
// stage s (A: 2 K-words x 4 columns, B: 2 K-words x 8 columns).
//
// What bounds it, measured on all SMs: one K stage takes ~935-950 cycles against 512 cycles
// of MMAs. No single unit is saturated (tensor pipe ~49 % busy, the tensor core's reads of
// shared memory ~40 %), and removing any one factor moves the stage by at most 7 %: the
// tensor pipe's four replicating B-scale copies (~85 cycles each) and A-scale copy (~30),
// the 4-byte scale gathers, a second TMA-issuing thread, one ring stage more or less. Per
// stage the SM's shared memory takes the 48 KB of operands from TMA and serves the same
// 48 KB to the MMAs; a CTA pair that loads half of B per SM is the way to fewer bytes per
// FLOP.
#include <cuda.h>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mx_phases.cuh"

namespace mx {

namespace {

constexpr int kABytes = kBM * kBK / 2;                 // 16 KB
constexpr int kTmemCols = 512;
constexpr int kSfTmemBase = 256;
constexpr int kSfColsPerStage = 24;
constexpr uint32_t kFullArrivals = 1;                  // producer (with the TMA bytes)
constexpr uint32_t kSfArrivals = 32;                   // every scale-loader lane (+1 with bulk copies)
constexpr int kStagingBytes = 1024;                    // per epilogue warp: 32 rows x 32 bytes
constexpr int kMaxStages = 5;

// Scale factors reach tensor memory by tcgen05.cp. The tensor core reads them per 32-row
// slice from that slice's own lane quarter: A's scale of row r at lane r, column r / 32
// (+4 for the stage's second K-word); B's scales, which every slice needs, at every lane of
// each quarter. So B's come by tcgen05.cp.32x128b.warpx4 from 512-byte blocks (32 lanes x
// 16 bytes, replicated into the four quarters), and A's by one tcgen05.cp.128x256b for
// both K-words from a 4 KB image: 128 rows x 32 bytes in 8-row x 16-byte core matrices
// (8-row groups 256 bytes apart, a row's two 16-byte halves 128 bytes apart), row r's word
// at byte 4 (r / 32) of each half. A replicating copy costs the tensor pipe ~85 cycles and
// the 128x256b copy ~30, so this takes a stage from six replicating copies to four (two at
// kN = 128).
//
// kN is the tile's width: 256 columns (L1: 128 gate + 128 up) for the routed forward, 128
// (64 + 64) where a grid of 256-wide tiles would leave SMs idle (the shared expert at a
// few hundred tokens). The narrower tile halves each CTA's work per stage, doubles the
// CTAs, and fits a fifth stage.
//
// kNv: NVFP4 operands (E4M3 scales per 16 elements of K, idesc scale format E4M3): four
// scale words per row and stage instead of two, so two A images, twice B's blocks and
// copies, twice the TMEM columns per slot, and three stages. The accumulator is scaled by
// the operands' global scales in the epilogue (L1: per expert, gate and up separately), and
// L1 re-quantises h to NVFP4 (E4M3 per 16 against h's global).
//
// kA8: MXFP8 activations over the MXFP4 weights (kind::mxf8f6f4, scale_vec::1X): A holds E4M3
// codes, one byte per element; B's E2M1 codes come through a TMA map that spreads each 8
// bytes of 16 codes over 16 bytes of shared memory, the layout this MMA kind reads. A stage
// then covers 128 elements of K (128 bytes per row of A and of B's image), four MMAs of
// K = 32, and one scale word per row (one E8M0 byte per MMA, chosen by the scale ids).
template <int kN, bool kNv = false, bool kA8 = false>
struct Cfg {
    static_assert(!(kNv && kA8), "one operand format per kernel");
    static constexpr int kStages = kNv ? 3 : (kN == 256 ? 4 : 5);
    static constexpr int kBBytes = kN * kBK / 2;                    // 32 or 16 KB
    static constexpr int kKStage = kA8 ? 128 : kBK;                 // elements of K per stage
    // bytes B's TMA box delivers: with kA8 the packed 8-byte chunks only (the 8-byte gap after
    // each is left unwritten), half of the box's 128 bytes per row of shared memory
    static constexpr int kBTxBytes = kA8 ? kBBytes / 2 : kBBytes;
    static constexpr int kWords = kNv ? 4 : (kA8 ? 1 : 2);          // scale words per row and stage
    static constexpr int kWordsHalf = kWords / 2;                   // ... at a K tail of 128
    static constexpr int kImages = (kWords + 1) / 2;                // A's wide images, two words each
    static constexpr int kSfaBytes = kImages * 4096;
    static constexpr int kSfbBytes = (kN / 128) * kWords * 512;     // per 128 rows: kWords x 512 B
    static constexpr int kSfCols = kNv ? 48 : kSfColsPerStage;      // A: 4 per word; B: 8 per word
    static constexpr uint32_t kIdesc = kNv ? (idesc_mxf4(kBM, kN) & ~(1u << 23))
                                           : (kA8 ? idesc_mxf8_e2m1(kBM, kN) : idesc_mxf4(kBM, kN));
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr uint32_t kDescStageStep = kStageBytes >> 4;
    static constexpr int kStagingOff = kStages * kStageBytes;
    static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(kStages <= kMaxStages, "barrier arrays");
    static_assert(kSfTmemBase + kStages * kSfCols <= kTmemCols, "scale slots must fit in TMEM");
    static_assert(!kNv || kN == 256, "NVFP4 runs 256-column tiles");
};

// Descriptor of a wide scale image: core matrices of 8 rows x 16 bytes, the two halves of a
// row 128 bytes apart (leading offset), 8-row groups 256 bytes apart (stride offset).
__device__ __forceinline__ uint64_t desc_sf_wide(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(256u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Byte of the wide image holding row r's word for half h: image row r (lane r of tensor
// memory), word position r / 32.
__device__ __forceinline__ uint32_t wide_off(int r, int h) {
    return (uint32_t)((r >> 3) * 256 + h * 128 + (r & 7) * 16 + (r >> 5) * 4);
}

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t sf_full[kMaxStages];
    uint64_t ready[kMaxStages];
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint64_t drain_cp;
    uint32_t tmem_base;
    int abort_flag;
};

template <int kN, bool kNv = false, bool kA8 = false>
constexpr size_t smem_bytes() {
    return (size_t)Cfg<kN, kNv, kA8>::kStagingOff + 8 * kStagingBytes + sizeof(Ctl) + 1024;
}

// Every configuration within the 227 KB of dynamic shared memory a CTA may have.
constexpr size_t kMaxDynSmem = 232448;
static_assert(smem_bytes<256>() <= kMaxDynSmem, "MXFP4 256-column tile");
static_assert(smem_bytes<128>() <= kMaxDynSmem, "MXFP4 128-column tile");
static_assert(smem_bytes<256, true>() <= kMaxDynSmem, "NVFP4 tile");
static_assert(smem_bytes<256, false, true>() <= kMaxDynSmem, "MXFP8-activation tile");

struct Tile {
    int32_t expert;
    int32_t rows;
    int64_t row0;
};

__device__ __forceinline__ int num_mtiles(const GemmArgs& a) {
    return a.num_mtiles_dev ? *a.num_mtiles_dev : a.num_mtiles_host;
}

__device__ __forceinline__ Tile get_tile(const GemmArgs& a, int mt) {
    Tile t;
    if (a.tile_expert != nullptr) {
        t.expert = a.tile_expert[mt];
        t.row0 = a.tile_row0[mt];
        t.rows = a.tile_rows[mt];
    } else {
        t.expert = 0;
        t.row0 = (int64_t)mt * kBM;
        const int64_t left = a.m_total - t.row0;
        t.rows = (int32_t)(left < kBM ? left : kBM);
    }
    return t;
}

// Row of the stacked B tensor behind row r of N tile nt (L1: the first kN / 2 tile rows
// are gate rows, the rest the matching up rows).
template <bool kL1, int kN>
__device__ __forceinline__ int64_t b_tile_row(const GemmArgs& a, int expert, int nt, int r) {
    if (kL1) {
        constexpr int kHalf = kN / 2;
        return (int64_t)expert * a.b_rows_per_expert + (r < kHalf ? 0 : a.n_half) + (int64_t)nt * kHalf +
               (r < kHalf ? r : r - kHalf);
    }
    return (int64_t)expert * a.b_rows_per_expert + (int64_t)nt * kN + r;
}

// Every lane polls; the warp proceeds only if all lanes saw the phase complete, so an
// abort never splits a warp between two code paths.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const StatusWords& status, uint32_t code) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, status, code)) != 0;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// A CTA's GEMM pipeline in shared and tensor memory. It is set up once per CTA; a persistent
// kernel runs several GEMMs through it, their barrier phases carried over.
struct GemmCtx {
    uint8_t* smem;        // 1024-byte aligned start of the stage ring
    uint32_t sbase;       // its shared-memory address
    Ctl* ctl;
    uint32_t tmem;        // base of the CTA's 512 tensor-memory columns
};

// A thread's position in the pipeline: the K stages (it) and accumulator tiles (tc) its role
// has passed, carried from one GEMM to the next.
struct PipePos {
    uint32_t it;
    uint32_t tc;
};

// Barrier initialisation and tensor-memory allocation; every thread of the CTA calls it.
template <int kN, bool kNv = false, bool kBTiled = true, bool kA8 = false>
__device__ __forceinline__ GemmCtx gemm_setup(uint8_t* smem_raw) {
    using C = Cfg<kN, kNv, kA8>;
    constexpr int kStages = C::kStages;
    GemmCtx g;
    const uint32_t raw_addr = smem_u32(smem_raw);
    g.smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    g.sbase = smem_u32(g.smem);
    g.ctl = reinterpret_cast<Ctl*>(g.smem + (size_t)C::kStagingOff + 8 * kStagingBytes);
    Ctl* ctl = g.ctl;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), kFullArrivals);
            mbar_init(smem_u32(&ctl->empty[s]), 1);  // MMA commit
            // + lane 0 of the loader once more with tile-layout B scales (their bulk copies'
            // byte count, or a plain arrival where they are gathered)
            mbar_init(smem_u32(&ctl->sf_full[s]), kSfArrivals + (kBTiled ? 1 : 0));
            mbar_init(smem_u32(&ctl->ready[s]), 1);   // scale copier commit
        }
        mbar_init(smem_u32(&ctl->tmem_full), 1);
        mbar_init(smem_u32(&ctl->tmem_empty), 8);    // one arrive per epilogue warp
        mbar_init(smem_u32(&ctl->drain), 1);
        mbar_init(smem_u32(&ctl->drain_cp), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    g.tmem = ctl->tmem_base;
    return g;
}

// One GEMM over its tile list (args), by every thread of the CTA in its role. Returns with the
// role's pipeline position advanced; the epilogue's output stores are complete.
template <bool kL1, bool kBTiled, int kN, bool kNv = false, bool kA8 = false>
__device__ __forceinline__ void gemm_run(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                                         const GemmArgs& args, const GemmCtx& g, PipePos& pos) {
    static_assert(!kNv || kBTiled, "NVFP4 weights come with tile-layout scales");
    static_assert(!kA8 || (kBTiled && kN == 256), "MXFP8 activations: tile-layout weight scales, 256-column tiles");
    using C = Cfg<kN, kNv, kA8>;
    constexpr int kXStage = kA8 ? C::kKStage : kBK / 2;    // TMA x step per stage (bytes of A, elements of B for kA8)
    constexpr int kBBytes = C::kBBytes;
    constexpr uint32_t kIdesc = C::kIdesc;
    constexpr int kStages = C::kStages;
    constexpr int kStageBytes = C::kStageBytes;
    constexpr int kSfaBytes = C::kSfaBytes;
    constexpr uint32_t kDescStageStep = C::kDescStageStep;
    constexpr int kStagingOff = C::kStagingOff;
    uint8_t* smem = g.smem;
    const uint32_t sbase = g.sbase;
    Ctl* ctl = g.ctl;
    const uint32_t tmem = g.tmem;
    volatile int* abort_flag = &ctl->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (*abort_flag) return;

    const int total = num_mtiles(args) * args.n_tiles;
    const int k_tiles = args.k_tiles;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            uint32_t& it = pos.it;
            for (int w = blockIdx.x; w < total; w += gridDim.x) {
                const Tile t = get_tile(args, w / args.n_tiles);
                const int nt = w % args.n_tiles;
                for (int kt = 0; kt < k_tiles; ++kt, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, args.status, kErrWaitEmpty))
                        goto producer_done;
                    const uint32_t st = sbase + s * kStageBytes;
                    const uint32_t bar = smem_u32(&ctl->full[s]);
                    mbar_arrive_expect_tx(bar, kABytes + C::kBTxBytes);
                    tma_load_2d(st, &tmA, kt * kXStage, (int32_t)t.row0, bar);
                    if (kL1) {
                        // w13 as [E][2][I][H/2]: kN / 2 gate rows then the matching up rows
                        tma_load_4d(st + kABytes, &tmB, kt * kXStage, nt * (kN / 2), 0, t.expert, bar);
                    } else {
                        tma_load_2d(st + kABytes, &tmB, kt * kXStage,
                                    (int32_t)b_tile_row<false, kN>(args, t.expert, nt, 0), bar);
                    }
                }
            }
        producer_done:;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread) ----------------
        if (lane == 0) {
            const uint64_t adesc0 = desc_sw128(sbase);
            const uint64_t bdesc0 = desc_sw128(sbase + kABytes);
            const uint32_t sf0 = tmem + kSfTmemBase;
            uint32_t& it = pos.it;
            uint32_t& tc = pos.tc;
            for (int w = blockIdx.x; w < total; w += gridDim.x) {
                if (!mbar_wait(smem_u32(&ctl->tmem_empty), (tc & 1u) ^ 1u, abort_flag, args.status,
                               kErrWaitTmemEmpty))
                    break;
                tc_fence_after();
                bool ok = true;
                for (int kt = 0; kt < k_tiles; ++kt, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&ctl->ready[s]), ph, abort_flag, args.status, kErrWaitFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = adesc0 + (uint64_t)(s * kDescStageStep);
                    const uint64_t bdesc = bdesc0 + (uint64_t)(s * kDescStageStep);
                    const uint32_t sfa = sf0 + s * C::kSfCols;
                    const uint32_t sfb = sfa + (kNv ? 16 : 8);
                    const uint32_t acc0 = kt != 0;
                    // 32 bytes of K per MMA, inside the 128-byte swizzle atom: 64 E2M1 elements, or
                    // with kA8 32 E4M3 elements of A and 32 spread E2M1 elements of B
                    if constexpr (kA8) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_mxf8(tmem, adesc + 2 * k, bdesc + 2 * k, idesc_with_sf_ids(kIdesc, k, k), sfa, sfb,
                                        k == 0 ? acc0 : 1u);
                        tc_commit(smem_u32(&ctl->empty[s]));
                        continue;
                    }
                    if constexpr (kNv) {
                        // one scale word per MMA: A's at +4k, B's at +8k; two MMAs at a K tail
                        const int nk = (args.k_tail_half && kt == k_tiles - 1) ? 2 : 4;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (k < nk)
                                tc_mma_nvf4(tmem, adesc + 2 * k, bdesc + 2 * k, kIdesc, sfa + 4 * k, sfb + 8 * k,
                                            k == 0 ? acc0 : 1u);
                        tc_commit(smem_u32(&ctl->empty[s]));
                        continue;
                    }
                    tc_mma_mxf4(tmem, adesc, bdesc, idesc_with_sf_ids(kIdesc, 0, 0), sfa, sfb, acc0);
                    tc_mma_mxf4(tmem, adesc + 2, bdesc + 2, idesc_with_sf_ids(kIdesc, 2, 2), sfa, sfb, 1);
                    if (!(args.k_tail_half && kt == k_tiles - 1)) {
                        tc_mma_mxf4(tmem, adesc + 4, bdesc + 4, idesc_with_sf_ids(kIdesc, 0, 0), sfa + 4, sfb + 8, 1);
                        tc_mma_mxf4(tmem, adesc + 6, bdesc + 6, idesc_with_sf_ids(kIdesc, 2, 2), sfa + 4, sfb + 8, 1);
                    }
                    tc_commit(smem_u32(&ctl->empty[s]));
                }
                if (!ok) break;
                tc_commit(smem_u32(&ctl->tmem_full));
                ++tc;
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------- scale-factor loader (A; and B when its scales are row-major) --------
        uint32_t& it = pos.it;
        bool aborted = false;
        for (int w = blockIdx.x; w < total && !aborted; w += gridDim.x) {
            const Tile t = get_tile(args, w / args.n_tiles);
            const int nt = w % args.n_tiles;
            for (int kt = 0; kt < k_tiles; ++kt, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, args.status, kErrWaitEmpty)) {
                    aborted = true;
                    break;
                }
                const bool half = args.k_tail_half && (kt == k_tiles - 1);
                const uint32_t st = sbase + s * kStageBytes;
                const int64_t kcol = (int64_t)kt * 4 * C::kWords;   // first scale byte of this stage
                if (kBTiled && (kN == 256 || !kL1) && lane == 0) {
                    // B scales: the stage's kWords K-words of each 128-row group (half of them at
                    // the K tail); each 128-row part of the tile is one whole group of the tile
                    // layout (L1's 128-column tiles are not: their gate and up halves are
                    // gathered below)
                    constexpr int kGroups = kN / 128;
                    const uint32_t sf_bytes = (uint32_t)((half ? C::kWordsHalf : C::kWords) * 512);
                    const uint32_t bar = smem_u32(&ctl->sf_full[s]);
                    int64_t grp[kGroups];
                    uint32_t tx = 0;
                    for (int h = 0; h < kGroups; ++h) {
                        grp[h] = b_tile_row<kL1, kN>(args, t.expert, nt, 128 * h) / 128;
                        if (grp[h] < args.b_groups) tx += sf_bytes;
                    }
                    mbar_arrive_expect_tx(bar, tx);
                    for (int h = 0; h < kGroups; ++h)
                        if (grp[h] < args.b_groups)
                            bulk_load(st + kABytes + kBBytes + kSfaBytes + h * (C::kWords * 512),
                                      args.sfb + (grp[h] * args.kw + C::kWords * kt) * 512, sf_bytes, bar);
                }
                if (kBTiled && kN == 128 && kL1) {
                    // B scales in tile layout for a 128-row tile of two 64-row pieces p (L1: gate
                    // and up) that need not share a 128-row group. A piece starts on a 64-row
                    // boundary, so in its group's block this lane's words of rows r0 + lane and
                    // r0 + 32 + lane are 8 contiguous bytes; they go to bytes 8 p .. 8 p + 7 of
                    // the lane's 16 (rows 64 p + lane, 64 p + 32 + lane of the tile), zero past
                    // the last row of B
                    const uint32_t sfb_s = st + kABytes + kBBytes + kSfaBytes;
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const int64_t r0 = b_tile_row<kL1, kN>(args, t.expert, nt, 64 * p);   // multiple of 64
                        const uint32_t n = (r0 + lane < args.b_rows ? 4u : 0u) +
                                           (r0 + 32 + lane < args.b_rows ? 4u : 0u);
                        const uint8_t* src = args.sfb + (n ? ((r0 >> 7) * args.kw + 2 * kt) * 512 + lane * 16 +
                                                                  ((r0 & 127) >> 5) * 4
                                                            : 0);
#pragma unroll
                        for (int wd = 0; wd < 2; ++wd) {
                            const uint32_t nb = (wd == 0 || !half) ? n : 0u;
                            cp_async_8(sfb_s + wd * 512 + lane * 16 + p * 8, nb ? src + 512 * wd : args.sfb, nb);
                        }
                    }
                    if (lane == 0) mbar_arrive(smem_u32(&ctl->sf_full[s]));   // the count's bulk share
                }
                // A's wide image: K-word wd of tile row r at wide_off(r, wd).
                if (!kA8 && args.a_sm) {
                    // Stage-major scales (routed MXFP4 and NVFP4 forwards): per K-word the tile's 128
                    // rows' words are 512 contiguous bytes. Instruction i takes rows (lane % 8) + 8 i +
                    // 32 (lane / 8): four 32-byte runs to read, and in the image every lane a
                    // different bank (row r's word sits in bank 4 (r % 8) + r / 32).
                    const uint32_t sfa_s = st + kABytes + kBBytes;
                    const int64_t mt = (int64_t)(w / args.n_tiles);
#pragma unroll
                    for (int wd = 0; wd < C::kWords; ++wd) {
                        const bool ok = wd < C::kWordsHalf || !half;
                        const uint8_t* src = args.sfa + ((mt * k_tiles + kt) * C::kWords + wd) * 512;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = (lane & 7) + 8 * i + 32 * (lane >> 3);
                            cp_async_4(sfa_s + 4096 * (wd >> 1) + wide_off(r, wd & 1), ok ? src + 4 * r : args.sfa,
                                       ok ? 4u : 0u);
                        }
                    }
                } else {
                    // Row-major scales: adjacent lanes take the kWords words of one row, which lie
                    // side by side, so one instruction touches 32 / kWords rows' cache lines
                    // rather than 32.
                    const uint32_t sfa_s = st + kABytes + kBBytes;
                    constexpr int kRowsPerInst = 32 / C::kWords;
                    const int wd = lane % C::kWords;
                    const bool word_ok = wd < C::kWordsHalf || !half;
#pragma unroll
                    for (int i = 0; i < 4 * C::kWords; ++i) {
                        const int r = kRowsPerInst * i + lane / C::kWords;
                        const int64_t grow = t.row0 + r;
                        const bool ok = grow < args.a_rows && word_ok;
                        const uint32_t dst = sfa_s + 4096 * (wd >> 1) + wide_off(r, wd & 1);
                        cp_async_4(dst, ok ? args.sfa + grow * args.ld_sf + kcol + 4 * wd : args.sfa, ok ? 4u : 0u);
                    }
                }
                // B's dense blocks (row-major B scales): 512 bytes per K-word, row r of a 128-row
                // group at byte (r % 32) * 16 + (r / 32) * 4. As for A, adjacent lanes take the
                // two K-words of one row.
                if (!kBTiled) {
                    const uint32_t sfb_s = st + kABytes + kBBytes + kSfaBytes;
                    const int wd = lane & 1;
                    const bool word_ok = wd == 0 || !half;
#pragma unroll
                    for (int i = 0; i < 8 * (kN / 128); ++i) {
                        const int r = 16 * i + (lane >> 1);              // row of the tile
                        const int h = r >> 7, rr = r & 127;
                        const int64_t brow = b_tile_row<kL1, kN>(args, t.expert, nt, r);
                        const bool ok = brow < args.b_rows && word_ok;
                        const uint32_t dst = sfb_s + h * 1024 + wd * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
                        cp_async_4(dst, ok ? args.sfb + brow * args.ld_sf + kcol + 4 * wd : args.sfb, ok ? 4u : 0u);
                    }
                }
                cp_async_arrive_noinc(smem_u32(&ctl->sf_full[s]));
            }
        }
        cp_async_wait<0>();
        __syncwarp();
    } else if (warp == 3) {
        // ---------------- scale-factor copier (one thread) ----------------
        if (lane == 0) {
            uint32_t& it = pos.it;
            bool ok = true;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
                for (int kt = 0; kt < k_tiles; ++kt, ++it) {
                    const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort_flag, args.status, kErrWaitFull) ||
                        !mbar_wait(smem_u32(&ctl->sf_full[s]), ph, abort_flag, args.status, kErrWaitFull)) {
                        ok = false;
                        break;
                    }
                    // the scale tiles were written by cp.async (generic proxy); tcgen05.cp
                    // reads them through the async proxy
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const int nwords = (args.k_tail_half && kt == k_tiles - 1) ? C::kWordsHalf : C::kWords;
                    const uint32_t sfa_s = sbase + s * kStageBytes + kABytes + kBBytes;
                    const uint32_t sfb_s = sfa_s + kSfaBytes;
                    const uint32_t sfa_t = tmem + kSfTmemBase + s * C::kSfCols;
                    const uint32_t sfb_t = sfa_t + (kNv ? 16 : 8);
#pragma unroll
                    for (int i = 0; i < C::kImages; ++i)                                      // A, two K-words each
                        tc_cp_128x256b(sfa_t + 8 * i, desc_sf_wide(sfa_s + 4096 * i));
                    for (int wd = 0; wd < nwords; ++wd) {
                        tc_cp_32x128b_x4(sfb_t + 8 * wd, desc_sf(sfb_s + wd * 512));          // B rows 0-127
                        if (kN == 256)                                                          // 128-255
                            tc_cp_32x128b_x4(sfb_t + 8 * wd + 4, desc_sf(sfb_s + C::kWords * 512 + wd * 512));
                    }
                    tc_commit(smem_u32(&ctl->ready[s]));   // arrives once the copies are in TMEM
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps 4..11 ----------------
        const int q = warp & 3;              // TMEM lane quarter this warp may access
        const int hf = (warp - 4) >> 2;      // which half of the columns
        const int row_in_tile = 32 * q + lane;
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
        uint8_t* staging = smem + kStagingOff + (warp - 4) * kStagingBytes;
        const uint32_t staging_s = smem_u32(staging);
        // NVFP4: the tile's global-scale products (L2: alpha_a; L1: gate alpha_a, up alpha_b)
        // and the re-quantisation global of L1's h with its 1 / (6 g)
        float alpha_a = 1.0f, alpha_b = 1.0f;
        const float q_g = kNv ? args.q_global : 0.0f;
        const float q_r = kNv && kL1 ? __frcp_rn(__fmul_rn(6.0f, q_g)) : 0.0f;
        // L2's output value of an accumulator word, with the scale of its 16-column block
        auto out_value = [&](uint32_t acc, float alpha) {
            return kNv ? __fmul_rn(__uint_as_float(acc), alpha) : __uint_as_float(acc);
        };
        // NVFP4 L2: the scale of the 16 output columns starting at col (its segment's, in a
        // fused projection)
        auto col_alpha = [&](int64_t col) {
            float a = alpha_a;
            if (kNv && !kL1 && args.nseg > 0) {
                a = args.seg_alpha[args.nseg - 1];
                for (int s = args.nseg - 2; s >= 0; --s)
                    if (col < args.seg_end[s]) a = args.seg_alpha[s];
            }
            return a;
        };
        // L1's h = bf16(silu(bf16(g)) * bf16(u)) for the 32 columns of one block, from the gate
        // and up accumulator words. Every BF16 rounding is done two values at a time by the
        // packed conversion (nearest even), which writes any NaN as a positive NaN: a NaN h is
        // re-quantised with sign 0, whatever produced it (a NaN g or u, silu(-inf), 0 * inf).
        auto h_block = [&](const uint32_t (&vg)[32], const uint32_t (&vu)[32], float (&h)[32]) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float g0 = __uint_as_float(vg[i]), g1 = __uint_as_float(vg[i + 1]);
                float u0 = __uint_as_float(vu[i]), u1 = __uint_as_float(vu[i + 1]);
                if (kNv) {
                    g0 = __fmul_rn(g0, alpha_a);
                    g1 = __fmul_rn(g1, alpha_a);
                    u0 = __fmul_rn(u0, alpha_b);
                    u1 = __fmul_rn(u1, alpha_b);
                }
                const uint32_t gp = bf16x2_rn(g0, g1), up = bf16x2_rn(u0, u1);
                const float s0 = silu_f32(__uint_as_float(gp << 16));
                const float s1 = silu_f32(__uint_as_float(gp & 0xFFFF0000u));
                const uint32_t hp = bf16x2_rn(s0 * __uint_as_float(up << 16), s1 * __uint_as_float(up & 0xFFFF0000u));
                h[i] = __uint_as_float(hp << 16);
                h[i + 1] = __uint_as_float(hp & 0xFFFF0000u);
            }
        };
        // Byte of h's MXFP4 scale for block b (32 columns) of global row grow, tile row r of M
        // tile mt: stage-major (hs_k_tiles > 0) or row-major
        auto hs_off = [&](int64_t grow, int r, int64_t mt, int64_t b) -> int64_t {
            if (args.hs_k_tiles <= 0) return grow * args.ld_hs + b;
            return kNv ? sm_scale_off<4>(mt, r, b, args.hs_k_tiles) : sm_scale_off<2>(mt, r, b, args.hs_k_tiles);
        };
        // Re-quantisation of 32 columns of h: 16 code bytes; the scale byte (MXFP4) or the two
        // E4M3 bytes of the two 16-column blocks, low byte first (NVFP4)
        auto requant32 = [&](const float (&h)[32], uint4& cd) -> uint32_t {
            if constexpr (kNv) {
                uint2 c0, c1;
                const uint32_t s0 = nv_quant16(h, q_g, q_r, c0);
                const uint32_t s1 = nv_quant16(h + 16, q_g, q_r, c1);
                cd = make_uint4(c0.x, c0.y, c1.x, c1.y);
                return s0 | (s1 << 8);
            } else {
                return mx_quant32(h, cd);
            }
        };
        uint32_t& tc = pos.tc;
        for (int w = blockIdx.x; w < total; w += gridDim.x, ++tc) {
            const Tile t = get_tile(args, w / args.n_tiles);
            const int nt = w % args.n_tiles;
            if (kNv) {
                alpha_a = alpha_b = args.alpha;
                if (args.w_global != nullptr) {
                    alpha_a = __fmul_rn(args.alpha, args.w_global[kL1 ? 2 * t.expert : t.expert]);
                    alpha_b = kL1 ? __fmul_rn(args.alpha, args.w_global[2 * t.expert + 1]) : alpha_a;
                }
            }
            if (!warp_wait(smem_u32(&ctl->tmem_full), tc & 1u, abort_flag, args.status, kErrWaitTmemFull)) break;
            tc_fence_after();
            // Warp (q, hf) owns rows 32 q..32 q + 31 and half hf of the tile's columns. L1: kHB
            // blocks of 32 columns of h, i.e. gate columns (kN / 4) hf + 32 b and the matching
            // up columns kN / 2 + (kN / 4) hf + 32 b; L2: kPieces pieces of 32 output columns.
            constexpr int kHB = kN / 128;
            constexpr int kPieces = kN / 64;
            uint32_t v[4][32];
            if (kL1) {
#pragma unroll
                for (int b = 0; b < kHB; ++b) {
                    tc_ld_32x32b_x32(taddr + (kN / 4) * hf + 32 * b, v[b]);               // gate
                    tc_ld_32x32b_x32(taddr + kN / 2 + (kN / 4) * hf + 32 * b, v[2 + b]);  // up
                }
            } else {
#pragma unroll
                for (int i = 0; i < kPieces; ++i) tc_ld_32x32b_x32(taddr + (kN / 2) * hf + 32 * i, v[i]);
            }
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tmem_empty));
            if (!kL1 && 32 * q + 32 <= t.rows) {
                // all 32 rows of this warp are in the tile: staged TMA stores
                const int32_t trow = (int32_t)(t.row0 + 32 * q);
#pragma unroll
                for (int i = 0; i < kPieces; ++i) {
                    const int64_t col = (int64_t)nt * kN + (kN / 2) * hf + 32 * i;
                    if (col >= args.n_valid) break;
                    const float al[2] = {col_alpha(col), col_alpha(col + 16)};
                    // the packed conversion writes a NaN as 0x7FFF; one test per piece finds it (a
                    // BF16 magnitude above 0x7F80 carries into bit 15 when 0x7F is added), and
                    // only such a piece is converted again with the NaN written as sign | 0x7FC0
                    uint32_t p[16];
                    uint32_t nan_bits = 0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        p[j] = bf16x2_rn(out_value(v[i][2 * j], al[j >> 3]), out_value(v[i][2 * j + 1], al[j >> 3]));
                        nan_bits |= ((p[j] & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u;
                    }
                    if (__builtin_expect(nan_bits != 0u, 0)) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            p[j] = pack_bf16x2(out_value(v[i][2 * j], al[j >> 3]),
                                               out_value(v[i][2 * j + 1], al[j >> 3]));
                    }
#pragma unroll
                    for (int c = 0; c < 2; ++c) {       // 16 columns (32 bytes) per row and store
                        if (col + 16 * c >= args.n_valid) break;
                        if (lane == 0) bulk_wait_read();   // the previous store has read the block
                        __syncwarp();
                        // the output map's 32-byte swizzle: row `lane`'s halves swap when bit 2
                        // of the row is set, which keeps the warp's 16-byte writes free of bank
                        // conflicts (4 wavefronts each instead of 8)
                        const int sw = (lane >> 2) & 1;
                        uint4* row = reinterpret_cast<uint4*>(staging + lane * 32);
                        row[sw] = make_uint4(p[8 * c + 0], p[8 * c + 1], p[8 * c + 2], p[8 * c + 3]);
                        row[sw ^ 1] = make_uint4(p[8 * c + 4], p[8 * c + 5], p[8 * c + 6], p[8 * c + 7]);
                        fence_proxy_async_smem();          // generic writes -> the TMA engine's reads
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmY, staging_s, (int32_t)(col + 16 * c), trow);
                            bulk_commit();
                        }
                    }
                }
                continue;
            }
            if (kA8 && kL1 && 32 * q + 32 <= t.rows) {
                // MXFP8 re-quant: 32 code bytes per 32 columns of h, one TMA store of 32 rows
                // x 32 bytes per block through the warp's staging block
                const int64_t grow = t.row0 + row_in_tile;
                const int64_t col0 = (int64_t)nt * (kN / 2) + (kN / 4) * hf;   // first column of h
                uint32_t es[kHB];
#pragma unroll
                for (int b = 0; b < kHB; ++b) {
                    float h[32];
                    h_block(v[b], v[2 + b], h);
                    uint4 c8[2];
                    es[b] = mx8_quant32(h, c8);
                    if (lane == 0) bulk_wait_read();   // the previous store has read the block
                    __syncwarp();
                    uint4* row = reinterpret_cast<uint4*>(staging + lane * 32);
                    row[0] = c8[0];
                    row[1] = c8[1];
                    fence_proxy_async_smem();          // generic writes -> the TMA engine's reads
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmY, staging_s, (int32_t)(col0 + 32 * b), (int32_t)(t.row0 + 32 * q));
                        bulk_commit();
                    }
                }
                if (kHB == 2)
                    *reinterpret_cast<uint16_t*>(args.hs + grow * args.ld_hs + col0 / 32) =
                        (uint16_t)(es[0] | (es[kHB - 1] << 8));
                else
                    args.hs[grow * args.ld_hs + col0 / 32] = (uint8_t)es[0];
                continue;
            }
            if (kL1 && 32 * q + 32 <= t.rows) {
                // all 32 rows of this warp are in the tile: codes through a staged TMA store
                // of 32 rows x 16 kHB bytes
                const int64_t grow = t.row0 + row_in_tile;
                const int64_t col0 = (int64_t)nt * (kN / 2) + (kN / 4) * hf;   // first column of h
                uint4 cds[kHB];
                uint32_t es[kHB];
#pragma unroll
                for (int b = 0; b < kHB; ++b) {
                    float h[32];
                    h_block(v[b], v[2 + b], h);
                    es[b] = requant32(h, cds[b]);
                }
                if (lane == 0) bulk_wait_read();   // the previous store has read the block
                __syncwarp();
                uint4* row = reinterpret_cast<uint4*>(staging + lane * 16 * kHB);
#pragma unroll
                for (int b = 0; b < kHB; ++b) row[b] = cds[b];
                fence_proxy_async_smem();          // generic writes -> the TMA engine's reads
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmY, staging_s, (int32_t)(col0 / 2), (int32_t)(t.row0 + 32 * q));
                    bulk_commit();
                }
                if (kNv)      // four E4M3 bytes, one word: 64 columns of h, 16 per byte
                    *reinterpret_cast<uint32_t*>(args.hs + hs_off(grow, row_in_tile, w / args.n_tiles, col0 / 16)) =
                        es[0] | (es[kHB - 1] << 16);
                else if (kHB == 2)   // two scale bytes of one stage-major word (col0 / 32 is even)
                    *reinterpret_cast<uint16_t*>(args.hs + hs_off(grow, row_in_tile, w / args.n_tiles, col0 / 32)) =
                        (uint16_t)(es[0] | (es[kHB - 1] << 8));
                else
                    args.hs[hs_off(grow, row_in_tile, w / args.n_tiles, col0 / 32)] = (uint8_t)es[0];
                continue;
            }
            if (row_in_tile >= t.rows) continue;
            const int64_t grow = t.row0 + row_in_tile;
            if (kL1) {
#pragma unroll
                for (int b = 0; b < kHB; ++b) {
                    float h[32];
                    h_block(v[b], v[2 + b], h);
                    const int64_t col = (int64_t)nt * (kN / 2) + (kN / 4) * hf + 32 * b;   // column of h
                    if constexpr (kA8) {
                        uint4 c8[2];
                        const uint32_t E = mx8_quant32(h, c8);
                        uint4* dst = reinterpret_cast<uint4*>(args.hq + grow * args.ld_hq + col);
                        dst[0] = c8[0];
                        dst[1] = c8[1];
                        args.hs[grow * args.ld_hs + col / 32] = (uint8_t)E;
                        continue;
                    }
                    uint4 codes;
                    const uint32_t E = requant32(h, codes);
                    *reinterpret_cast<uint4*>(args.hq + grow * args.ld_hq + col / 2) = codes;
                    if (kNv)   // two E4M3 bytes of one word (col / 16 is even)
                        *reinterpret_cast<uint16_t*>(args.hs + hs_off(grow, row_in_tile, w / args.n_tiles, col / 16)) =
                            (uint16_t)E;
                    else
                        args.hs[hs_off(grow, row_in_tile, w / args.n_tiles, col / 32)] = (uint8_t)E;
                }
            } else {
#pragma unroll
                for (int i = 0; i < kPieces; ++i) {
                    const int64_t col = (int64_t)nt * kN + (kN / 2) * hf + 32 * i;
                    const float al[2] = {col_alpha(col), col_alpha(col + 16)};
                    uint32_t p[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        p[j] = pack_bf16x2(out_value(v[i][2 * j], al[j >> 3]), out_value(v[i][2 * j + 1], al[j >> 3]));
                    uint16_t* dst = args.y + grow * args.ld_y + col;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        if (col + 16 * c < args.n_valid) {
                            uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * c);
                            d4[0] = make_uint4(p[8 * c + 0], p[8 * c + 1], p[8 * c + 2], p[8 * c + 3]);
                            d4[1] = make_uint4(p[8 * c + 4], p[8 * c + 5], p[8 * c + 6], p[8 * c + 7]);
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();   // staged stores complete: later readers see them
    }
}

// End of the CTA's GEMM work: the producer waits for the MMA commits that release the last
// stages (no asynchronous arrive may reach shared memory after the CTA exits); after an
// abort, copies in flight land and the tensor pipe drains before tensor memory is released.
template <int kN, bool kNv = false, bool kA8 = false>
__device__ __forceinline__ void gemm_finish(const GemmCtx& g, const PipePos& pos, const StatusWords& status) {
    constexpr int kStages = Cfg<kN, kNv, kA8>::kStages;
    Ctl* ctl = g.ctl;
    volatile int* abort_flag = &ctl->abort_flag;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (lane == 0 && warp <= 3) {
        if (warp == 0 && !*abort_flag) {
            const uint32_t it = pos.it;
            for (uint32_t i = it > (uint32_t)kStages ? it - kStages : 0; i < it; ++i)
                if (!mbar_wait(smem_u32(&ctl->empty[i % kStages]), (i / kStages) & 1u, abort_flag, status,
                               kErrWaitEmpty))
                    break;
        }
        if (*abort_flag) {
            if (warp == 0 || warp == 2) __nanosleep(20000);   // TMA and bulk copies in flight land
            if (warp == 1 || warp == 3) {
                // no MMA or scale copy may still write tensor memory when it is released
                const uint32_t bar = smem_u32(warp == 1 ? &ctl->drain : &ctl->drain_cp);
                tc_commit(bar);
                volatile int never = 0;
                mbar_wait(bar, 0, &never, status, kErrWaitDrain);
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(g.tmem, kTmemCols);
    }
}

// One GEMM per launch: the expert GEMMs of the multi-kernel forward and the dense GEMMs.
template <bool kL1, bool kBTiled, int kN, bool kNv = false, bool kA8 = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    mxf4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmY, const GemmArgs args) {
    extern __shared__ uint8_t smem_raw[];
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmY);
    }
    const GemmCtx g = gemm_setup<kN, kNv, kBTiled, kA8>(smem_raw);
    // Setup done: wait for the kernels before this one, then let the next one be scheduled
    // (all of this persistent grid's CTAs are resident already, so it cannot take their SMs).
    pdl_wait();
    pdl_launch_dependents();
    PipePos pos{0u, 0u};
    gemm_run<kL1, kBTiled, kN, kNv, kA8>(tmA, tmB, tmY, args, g, pos);
    gemm_finish<kN, kNv, kA8>(g, pos, args.status);
}

// The whole forward in one persistent cooperative launch ("Current Bug: vLLM produces
// empty/garbage output": the nvfp4-megamoe-kernel plan, "Phase 1: CuTeDSL Shared Expert
// Kernel": routing, L1 GEMM -> SiLU -> re-quant -> L2 GEMM, scatter), one CTA per SM. The
// phases are the multi-kernel forward's, with the same device code; where that forward
// starts a new kernel this one passes a grid-wide barrier:
//   routed: count chunks | scan (CTA 0) | quantise and gather x | L1 | L2 | combine
//   shared expert: quantise x | L1 | L2 (writes out)
// The GEMM pipeline is set up once; L2 continues L1's barrier phases (PipePos). Routing
// scratch lives in the stage ring, unused until L1.
template <int kN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_fused_kernel(const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1,
                     const __grid_constant__ CUtensorMap ty1, const __grid_constant__ CUtensorMap ta2,
                     const __grid_constant__ CUtensorMap tb2, const __grid_constant__ CUtensorMap ty2,
                     const FusedArgs fa) {
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x;
    if (tid == 0) {
        tma_prefetch_desc(&ta1);
        tma_prefetch_desc(&tb1);
        tma_prefetch_desc(&ty1);
        tma_prefetch_desc(&ta2);
        tma_prefetch_desc(&tb2);
        tma_prefetch_desc(&ty2);
        if (blockIdx.x == 0 && fa.clear_word != nullptr) *fa.clear_word = 0u;
    }
    const GemmCtx g = gemm_setup<kN, false, true>(smem_raw);
    volatile int* abort_flag = &g.ctl->abort_flag;
    uint32_t target = 0;
    auto barrier = [&]() {
        target += gridDim.x;
        grid_sync(fa.sync, target, abort_flag, fa.status);
    };
    int32_t* scratch = reinterpret_cast<int32_t*>(g.smem);
    const uint4* x8 = reinterpret_cast<const uint4*>(fa.x);
    const int64_t cta_thread = (int64_t)blockIdx.x * kGemmThreads + tid;
    const int64_t grid_threads = (int64_t)gridDim.x * kGemmThreads;
    const bool routed = fa.ids != nullptr;
    if (routed) {
        for (int64_t c = blockIdx.x; c < fa.rb.nchunks; c += gridDim.x)
            route_count_chunk(fa.ids, fa.T * fa.K, fa.E, c, fa.rb.chunk_counts, fa.rb.local_rank, scratch,
                              scratch + fa.E, tid);
        barrier();
        if (blockIdx.x == 0)
            route_scan(fa.rb.chunk_counts, fa.rb.nchunks, fa.E, fa.rb, scratch, scratch + fa.E,
                       scratch + 2 * fa.E + 1, tid, kGemmThreads);
        barrier();
        for (int64_t t = blockIdx.x; t < fa.T; t += gridDim.x)
            quant_gather_token<kQMx4>(x8, fa.ids, fa.K, fa.E, fa.H / 32, fa.rb, fa.xq, fa.xs, 0.0f, t, scratch, tid,
                                      kGemmThreads);
    } else {
        act_quant_blocks(x8, reinterpret_cast<uint4*>(fa.xq), fa.xs, fa.T * (fa.H / 32), cta_thread, grid_threads);
    }
    barrier();
    PipePos pos{0u, 0u};
    gemm_run<true, true, kN, false>(ta1, tb1, ty1, fa.g1, g, pos);
    barrier();
    gemm_run<false, true, kN, false>(ta2, tb2, ty2, fa.g2, g, pos);
    if (routed) {
        barrier();
        if (!*abort_flag)
            combine_groups<true>(reinterpret_cast<const uint4*>(fa.y), fa.rb.row_of, fa.topk_w,
                                 reinterpret_cast<uint4*>(fa.out), fa.T * (fa.H / 8), fa.H / 8, fa.K, cta_thread,
                                 grid_threads);
    }
    gemm_finish<kN, false>(g, pos, fa.status);
}

// The persistent forward's routing scratch (count, scan, and the quantise-gather's K row
// indices) lives in the stage ring, which it must fit for the largest expert count.
static_assert(route_count_smem(kMaxExperts) <= (size_t)Cfg<128>::kStagingOff &&
                  route_scan_smem(kMaxExperts) <= (size_t)Cfg<128>::kStagingOff &&
                  (size_t)kMaxTopK * 8 <= (size_t)Cfg<128>::kStagingOff,
              "routing scratch must fit in the stage ring");
static_assert(Cfg<128>::kStagingOff <= Cfg<256>::kStagingOff, "the 128-column ring is the smaller");

// Self-test of the grid barrier's failure path: every CTA waits for one arrival more than the
// grid has, runs out after the wait limit, records kErrWaitGrid and returns.
__global__ void __launch_bounds__(32) grid_sync_probe_kernel(uint32_t* counter, StatusWords status) {
    __shared__ int abort_flag;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncthreads();
    grid_sync(counter, gridDim.x + 1, &abort_flag, status);
}

template <bool kL1, bool kBTiled, int kN, bool kNv = false, bool kA8 = false>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a, int grid,
                   cudaStream_t s) {
    static int configured_mask = 0;   // one bit per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 31 && !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        err = cudaFuncSetAttribute(mxf4_gemm_kernel<kL1, kBTiled, kN, kNv, kA8>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<kN, kNv, kA8>());
        if (err != cudaSuccess) return err;
        __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    return launch_pdl(mxf4_gemm_kernel<kL1, kBTiled, kN, kNv, kA8>, dim3(grid), dim3(kGemmThreads),
                      smem_bytes<kN, kNv, kA8>(), s,
                      ta, tb, ty, a);
}

template <bool kL1>
cudaError_t launch_any(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                       int grid, bool b_tiled, int n_cols, cudaStream_t s) {
    if (n_cols == 128)
        return b_tiled ? launch<kL1, true, 128>(ta, tb, ty, a, grid, s) : launch<kL1, false, 128>(ta, tb, ty, a, grid, s);
    return b_tiled ? launch<kL1, true, 256>(ta, tb, ty, a, grid, s) : launch<kL1, false, 256>(ta, tb, ty, a, grid, s);
}

template <int kN>
cudaError_t launch_fused(const CUtensorMap& ta1, const CUtensorMap& tb1, const CUtensorMap& ty1,
                         const CUtensorMap& ta2, const CUtensorMap& tb2, const CUtensorMap& ty2, const FusedArgs& fa,
                         int num_sms, cudaStream_t s) {
    static int configured_mask = 0;   // one bit per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 31 && !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        err = cudaFuncSetAttribute(moe_fused_kernel<kN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem_bytes<kN>());
        if (err != cudaSuccess) return err;
        __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    // Cooperative: the runtime launches the grid only if every CTA can be resident at once,
    // which the grid-wide barriers need.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem_bytes<kN>();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_fused_kernel<kN>, ta1, tb1, ty1, ta2, tb2, ty2, fa);
}

}  // namespace

cudaError_t launch_moe_fused(const CUtensorMap& ta1, const CUtensorMap& tb1, const CUtensorMap& ty1,
                             const CUtensorMap& ta2, const CUtensorMap& tb2, const CUtensorMap& ty2,
                             const FusedArgs& fa, int n_cols, int num_sms, cudaStream_t s) {
    return n_cols == 128 ? launch_fused<128>(ta1, tb1, ty1, ta2, tb2, ty2, fa, num_sms, s)
                         : launch_fused<256>(ta1, tb1, ty1, ta2, tb2, ty2, fa, num_sms, s);
}

cudaError_t launch_grid_sync_probe(uint32_t* counter, StatusWords status, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grid_sync_probe_kernel, counter, status);
}

size_t gemm_smem_bytes() {
    const size_t a = smem_bytes<256>(), b = smem_bytes<128>(), c = smem_bytes<256, true>(),
                 d = smem_bytes<256, false, true>();
    const size_t ab = a > b ? a : b, cd = c > d ? c : d;
    return ab > cd ? ab : cd;
}

cudaError_t launch_gemm_l1(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                           int grid, bool b_tiled, int n_cols, cudaStream_t s) {
    return launch_any<true>(ta, tb, ty, a, grid, b_tiled, n_cols, s);
}

cudaError_t launch_gemm_l2(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                           int grid, bool b_tiled, int n_cols, cudaStream_t s) {
    return launch_any<false>(ta, tb, ty, a, grid, b_tiled, n_cols, s);
}

cudaError_t launch_gemm_nvfp4(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                              int grid, cudaStream_t s) {
    return launch<false, true, 256, true>(ta, tb, ty, a, grid, s);
}

cudaError_t launch_gemm_nvfp4_l1(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty,
                                 const GemmArgs& a, int grid, cudaStream_t s) {
    return launch<true, true, 256, true>(ta, tb, ty, a, grid, s);
}

cudaError_t launch_gemm_a8(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty, const GemmArgs& a,
                           int grid, bool l1, cudaStream_t s) {
    return l1 ? launch<true, true, 256, false, true>(ta, tb, ty, a, grid, s)
              : launch<false, true, 256, false, true>(ta, tb, ty, a, grid, s);
}

}  // namespace mx
