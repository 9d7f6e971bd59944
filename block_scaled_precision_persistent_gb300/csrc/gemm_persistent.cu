// Persistent, warp-specialised block-scaled GEMM on the 5th-generation tensor
// cores of sm_103a:
//
//     D[M][N] = bf16( alpha * sum_k (A[m][k] * sA) (B[n][k] * sB) )
//
// Design ("Together AI Ports ThunderKittens GEMM Kernels to NVIDIA Vera Rubin
// NVL72", introduction): a loader warp streams A and B tiles into a ring of
// shared-memory stages with TMA, one MMA thread drives tcgen05.mma with the
// accumulator in tensor memory, and an epilogue warpgroup drains finished
// accumulators to HBM; the kernel is persistent, so the next tile's loads
// stream in while the previous tile's outputs drain. For NVFP4 the block
// scales are written from shared memory into tensor memory (tcgen05.st) next
// to the accumulators ("Building the GEMM": the scale factors need TMEM
// columns beside the accumulators, which bounds the tile shape within the
// 512 columns of this GPU).
//
// CTA roles (320 threads, one CTA per SM):
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator + MMA issuer (one elected lane)
//   warps 2..5  NVFP4 scale writers smem -> TMEM (one per TMEM sub-partition)
//   warps 6..9  epilogue: TMEM -> registers -> *alpha -> BF16 -> swizzled
//               smem -> TMA store; warp w reads TMEM lanes 32*(w%4)..+31
//
// Every mbarrier wait is bounded (see ptx.cuh): a wait that runs out records
// BSG_ERR_DEVICE_TIMEOUT in the status word and the CTA drains and exits.
#include <cuda_bf16.h>

#include "bsg_internal.h"
#include "gemm_common.cuh"
#include "group.cuh"
#include "ptx.cuh"

namespace bsg {

template <Kind KIND, int BN, int STAGES, int NUM_ACC>
struct Tile {
    static constexpr bool kFp4 = KIND == Kind::NVFP4;
    // NVFP4 activations x dense BF16 weights: A arrives as E2M1 codes plus
    // block scales and is expanded to BF16 in shared memory by the four
    // warps that write NVFP4 scales in the other kind (kind::f16 MMA)
    static constexpr bool kDense = KIND == Kind::NVFP4_BF16 || KIND == Kind::NVFP4_BF16_TMEM;
    // dense variant: the expanded A staged in tensor memory (32 columns per
    // stage: 64 BF16 per row), the MMA reading A from there, which frees the
    // 16 KB of shared memory per stage for more ring stages
    static constexpr bool kTmemA = KIND == Kind::NVFP4_BF16_TMEM;
    static constexpr int BM = 128;
    static constexpr int ROW_BYTES = 128;                 // K bytes of one row per stage
    static constexpr int K_BLOCK = kFp4 ? 256 : kDense ? 64 : 128;   // K elements per stage
    static constexpr int MMA_K_BYTES = 32;                // K bytes per tcgen05.mma
    static constexpr int MMAS = ROW_BYTES / MMA_K_BYTES;  // MMAs per stage
    static constexpr int A_BYTES = kTmemA ? 0 : BM * ROW_BYTES;
    static constexpr int A_COLS = kTmemA ? ROW_BYTES / 4 : 0;          // TMEM columns of one stage's A
    static constexpr int B_BYTES = BN * ROW_BYTES;
    // NVFP4 scales of one stage: 128 rows x 16 scales = four 512-byte blocks
    static constexpr int SF_BLOCK_BYTES = 2048;
    static constexpr int SFB_CHUNKS = kFp4 ? BN / 128 : 0;
    static constexpr int SFA_BYTES = kFp4 ? SF_BLOCK_BYTES : 0;
    static constexpr int SFB_BYTES = SFB_CHUNKS * SF_BLOCK_BYTES;
    // dense: A's packed codes (128 rows x 32 bytes, TMA) and their scales
    // (one 512-byte block of the swizzled layout: 128 rows x 4 scales)
    static constexpr int APK_BYTES = kDense ? BM * 32 : 0;
    static constexpr int ASF_BYTES = kDense ? 512 : 0;
    static constexpr int STAGE_BYTES =
        (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES + APK_BYTES + ASF_BYTES + 1023) / 1024 * 1024;
    static constexpr int EPI_WARPS = 4;
    static constexpr int EPI_COLS = 64;                   // BF16 columns per store box
    static constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 2;
    static constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;
    // mbarrier layout (8 bytes each): full, empty per stage; full, empty per
    // accumulator; the drain barrier; scale-ready, scale-full per stage
    static constexpr int BAR_FULL = 0;
    static constexpr int BAR_EMPTY = BAR_FULL + STAGES;
    static constexpr int BAR_TFULL = BAR_EMPTY + STAGES;
    static constexpr int BAR_TEMPTY = BAR_TFULL + NUM_ACC;
    static constexpr int BAR_DRAIN = BAR_TEMPTY + NUM_ACC;
    static constexpr int BAR_SFREADY = BAR_DRAIN + 1;
    static constexpr int BAR_SFFULL = BAR_SFREADY + STAGES;
    static constexpr int NUM_BARS = BAR_SFFULL + STAGES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16;
    // NVFP4: one scale writer per TMEM sub-partition; dense: two expansion
    // warps per sub-partition, each taking half of every row
    static constexpr int SCALE_WARPS = kDense ? 8 : 4;
    static constexpr int EPI_WARP0 = 2 + SCALE_WARPS;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);   // producer, MMA, scale warps, epilogue
    // TMEM columns: NUM_ACC accumulators of BN columns, then one set of scale
    // columns per ring stage (a stage's scales are overwritten only after the
    // MMAs that read them completed, which the ring's empty barrier proves).
    static constexpr int SFA_COLS = kFp4 ? 4 * MMAS : 0;
    static constexpr int SFB_COLS = kFp4 ? 4 * SFB_CHUNKS * MMAS : 0;
    static constexpr int SF_COLS = SFA_COLS + SFB_COLS;
    static constexpr int TMEM_USED = NUM_ACC * BN + STAGES * (SF_COLS + A_COLS);
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static constexpr uint32_t IDESC = kFp4 ? idesc_nvfp4(BM, BN) : kDense ? idesc_bf16(BM, BN) : idesc_fp8(BM, BN);
    static constexpr uint32_t IDESC_F16 = idesc_f16(BM, BN);   // dense kind with FP16 B

    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "tile N");
    static_assert(!kFp4 || BN % 128 == 0, "NVFP4 scale blocks cover 128 rows");
    static_assert(TMEM_USED <= 512, "TMEM: accumulators plus scales exceed 512 columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-byte aligned (128B swizzle)");
};

// MODE: kModePlain, kModeEpi (bias, gamma, scattered rows) or kModeGrouped
// (the grouped GEMM over ragged row slices, NVFP4 only, with the variants'
// epilogue).
template <Kind KIND, int BN, int STAGES, int NUM_ACC, int MODE>
__global__ void __launch_bounds__(Tile<KIND, BN, STAGES, NUM_ACC>::THREADS, 1)
    gemm_persistent_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmD, const GemmArgs args)
{
    using T = Tile<KIND, BN, STAGES, NUM_ACC>;
    constexpr bool EPI = MODE != kModePlain;
    constexpr bool GROUPED = MODE == kModeGrouped;
    constexpr bool KGROUPED = MODE == kModeKGrouped;
    static_assert(!GROUPED || ((T::kFp4 || T::kTmemA) && T::SMEM_BYTES + kGroupTableBytes <= 232448),
                  "grouped GEMM: NVFP4 or TMEM-staged dense plans whose shared memory has room for the slice table");
    static_assert(!KGROUPED || (T::kTmemA && T::SMEM_BYTES + kGroupTableBytes <= 232448),
                  "K-ragged GEMM: TMEM-staged dense plans whose shared memory has room for the slice table");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t s_epi = base + STAGES * T::STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + STAGES * T::STAGE_BYTES + T::EPI_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t full0 = bar0 + 8u * T::BAR_FULL;           // [STAGES] TMA -> MMA
    const uint32_t empty0 = bar0 + 8u * T::BAR_EMPTY;         // [STAGES] MMA -> TMA
    const uint32_t tfull0 = bar0 + 8u * T::BAR_TFULL;         // [NUM_ACC] MMA -> epilogue
    const uint32_t tempty0 = bar0 + 8u * T::BAR_TEMPTY;       // [NUM_ACC] epilogue -> MMA
    const uint32_t drain_bar = bar0 + 8u * T::BAR_DRAIN;      // MMA teardown
    const uint32_t sfready0 = bar0 + 8u * T::BAR_SFREADY;     // [STAGES] scales in TMEM -> MMA
    const uint32_t sffull0 = bar0 + 8u * T::BAR_SFFULL;       // [STAGES] scale loads -> scale warps
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + T::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // grouped: slice boundaries and first 128-row tile of each slice (group.cuh)
    int *const s_go = reinterpret_cast<int *>(tmem_slot + 4);
    int *const s_gb = s_go + (kMaxGroups + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Watchdog wd{args.status, args.timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            mbar_init(tempty0 + 8u * a, T::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(sfready0 + 8u * s, T::SCALE_WARPS);
            mbar_init(sffull0 + 8u * s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmD);
        if constexpr (!GROUPED && !KGROUPED) {
            // B not written by the previous kernel: warm L2 with the first
            // tile's B while that kernel finishes
            if (args.pdl == 2 && (int)blockIdx.x < args.num_m_tiles * args.num_n_tiles) {
                int mt, nt;
                raster_tile((int)blockIdx.x, args, mt, nt);
                const int nkb = min(args.num_k_blocks, kEarlyKBlocks);
                for (int kb = 0; kb < nkb; ++kb)
                    tma_prefetch_2d(&tmB, kb * T::ROW_BYTES, nt * BN);
            }
        }
    }
    __syncwarp();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
        tmem_relinquish();
    }
    if constexpr (GROUPED || KGROUPED) {
        if (warp == 2) {
            griddep_wait();      // the offsets may come from the previous grid
            // slice boundaries over M (routed rows) or over K (K-ragged)
            build_group_table(args.group_offs, args.num_groups, KGROUPED ? args.K : args.M, s_go, s_gb, lane);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    griddep_wait();              // a dependent launch: the previous grid's writes are visible
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    // grouped: one 128-row tile row per 128 rows of each slice
    const int num_m_tiles = GROUPED ? s_gb[args.num_groups] : args.num_m_tiles;
    // K-ragged: every slice of K is a whole M x N problem of its own
    const int tiles_per_slice = num_m_tiles * args.num_n_tiles;
    const int num_tiles = KGROUPED ? args.num_groups * tiles_per_slice : tiles_per_slice;
    const int nkb = args.num_k_blocks;
    const bool b_f16 = args.b_f16 != 0;   // dense kind: B (and the expanded A) are FP16, not BF16
    // m tile -> its slice, first row of A, end of the slice's rows
    auto tile_rows = [&](int mt, int &g, int &row0, int &row_end) {
        if constexpr (GROUPED) {
            g = group_of_block(s_gb, args.num_groups, mt);
            row0 = s_go[g] + (mt - s_gb[g]) * T::BM;
            row_end = s_go[g + 1];
        } else {
            g = 0;
            row0 = mt * T::BM;
            row_end = args.M;
        }
    };
    // tile -> its m / n tile, slice, rows, and k-blocks [kb0, kb1): all of K,
    // or (K-ragged) the slice's k-blocks, with g the K slice
    auto tile_pos = [&](int tile, int &mt, int &nt, int &g, int &row0, int &row_end, int &kb0, int &kb1) {
        int ks = 0;
        if constexpr (KGROUPED) {
            ks = tile / tiles_per_slice;
            tile -= ks * tiles_per_slice;
        }
        raster_tile(tile, args.raster_group, num_m_tiles, args.num_n_tiles, mt, nt);
        tile_rows(mt, g, row0, row_end);
        kb0 = 0;
        kb1 = nkb;
        if constexpr (KGROUPED) {
            g = ks;
            kb0 = s_go[ks] / T::K_BLOCK;
            kb1 = s_go[ks + 1] / T::K_BLOCK;
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, armed_mask = 0, armed_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int mt, nt, g, row0, row_end, kb0, kb1;
                tile_pos(tile, mt, nt, g, row0, row_end, kb0, kb1);
                const uint8_t *const sfb_g = args.sfb + (size_t)(GROUPED ? g : 0) * args.sfb_group_bytes;
                const int b_row0 = (GROUPED ? g * args.N : 0) + nt * BN;   // a routed slice's own weights
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, wd, abort_flag, 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * T::STAGE_BYTES;
                    const uint32_t sb = sa + T::A_BYTES;
                    const uint32_t fb = full0 + 8u * stage;
                    if constexpr (T::kFp4) {
                        // scales first, on their own barrier: the scale warps can
                        // copy them into TMEM while A and B are still in flight.
                        // The stage's 16 scale columns are 4 consecutive
                        // 512-byte blocks of the swizzled layout.
                        const int nchunks = min(T::SFB_CHUNKS, args.sfb_row_blocks - nt * T::SFB_CHUNKS);
                        const uint32_t sfb = sffull0 + 8u * stage;
                        mbar_arrive_expect_tx(sfb, T::SF_BLOCK_BYTES * (1 + nchunks));
                        const uint32_t ssfa = sb + T::B_BYTES;
                        const size_t cb = (size_t)kb * 4u;
                        bulk_load(ssfa, args.sfa + ((size_t)mt * args.sf_col_blocks + cb) * 512u,
                                  T::SF_BLOCK_BYTES, sfb);
                        for (int c = 0; c < nchunks; ++c) {
                            const size_t rb = (size_t)nt * T::SFB_CHUNKS + (size_t)c;
                            bulk_load(ssfa + T::SFA_BYTES + c * T::SF_BLOCK_BYTES,
                                      sfb_g + (rb * args.sf_col_blocks + cb) * 512u,
                                      T::SF_BLOCK_BYTES, sfb);
                        }
                    }
                    if constexpr (T::kDense) {
                        // A's codes and scales on the expansion barrier, B on the full one
                        const uint32_t sfb = sffull0 + 8u * stage;
                        const uint32_t sapk = sb + T::B_BYTES;
                        mbar_arrive_expect_tx(sfb, T::APK_BYTES + T::ASF_BYTES);
                        tma_load_2d(sapk, &tmA, sfb, kb * 32, row0);
                        bulk_load(sapk + T::APK_BYTES, args.sfa + ((size_t)mt * args.sf_col_blocks + kb) * 512u,
                                  T::ASF_BYTES, sfb);
                        mbar_arrive_expect_tx(fb, T::B_BYTES);
                        tma_load_2d(sb, &tmB, fb, kb * T::ROW_BYTES, b_row0);
                    } else {
                        mbar_arrive_expect_tx(fb, T::A_BYTES + T::B_BYTES);
                        tma_load_2d(sa, &tmA, fb, kb * T::ROW_BYTES, row0);
                        tma_load_2d(sb, &tmB, fb, kb * T::ROW_BYTES, b_row0);
                    }
                    armed_mask |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let copies already issued land before the CTA goes away
                for (int s = 0; s < STAGES; ++s)
                    if ((armed_mask >> s) & 1u) {
                        mbar_wait_quiet(full0 + 8u * s, (armed_parity >> s) & 1u, wd.limit_ns);
                        if constexpr (T::kFp4 || T::kDense)
                            mbar_wait_quiet(sffull0 + 8u * s, (armed_parity >> s) & 1u, wd.limit_ns);
                    }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t idesc = b_f16 ? T::IDESC_F16 : T::IDESC;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(tempty0 + 8u * acc, acc_phase ^ 1u, wd, abort_flag, 2)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                int kb0 = 0, kb1 = nkb;
                if constexpr (KGROUPED) {
                    int mt, nt, g, row0, row_end;
                    tile_pos(tile, mt, nt, g, row0, row_end, kb0, kb1);
                }
                // (a K-ragged slice with no k-blocks issues no MMA: its
                // epilogue reads the accumulator as zero)
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full0 + 8u * stage, phase, wd, abort_flag, 3)) {
                        ok = false;
                        break;
                    }
                    if constexpr (T::kFp4 || T::kDense) {
                        // the scale warps have written this stage's scales to
                        // TMEM (NVFP4) / its expanded A to shared memory (dense)
                        if (!mbar_wait(sfready0 + 8u * stage, phase, wd, abort_flag, 5)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = base + stage * T::STAGE_BYTES;
                    const uint32_t sb = sa + T::A_BYTES;
                    if constexpr (T::kFp4) {
                        const uint32_t sfa_t = tmem + (uint32_t)(NUM_ACC * BN + stage * T::SF_COLS);
                        const uint32_t sfb_t = sfa_t + T::SFA_COLS;
#pragma unroll
                        for (int j = 0; j < T::MMAS; ++j)
                            mma_nvfp4(d_tmem, desc_kmajor_sw128(sa + T::MMA_K_BYTES * j),
                                      desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                      sfa_t + 4u * j, sfb_t + 4u * j * T::SFB_CHUNKS,
                                      (kb != kb0 || j != 0) ? 1u : 0u);
                    } else if constexpr (T::kTmemA) {
                        const uint32_t a_t = tmem + (uint32_t)(NUM_ACC * BN + stage * T::A_COLS);
#pragma unroll
                        for (int j = 0; j < T::MMAS; ++j)
                            mma_bf16_tmem_a(d_tmem, a_t + (uint32_t)(j * T::MMA_K_BYTES / 4),
                                            desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                            (kb != kb0 || j != 0) ? 1u : 0u);
                    } else if constexpr (T::kDense) {
#pragma unroll
                        for (int j = 0; j < T::MMAS; ++j)
                            mma_bf16(d_tmem, desc_kmajor_sw128(sa + T::MMA_K_BYTES * j),
                                     desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                     (kb != kb0 || j != 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int j = 0; j < T::MMAS; ++j)
                            mma_fp8(d_tmem, desc_kmajor_sw128(sa + T::MMA_K_BYTES * j),
                                    desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                    (kb != kb0 || j != 0) ? 1u : 0u);
                    }
                    tc_commit(empty0 + 8u * stage);   // frees the stage once these MMAs finish
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc_commit(tfull0 + 8u * acc);         // accumulator ready for the epilogue
                if (++acc == NUM_ACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA and copy issued above completes before TMEM is freed
            // (a grouped GEMM's grid is sized for a bound on its tiles: a CTA
            // past the actual ones issued nothing and has nothing to drain)
            if ((int)blockIdx.x < num_tiles) {
                tc_commit(drain_bar);
                mbar_wait_quiet(drain_bar, 0, wd.limit_ns);
            }
        }
    } else if (warp < T::EPI_WARP0) {
        // ------------------------------------------------------------------
        // Scale warps (NVFP4) : one per TMEM sub-partition
        // (warp % 4), each writing the stage's block scales from shared
        // memory into its own 32 TMEM lanes with tcgen05.st -- two store
        // instructions per warp per stage, in parallel across the four
        // sub-partitions -- then signalling the MMA thread.
        // ------------------------------------------------------------------
        if constexpr (T::kFp4) {
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                for (int kb = 0; kb < nkb; ++kb) {
                    // a stage's scale columns are rewritten only after its
                    // scales were reloaded, i.e. after the MMAs that read the
                    // previous contents completed (empty -> producer -> sf full)
                    if (!warp_wait(sffull0 + 8u * stage, phase, wd, abort_flag, 6, lane)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sfa_t = tmem + lane_off + (uint32_t)(NUM_ACC * BN + stage * T::SF_COLS);
                    const uint32_t ssfa = base + stage * T::STAGE_BYTES + T::A_BYTES + T::B_BYTES;
                    store_stage_scales<T::SFB_CHUNKS>(sfa_t, sfa_t + T::SFA_COLS, ssfa, ssfa + T::SFA_BYTES,
                                                      lane);
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(sfready0 + 8u * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else if constexpr (T::kDense) {
            // ----------------------------------------------------------------
            // Expansion warps (NVFP4 x BF16), two per TMEM sub-partition: row
            // r = 32 (warp % 4) + lane of the stage's A, column half hc, from
            // E2M1 codes and block scales to BF16 -- into TMEM (one
            // tcgen05.st of 16 columns) or the 128B-swizzled shared tile the
            // MMA reads (then a proxy fence) -- then the stage's ready barrier
            // ----------------------------------------------------------------
            const int r = (warp & 3) * 32 + lane;
            const int hc = (warp - 2) >> 2;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int kb0 = 0, kb1 = nkb;
                if constexpr (KGROUPED) {
                    int mt, nt, g, row0, row_end;
                    tile_pos(tile, mt, nt, g, row0, row_end, kb0, kb1);
                }
                for (int kb = kb0; kb < kb1; ++kb) {
                    // the stage's codes were reloaded after the MMAs that read
                    // its previous expansion completed (empty -> producer)
                    if (!warp_wait(sffull0 + 8u * stage, phase, wd, abort_flag, 6, lane)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint8_t *apk = gbase + stage * T::STAGE_BYTES + T::A_BYTES + T::B_BYTES;
                    const uint32_t sc = *reinterpret_cast<const uint32_t *>(apk + T::APK_BYTES + (r & 31) * 16 +
                                                                             (r >> 5) * 4);
                    uint32_t w[16];
                    if (b_f16)
                        expand_half_row_nvfp4<true>(apk + r * 32, sc, hc, w);
                    else
                        expand_half_row_nvfp4<false>(apk + r * 32, sc, hc, w);
                    if constexpr (T::kTmemA) {
                        // lane r of this warp's sub-partition, 16 of the stage's 32 A columns
                        tmem_st_32x32b_x16(tmem + ((uint32_t)((warp & 3) * 32) << 16) +
                                               (uint32_t)(NUM_ACC * BN + stage * T::A_COLS + 16 * hc),
                                           w);
                        tmem_st_wait();
                        tc_fence_before_sync();
                    } else {
                        store_half_row_sw128(w, base + stage * T::STAGE_BYTES, r, hc);
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(sfready0 + 8u * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------------
        // Epilogue warpgroup
        // ------------------------------------------------------------------
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t ebuf = s_epi + (uint32_t)(warp - T::EPI_WARP0) * 2u * T::EPI_BUF_BYTES;
        float scale = args.alpha;
        if constexpr (!T::kFp4) {
            if (args.sA)
                scale *= *args.sA;
            if (args.sB)
                scale *= *args.sB;
        }
        int acc = 0, buf = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mt, nt, g, row0, row_end, kb0, kb1;
            tile_pos(tile, mt, nt, g, row0, row_end, kb0, kb1);
            const float *const bias = args.bias ? args.bias + (size_t)g * args.N : nullptr;
            const int y = row0 + q * 32;              // first row of this warp's 32
            // rows of the warp that TMA could store past the slice's end (or,
            // K-ragged, into the next slice's rows of D): the warp stores its
            // rows one by one instead (as scattered rows)
            const bool per_row = EPI && (args.scatter || ((GROUPED || KGROUPED) && y + 32 > row_end));
            // K-ragged: slice g's output is rows [g*M, g*M + M) of D
            const int y_out = KGROUPED ? g * args.M + y : y;
            const bool zero_acc = KGROUPED && kb1 <= kb0;   // an empty slice: nothing was summed
            RowEpi re{1.0f, -1};
            if constexpr (EPI) {
                re = load_row_epi(args, y + lane, row_end);
                if (KGROUPED && re.dst >= 0)
                    re.dst += g * args.M;
                prefetch_bias(bias, args.N, nt * BN, BN, lane);
            }
            if (!warp_wait(tfull0 + 8u * acc, acc_phase, wd, abort_flag, 4, lane))
                break;
            tc_fence_after_sync();
            const uint32_t t_acc = tmem + lane_off + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int ch = 0; ch < BN / T::EPI_COLS; ++ch) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(t_acc + ch * T::EPI_COLS, v0);
                tmem_ld_32x32b_x32(t_acc + ch * T::EPI_COLS + 32, v1);
                const int x = nt * BN + ch * T::EPI_COLS;
                tmem_ld_wait();
                if (zero_acc) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v0[i] = v1[i] = 0u;
                }
                if (ch == BN / T::EPI_COLS - 1) {
                    // the whole accumulator is in registers: hand it back
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(tempty0 + 8u * acc);
                }
                // the store that last read this staging buffer must be done
                if (lane == 0)
                    bulk_wait_group_read<1>();
                __syncwarp();
                const uint32_t sbuf = ebuf + (uint32_t)buf * T::EPI_BUF_BYTES;
                const uint32_t row = sbuf + (uint32_t)lane * 128u;
                // 128-byte swizzle: 16-byte chunk c of row r lands at chunk c ^ (r % 8)
                if constexpr (EPI) {
                    uint32_t pk[32];
                    convert64_epi(v0, v1, pk, scale, re, args, bias, x);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(row + ((uint32_t)(c ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1],
                                     pk[4 * c + 2], pk[4 * c + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_shared_v4(row + ((uint32_t)(c ^ (lane & 7)) << 4),
                                     pack_bf16x2(__uint_as_float(v0[8 * c + 0]) * scale, __uint_as_float(v0[8 * c + 1]) * scale),
                                     pack_bf16x2(__uint_as_float(v0[8 * c + 2]) * scale, __uint_as_float(v0[8 * c + 3]) * scale),
                                     pack_bf16x2(__uint_as_float(v0[8 * c + 4]) * scale, __uint_as_float(v0[8 * c + 5]) * scale),
                                     pack_bf16x2(__uint_as_float(v0[8 * c + 6]) * scale, __uint_as_float(v0[8 * c + 7]) * scale));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_shared_v4(row + ((uint32_t)((c + 4) ^ (lane & 7)) << 4),
                                     pack_bf16x2(__uint_as_float(v1[8 * c + 0]) * scale, __uint_as_float(v1[8 * c + 1]) * scale),
                                     pack_bf16x2(__uint_as_float(v1[8 * c + 2]) * scale, __uint_as_float(v1[8 * c + 3]) * scale),
                                     pack_bf16x2(__uint_as_float(v1[8 * c + 4]) * scale, __uint_as_float(v1[8 * c + 5]) * scale),
                                     pack_bf16x2(__uint_as_float(v1[8 * c + 6]) * scale, __uint_as_float(v1[8 * c + 7]) * scale));
                }
                if (per_row) {
                    __syncwarp();
                    scatter_chunk(gbase + (sbuf - base), re.dst, args.d, args.N, x, lane);
                } else {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (x < args.N && y < args.M)
                            tma_store_2d(&tmD, sbuf, x, y_out);
                        bulk_commit_group();
                    }
                }
                buf ^= 1;
            }
            if (++acc == NUM_ACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0)
            bulk_wait_group<0>();
        __syncwarp();
    }

    // Reconverge each warp before the block barrier: the producer and MMA
    // roles ran on lane 0 only, and the teardown below (tcgen05.dealloc) is a
    // warp-collective instruction that needs all 32 lanes together.
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Plans: the compiled configurations and their host launchers
// ---------------------------------------------------------------------------
template <Kind KIND, int BN, int STAGES, int NUM_ACC, int MODE>
static cudaError_t launch_mode(const GemmMaps &maps, const GemmArgs &args, int grid, cudaStream_t stream)
{
    using T = Tile<KIND, BN, STAGES, NUM_ACC>;
    constexpr int smem = T::SMEM_BYTES + ((MODE == kModeGrouped || MODE == kModeKGrouped) ? kGroupTableBytes : 0);
    auto kern = gemm_persistent_kernel<KIND, BN, STAGES, NUM_ACC, MODE>;
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(T::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = args.pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, maps.a, maps.b, maps.d, args);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <Kind KIND, int BN, int STAGES, int NUM_ACC>
static cudaError_t launch_impl(const GemmMaps &maps, const GemmArgs &args, int grid,
                               cudaStream_t stream)
{
    if (args.group_offs && args.k_grouped) {
        // K-ragged GEMMs: NVFP4 x dense with A staged in TMEM
        if constexpr (KIND == Kind::NVFP4_BF16_TMEM &&
                      Tile<KIND, BN, STAGES, NUM_ACC>::SMEM_BYTES + kGroupTableBytes <= 232448)
            return launch_mode<KIND, BN, STAGES, NUM_ACC, kModeKGrouped>(maps, args, grid, stream);
        else
            return cudaErrorInvalidValue;
    }
    if (args.group_offs) {
        // grouped GEMMs: NVFP4, and NVFP4 x dense with A staged in TMEM
        if constexpr (KIND == Kind::NVFP4 ||
                      (KIND == Kind::NVFP4_BF16_TMEM &&
                       Tile<KIND, BN, STAGES, NUM_ACC>::SMEM_BYTES + kGroupTableBytes <= 232448))
            return launch_mode<KIND, BN, STAGES, NUM_ACC, kModeGrouped>(maps, args, grid, stream);
        else
            return cudaErrorInvalidValue;
    }
    if (has_epilogue(args))
        return launch_mode<KIND, BN, STAGES, NUM_ACC, kModeEpi>(maps, args, grid, stream);
    return launch_mode<KIND, BN, STAGES, NUM_ACC, kModePlain>(maps, args, grid, stream);
}

template <Kind KIND, int BN, int STAGES, int NUM_ACC>
static constexpr PlanInfo make_plan(const char *name)
{
    using T = Tile<KIND, BN, STAGES, NUM_ACC>;
    // the TMEM-staged dense variant serves calls of kind NVFP4_BF16
    constexpr Kind kind = KIND == Kind::NVFP4_BF16_TMEM ? Kind::NVFP4_BF16 : KIND;
    return PlanInfo{name, kind, Family::TC1, 1, T::BM, BN, STAGES, NUM_ACC, T::K_BLOCK, T::SMEM_BYTES,
                    T::THREADS, T::TMEM_COLS};
}

#define BSG_TC1_PLANS(X)                                         \
    X(Kind::NVFP4, 256, 3, 1, "nvfp4_tc1_128x256_s3_acc1")       \
    X(Kind::NVFP4, 128, 5, 2, "nvfp4_tc1_128x128_s5_acc2")       \
    X(Kind::FP8, 256, 4, 2, "fp8_tc1_128x256_s4_acc2")           \
    X(Kind::FP8, 128, 6, 2, "fp8_tc1_128x128_s6_acc2")           \
    X(Kind::NVFP4_BF16, 256, 3, 2, "nvfp4bf16_tc1_128x256_s3_acc2") \
    X(Kind::NVFP4_BF16, 128, 5, 2, "nvfp4bf16_tc1_128x128_s5_acc2") \
    X(Kind::NVFP4_BF16_TMEM, 256, 5, 1, "nvfp4bf16_tc1_128x256_s5_acc1_tmema") \
    X(Kind::NVFP4_BF16_TMEM, 128, 8, 2, "nvfp4bf16_tc1_128x128_s8_acc2_tmema")

#define BSG_PLAN_INFO(K, BN, S, A, NAME) make_plan<K, BN, S, A>(NAME),
static const PlanInfo kTc1Plans[] = {BSG_TC1_PLANS(BSG_PLAN_INFO)};
#undef BSG_PLAN_INFO

int tc1_num_plans() { return (int)(sizeof(kTc1Plans) / sizeof(kTc1Plans[0])); }

const PlanInfo &tc1_plan(int i) { return kTc1Plans[i]; }

cudaError_t tc1_launch(int id, const GemmMaps &maps, const GemmArgs &args, int grid,
                       cudaStream_t stream)
{
    int i = 0;
#define BSG_PLAN_LAUNCH(K, BN, S, A, NAME)                         \
    if (id == i)                                                  \
        return launch_impl<K, BN, S, A>(maps, args, grid, stream); \
    ++i;
    BSG_TC1_PLANS(BSG_PLAN_LAUNCH)
#undef BSG_PLAN_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace bsg
