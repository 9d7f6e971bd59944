// CTA-pair persistent block-scaled GEMM: one 256 x BN output tile per pair of
// CTAs on two SMs, computed by tcgen05.mma.cta_group::2 -- a single MMA
// spans both CTAs' shared and tensor memory ("Together AI Ports ThunderKittens
// GEMM Kernels to NVIDIA Vera Rubin NVL72", introduction: one MMA spans two
// CTAs across two SMs, loaders / one MMA warp / a consumer warpgroup, and a
// persistent kernel whose next tile streams in while the last one drains).
//
// Per CTA of the pair (rank r = 0 leader, 1 peer):
//   A rows   [256*pm + 128*r, +128)      -> own smem (16 KiB per stage)
//   B rows   [BN*nt + (BN/2)*r, +BN/2)    -> own smem; the MMA reads both halves
//   NVFP4 scales: own 128 rows of A, all BN rows of B, written smem -> own TMEM
//   D rows   [256*pm + 128*r, +128) x BN  in own TMEM, drained by own epilogue
// Each CTA therefore loads half of B per output tile instead of all of it,
// which halves the B bytes per SM and leaves room for a deeper ring.
//
// Roles: warp 0 TMA producer (both CTAs), warp 1 TMEM allocation (both) and
// the MMA thread (leader), warps 2..5 the scale writers (both CTAs, NVFP4),
// warps 6..9 the epilogue (both).
//
// NVFP4 scales: each CTA's producer loads a stage's scales first, on the
// CTA's own barrier; four scale writers per CTA (one per TMEM sub-partition)
// move them from shared memory into their TMEM lanes with tcgen05.st and
// arrive on the leader's scale-ready barrier, which the MMA thread waits on
// beside the A/B full barrier. Copying them with tcgen05.cp from the MMA
// thread instead was measured to cost ~90 cycles per pair copy, 12 copies per
// stage, which bounded the MMA rate.
//
// Synchronisation: every load of both CTAs completes on the LEADER's full
// barrier (TMA .cta_group::2); the leader's MMA thread issues the pair MMAs
// and commits with multicast to both CTAs' empty / accumulator-full
// barriers; both epilogues arrive on the leader's accumulator-empty barrier.
#include "bsg_internal.h"
#include "gemm_common.cuh"
#include "group.cuh"
#include "ptx.cuh"

namespace bsg {

template <Kind KIND, int BN, int STAGES, int NUM_ACC, bool PACKED = false>
struct PairTile {
    static constexpr bool kFp4 = KIND == Kind::NVFP4;
    // NVFP4 activations x dense BF16 weights: each CTA expands its own 128
    // rows of A (E2M1 codes + block scales) into its own TMEM, 32 columns per
    // stage, with the warps that write NVFP4 scales in the other kind; the
    // leader's pair MMA (kind::f16) reads A from both CTAs' TMEM
    static constexpr bool kDense = KIND == Kind::NVFP4_BF16_TMEM;
    static constexpr int CLUSTER = 2;                     // CTAs per cluster: one pair
    static constexpr int BM = 128;                        // rows per CTA
    static constexpr int TILE_M = 256;                    // rows per pair
    static constexpr int ROW_BYTES = 128;
    static constexpr int K_BLOCK = kFp4 ? 256 : kDense ? 64 : 128;
    static constexpr int MMA_K_BYTES = 32;
    static constexpr int MMAS = ROW_BYTES / MMA_K_BYTES;
    static constexpr int B_ROWS = BN / 2;                 // B rows held by each CTA
    // FP8 tiles 512 wide: two pair MMAs of N = 256 per K step, into
    // accumulator columns [0, 256) and [256, 512); each CTA holds 128 B rows
    // of each N half (one 3-D copy of 2 x 128 rows), the whole accumulator
    // filling TMEM (no block scales in this kind)
    static constexpr bool kWideN = BN == 512;
    static constexpr int MMA_N = kWideN ? 256 : BN;
    static constexpr int A_BYTES = kDense ? 0 : BM * ROW_BYTES;
    static constexpr int B_BYTES = B_ROWS * ROW_BYTES;
    static constexpr int APK_BYTES = kDense ? BM * 32 : 0;   // dense: this CTA's codes (128 rows x 32 bytes)
    static constexpr int ASF_BYTES = kDense ? 512 : 0;       // and their scales (one 512-byte block)
    static constexpr int A_COLS = kDense ? ROW_BYTES / 4 : 0; // TMEM columns of one stage's expanded A
    static constexpr int SF_BLOCK_BYTES = 2048;           // 128 rows x 16 scales
    static constexpr int SFB_CHUNKS = kFp4 ? BN / 128 : 0;
    static constexpr int SFA_BYTES = kFp4 ? SF_BLOCK_BYTES : 0;
    static constexpr int SFB_BYTES = SFB_CHUNKS * SF_BLOCK_BYTES;
    static constexpr int STAGE_BYTES =
        (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES + APK_BYTES + ASF_BYTES + 1023) / 1024 * 1024;
    // Epilogue warps: each drains 32 TMEM lanes x 128 columns. 256-wide NVFP4
    // tiles (one accumulator, so every tile's drain stalls the MMA) use two
    // per sub-partition to release TMEM sooner; FP8 tiles (two accumulators,
    // drain overlapped) and 128-wide tiles use one.
    // (dense: 4, since its eight expansion warps would otherwise leave too
    // few registers per thread for the epilogue variants)
    static constexpr int EPI_WARPS = ((kFp4 && BN == 256) || kWideN) ? 8 : 4;
    static constexpr int EPI_COLS = 64;
    static constexpr int EPI_CHUNKS = BN * 4 / EPI_WARPS / EPI_COLS;   // 64-column chunks per warp (2 or 4)
    static constexpr int EPI_BUFS = (EPI_CHUNKS == 2 || kWideN) ? 1 : 2;   // 4 KiB staging buffers per warp
    static constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 2;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
    // mbarrier layout (8 bytes each): full, empty per stage; full, empty per
    // accumulator; the drain barrier; scale-ready, scale-full per stage
    static constexpr int BAR_FULL = 0;
    static constexpr int BAR_EMPTY = BAR_FULL + STAGES;
    static constexpr int BAR_TFULL = BAR_EMPTY + STAGES;
    static constexpr int BAR_TEMPTY = BAR_TFULL + NUM_ACC;
    static constexpr int BAR_DRAIN = BAR_TEMPTY + NUM_ACC;
    static constexpr int BAR_SFREADY = BAR_DRAIN + 1;
    static constexpr int BAR_SFFULL = BAR_SFREADY + STAGES;
    static constexpr int BAR_PFULL = BAR_SFFULL + STAGES;   // PACKED: the peer's own A/B tiles landed
    static constexpr int NUM_BARS = BAR_PFULL + (PACKED ? STAGES : 0);
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + NUM_BARS * 8 + 16;
    // NVFP4: one scale writer per TMEM sub-partition; dense: two expansion
    // warps per sub-partition, each taking half of every row
    static constexpr int SCALE_WARPS = kDense ? 8 : 4;
    static constexpr int EPI_WARP0 = 2 + SCALE_WARPS;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);   // producer, MMA, scale warps, epilogue
    static constexpr int SFA_COLS = kFp4 ? 4 * MMAS : 0;
    static constexpr int SFB_COLS = kFp4 ? 4 * SFB_CHUNKS * MMAS : 0;
    static constexpr int SF_COLS = SFA_COLS + SFB_COLS;
    static constexpr int TMEM_USED = NUM_ACC * BN + STAGES * (SF_COLS + A_COLS);
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static constexpr uint32_t IDESC =
        kFp4 ? idesc_nvfp4(TILE_M, BN) : kDense ? idesc_bf16(TILE_M, BN) : idesc_fp8(TILE_M, MMA_N);
    static constexpr uint32_t IDESC_F16 = idesc_f16(TILE_M, BN);   // dense kind with FP16 B

    static_assert(BN % 128 == 0 && (BN <= 256 || (BN == 512 && KIND == Kind::FP8 && NUM_ACC == 1 && !PACKED)),
                  "pair tile N: B halves of 64 or 128 rows, or FP8 tiles of two 256-wide halves");
    static_assert(!PACKED || (kFp4 && BN == 256 && A_BYTES == 16384 && B_BYTES == 16384),
                  "tile-packed operands: NVFP4 256-wide pairs, one 16 KiB tile of A and of B per CTA and stage");
    static_assert(TMEM_USED <= 512, "TMEM: accumulators plus scales exceed 512 columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-byte aligned (128B swizzle)");
};

// Grouped (routed MoE) mode of the pair: one 256-row pair tile row per 256
// rows of each slice, so a slice of up to 256 rows is one tile row whose
// weight tile each CTA streams half of. The slice table (boundaries, first
// 128-row scale block and first pair tile row of every slice) sits beside
// the barriers; it bounds the slices to kPairMaxGroups (bsg_internal.h).
constexpr int kPairGroupTableBytes = 3 * (kPairMaxGroups + 1) * 4;

// EPI: the epilogue-variant instantiation (bias, gamma, scattered rows).
// GROUPED: the grouped GEMM over ragged row slices (with the variants'
// epilogue; NVFP4 256-wide tiles).
// PACKED: A and B arrive as tile-packed operands, one 16 KiB bulk copy per
// CTA, tile and stage (a copy of contiguous bytes takes operands into an SM
// faster than a tensor-map box of 128 rows); each CTA's copies complete on
// its own barrier, and the peer's warp 1 relays their arrival to the leader.
template <Kind KIND, int BN, int STAGES, int NUM_ACC, bool EPI, bool PACKED = false, bool GROUPED = false>
__global__ void __launch_bounds__(PairTile<KIND, BN, STAGES, NUM_ACC, PACKED>::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmSFA,
                     const __grid_constant__ CUtensorMap tmSFB, const GemmArgs args)
{
    using T = PairTile<KIND, BN, STAGES, NUM_ACC, PACKED>;
    static_assert(!GROUPED || (EPI && T::kFp4 && BN == 256 && !PACKED &&
                               T::SMEM_BYTES + kPairGroupTableBytes <= 232448),
                  "grouped pair: NVFP4 256-wide tiles with room for the slice table");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const uint32_t s_epi = base + STAGES * T::STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + STAGES * T::STAGE_BYTES + T::EPI_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t full0 = bar0 + 8u * T::BAR_FULL;          // [STAGES] loads -> MMA (leader's used)
    const uint32_t empty0 = bar0 + 8u * T::BAR_EMPTY;        // [STAGES] MMA -> loads (both CTAs)
    const uint32_t tfull0 = bar0 + 8u * T::BAR_TFULL;        // [NUM_ACC] MMA -> epilogues (both)
    const uint32_t tempty0 = bar0 + 8u * T::BAR_TEMPTY;      // [NUM_ACC] epilogues -> MMA (leader's)
    const uint32_t drain_bar = bar0 + 8u * T::BAR_DRAIN;
    const uint32_t sfready0 = bar0 + 8u * T::BAR_SFREADY;    // [STAGES] scales in TMEM (both CTAs) -> MMA (leader's)
    const uint32_t sffull0 = bar0 + 8u * T::BAR_SFFULL;      // [STAGES] own scale loads -> own scale warps
    const uint32_t pfull0 = bar0 + 8u * T::BAR_PFULL;        // [STAGES] PACKED: own operand tiles (peer)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + T::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // grouped: slice boundaries, first 128-row block and first pair tile row
    // of each slice (group.cuh)
    int *const s_go = reinterpret_cast<int *>(tmem_slot + 4);
    int *const s_gb = s_go + (kPairMaxGroups + 1);
    int *const s_gp = s_gb + (kPairMaxGroups + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const uint32_t rank = crank & 1u;           // within the pair: 0 leader, 1 peer
    const uint32_t lead = crank & ~1u;          // cluster rank of this pair's leader
    const bool leader = rank == 0;
    const Watchdog wd{args.status, args.timeout_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // PACKED: the leader's own arrival plus the peer's relay
            mbar_init(full0 + 8u * s, PACKED ? 2 : 1);
            if constexpr (PACKED)
                mbar_init(pfull0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);    // one commit of the pair's MMAs
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            mbar_init(tfull0 + 8u * a, 1);
            mbar_init(tempty0 + 8u * a, 2 * T::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(sfready0 + 8u * s, 2 * T::SCALE_WARPS);
            mbar_init(sffull0 + 8u * s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmD);
        if constexpr (T::kFp4) {
            prefetch_tensormap(&tmSFA);
            prefetch_tensormap(&tmSFB);
        }
    }
    __syncwarp();
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), T::TMEM_COLS);
        tmem_relinquish_pair();
    }
    if constexpr (GROUPED) {
        if (warp == 2) {
            griddep_wait();      // the offsets may come from the previous grid
            build_group_table(args.group_offs, args.num_groups, args.M, s_go, s_gb, lane);
            build_block_prefix(s_go, args.num_groups, T::TILE_M, s_gp, lane);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    // both CTAs' barriers exist before any remote use: thread 0's
    // fence.mbarrier_init.release.cluster orders its initialisations before
    // its (relaxed) cluster arrival
    cluster_arrive_relaxed();
    cluster_wait();
    tc_fence_after_sync();
    griddep_wait();              // a dependent launch: the previous grid's writes are visible
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    // grouped: one pair tile row per 256 rows of each slice
    const int num_m_tiles = GROUPED ? s_gp[args.num_groups] : args.num_m_tiles;
    const int num_tiles = num_m_tiles * args.num_n_tiles;
    const int nkb = args.num_k_blocks;
    const bool b_f16 = args.b_f16 != 0;   // dense kind: B (and the expanded A) are FP16, not BF16
    const int cluster_id = blockIdx.x / T::CLUSTER;
    const int num_clusters = gridDim.x / T::CLUSTER;
    auto tile_coords = [&](int tile, int &pm, int &nt) {
        raster_tile(tile, args.raster_group, num_m_tiles, args.num_n_tiles, pm, nt);
    };
    // pair tile row pm -> its slice g, first row of A, end of the slice's
    // rows and first 128-row block of the (per-slice) swizzled A scales
    auto pair_rows = [&](int pm, int &g, int &row0, int &row_end, int &ablk0) {
        if constexpr (GROUPED) {
            g = group_of_block(s_gp, args.num_groups, pm);
            const int t = pm - s_gp[g];
            row0 = s_go[g] + t * T::TILE_M;
            row_end = s_go[g + 1];
            ablk0 = s_gb[g] + 2 * t;
        } else {
            g = 0;
            row0 = pm * T::TILE_M;
            row_end = args.M;
            ablk0 = 2 * pm;
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer (both CTAs): own A half, own B half, own scales
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // A's row panels and their scales are re-read by the later tiles
            // of the raster group (its M tiles sweep every N tile), so they
            // are kept in L2 first; B's panels, read by the group's M tiles
            // one after another, keep the default policy (evict-first for
            // them measured 0.7 % slower)
            const uint64_t pol_a = l2_policy_evict_last();
            for (int tile = cluster_id; ok && tile < num_tiles; tile += num_clusters) {
                int pm, nt, g, row0, row_end, ablk0;
                tile_coords(tile, pm, nt);
                pair_rows(pm, g, row0, row_end, ablk0);
                // grouped: a CTA whose 128 rows all lie past its slice loads
                // no A and no A scales (its rows are never stored); B comes
                // from the slice's own weights
                const bool a_in = !GROUPED || row0 + (int)rank * T::BM < row_end;
                const bool peer_a_in = !GROUPED || row0 + T::BM < row_end;
                const int b_row0 = (GROUPED ? g * args.N : 0) + nt * BN + (int)rank * T::B_ROWS;
                const int sfb_blk0 = (GROUPED ? g * args.sfb_row_blocks : 0) + nt * T::SFB_CHUNKS;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, wd, abort_flag, 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * T::STAGE_BYTES;
                    const uint32_t sb = sa + T::A_BYTES;
                    const uint32_t fb = mapa_shared(full0 + 8u * stage, lead);
                    if constexpr (T::kFp4) {
                        // scales first, on this CTA's own barrier: its scale warps
                        // write them into its TMEM while A and B are in flight.
                        // 256-byte rows of the swizzled scale layout: a stage is
                        // the 8 rows starting at (row_block * ncb + 4 kb) * 2.
                        const uint32_t sfb = sffull0 + 8u * stage;
                        mbar_arrive_expect_tx(sfb, (a_in ? T::SFA_BYTES : 0) + T::SFB_BYTES);
                        const uint32_t ssfa = sb + T::B_BYTES;
                        const int rba = ablk0 + (int)rank;
                        if (a_in)
                            tma_load_2d_hint(ssfa, &tmSFA, sfb, 0, (rba * args.sf_col_blocks + 4 * kb) * 2, pol_a);
                        // all SFB_CHUNKS 128-row blocks of B's scales in one
                        // copy: a 3-D view (256-byte rows, rows of a row block,
                        // row blocks), box 8 rows x SFB_CHUNKS row blocks
                        tma_load_3d(ssfa + T::SFA_BYTES, &tmSFB, sfb, 0, 8 * kb, sfb_blk0);
                    }
                    if constexpr (T::kDense) {
                        // this CTA's codes and scales on its own expansion
                        // barrier; its B half on the leader's full barrier
                        // (a CTA whose 128 rows all lie past M has no scale
                        // block to read: its codes are zero-filled, so
                        // whatever scales its shared memory holds give zeros,
                        // and its rows are never stored)
                        const uint32_t sfb = sffull0 + 8u * stage;
                        const uint32_t sapk = sb + T::B_BYTES;
                        const int sf_row = 2 * pm + (int)rank;
                        const bool rows_in = sf_row * T::BM < args.M;
                        mbar_arrive_expect_tx(sfb, T::APK_BYTES + (rows_in ? T::ASF_BYTES : 0));
                        tma_load_2d(sapk, &tmA, sfb, kb * 32, pm * T::TILE_M + (int)rank * T::BM);
                        if (rows_in)
                            bulk_load(sapk + T::APK_BYTES,
                                      args.sfa + ((size_t)sf_row * args.sf_col_blocks + kb) * 512u, T::ASF_BYTES,
                                      sfb);
                        if (leader)
                            mbar_arrive_expect_tx(full0 + 8u * stage, 2u * T::B_BYTES);
                    } else if constexpr (PACKED) {
                        // this CTA's A tile (row block 2 pm + r) and B tile
                        // (row block 2 nt + r) of k-block kb, one bulk copy
                        // each, on its own barrier (the leader's full one, or
                        // the peer's relayed one); a row block past M or N is
                        // not loaded -- its rows are never stored
                        const uint32_t own = leader ? full0 + 8u * stage : pfull0 + 8u * stage;
                        const int rba = 2 * pm + (int)rank, rbb = 2 * nt + (int)rank;
                        const bool a_in = rba * 128 < args.M, b_in = rbb * 128 < args.N;
                        mbar_arrive_expect_tx(own, (a_in ? T::A_BYTES : 0) + (b_in ? T::B_BYTES : 0));
                        if (a_in)
                            bulk_load(sa, args.a_packed + ((size_t)rba * nkb + kb) * 16384u, T::A_BYTES, own);
                        if (b_in)
                            bulk_load(sb, args.b_packed + ((size_t)rbb * nkb + kb) * 16384u, T::B_BYTES, own);
                    } else {
                        if (leader)
                            mbar_arrive_expect_tx(full0 + 8u * stage, (a_in ? T::A_BYTES : 0) +
                                                                          (peer_a_in ? T::A_BYTES : 0) +
                                                                          2u * T::B_BYTES);
                        if (a_in)
                            tma_load_2d_pair_hint(sa, &tmA, fb, kb * T::ROW_BYTES, row0 + (int)rank * T::BM, pol_a);
                    }
                    if constexpr (T::kWideN)
                        // rows nt * 512 + h * 256 + rank * 128 .. + 128 of
                        // both halves h: a 3-D view (k bytes, rows of a half,
                        // halves), one copy into two 16 KiB tiles
                        tma_load_3d_pair(sb, &tmB, fb, kb * T::ROW_BYTES, (int)rank * 128, 2 * nt);
                    else if constexpr (!PACKED)
                        tma_load_2d_pair(sb, &tmB, fb, kb * T::ROW_BYTES, b_row0);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let copies already issued land before the CTA goes away
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer: one thread of the leader drives both SMs' tensor cores
        // ------------------------------------------------------------------
        if (leader && lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t idesc = b_f16 ? T::IDESC_F16 : T::IDESC;
            for (int tile = cluster_id; ok && tile < num_tiles; tile += num_clusters) {
                if (!mbar_wait(tempty0 + 8u * acc, acc_phase ^ 1u, wd, abort_flag, 2)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(full0 + 8u * stage, phase, wd, abort_flag, 3)) {
                        ok = false;
                        break;
                    }
                    if constexpr (T::kFp4 || T::kDense) {
                        // the scale warps have written this stage's scales
                        // (NVFP4) / expanded A (dense) to both CTAs' TMEM
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
                            mma_nvfp4_pair(d_tmem, desc_kmajor_sw128(sa + T::MMA_K_BYTES * j),
                                           desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                           sfa_t + 4u * j, sfb_t + 4u * j * T::SFB_CHUNKS,
                                           (kb | j) != 0 ? 1u : 0u);
                    } else if constexpr (T::kDense) {
                        const uint32_t a_t = tmem + (uint32_t)(NUM_ACC * BN + stage * T::A_COLS);
#pragma unroll
                        for (int j = 0; j < T::MMAS; ++j)
                            mma_bf16_pair_tmem_a(d_tmem, a_t + (uint32_t)(j * T::MMA_K_BYTES / 4),
                                                 desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                                 (kb | j) != 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int j = 0; j < T::MMAS; ++j) {
                            if constexpr (T::kWideN) {
                                // one A slice, both N halves: the second MMA
                                // reads A from the collector buffer
                                mma_fp8_pair_a_fill(d_tmem, desc_kmajor_sw128(sa + T::MMA_K_BYTES * j),
                                                    desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                                    (kb | j) != 0 ? 1u : 0u);
                                mma_fp8_pair_a_lastuse(d_tmem + (uint32_t)T::MMA_N,
                                                       desc_kmajor_sw128(sa + T::MMA_K_BYTES * j),
                                                       desc_kmajor_sw128(sb + T::B_BYTES / 2 + T::MMA_K_BYTES * j),
                                                       idesc, (kb | j) != 0 ? 1u : 0u);
                            } else {
                                mma_fp8_pair(d_tmem, desc_kmajor_sw128(sa + T::MMA_K_BYTES * j),
                                             desc_kmajor_sw128(sb + T::MMA_K_BYTES * j), idesc,
                                             (kb | j) != 0 ? 1u : 0u);
                            }
                        }
                    }
                    // frees the stage in both CTAs
                    tc_commit_pair_multicast(empty0 + 8u * stage, 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc_commit_pair_multicast(tfull0 + 8u * acc, (uint16_t)(0x3u << lead));   // both epilogues may drain
                if (++acc == NUM_ACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            tc_commit_pair(drain_bar);
            mbar_wait_quiet(drain_bar, 0, wd.limit_ns);
        }
        if constexpr (PACKED) {
            // the peer's relay: its operand tiles of each stage have landed
            // (own barrier), so the leader's full barrier gets its second
            // arrival -- a relaxed remote arrive, as the scale writers'
            if (!leader && lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                for (int tile = cluster_id; ok && tile < num_tiles; tile += num_clusters) {
                    for (int kb = 0; kb < nkb; ++kb) {
                        if (!mbar_wait(pfull0 + 8u * stage, phase, wd, abort_flag, 11)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_remote_relaxed(mapa_shared(full0 + 8u * stage, lead));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
    } else if (warp < T::EPI_WARP0) {
        // ------------------------------------------------------------------
        // Scale warps (NVFP4) (both CTAs: each writes its own TMEM): one per TMEM sub-partition
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
            for (int tile = cluster_id; ok && tile < num_tiles; tile += num_clusters) {
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
                    if (lane == 0) {
                        // the stores have completed (wait::st): the leader's own
                        // writers arrive locally, the peer's with a relaxed remote
                        // arrive (a release at cluster scope measured ~1100 cycles)
                        if (leader)
                            mbar_arrive(sfready0 + 8u * stage);
                        else
                            mbar_arrive_remote_relaxed(mapa_shared(sfready0 + 8u * stage, lead));
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else if constexpr (T::kDense) {
            // expansion warps (both CTAs), two per TMEM sub-partition: row r
            // of this CTA's 128 rows of A, column half hc, from codes + block
            // scales to BF16 in its own TMEM lanes, then the leader's ready
            // barrier (as the scale writers above)
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const int r = (warp & 3) * 32 + lane;
            const int hc = (warp - 2) >> 2;                // column half of the row
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = cluster_id; ok && tile < num_tiles; tile += num_clusters) {
                for (int kb = 0; kb < nkb; ++kb) {
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
                    tmem_st_32x32b_x16(tmem + lane_off + (uint32_t)(NUM_ACC * BN + stage * T::A_COLS + 16 * hc), w);
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            mbar_arrive(sfready0 + 8u * stage);
                        else
                            mbar_arrive_remote_relaxed(mapa_shared(sfready0 + 8u * stage, lead));
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------------
        // Epilogue (both CTAs): own 128 rows of the pair's tile
        // ------------------------------------------------------------------
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        constexpr int COLS_PER_WARP = T::EPI_CHUNKS * T::EPI_COLS;   // 128 or 256 columns per warp
        const int h = (warp - T::EPI_WARP0) / 4;                  // column block of this warp
        const uint32_t ebuf = s_epi + (uint32_t)(warp - T::EPI_WARP0) * T::EPI_BUFS * T::EPI_BUF_BYTES;
        float scale = args.alpha;
        if constexpr (!T::kFp4) {
            if (args.sA)
                scale *= *args.sA;
            if (args.sB)
                scale *= *args.sB;
        }
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint64_t pol_d = l2_policy_evict_first();
        for (int tile = cluster_id; tile < num_tiles; tile += num_clusters) {
            int pm, nt, g, row0, row_end, ablk0;
            tile_coords(tile, pm, nt);
            pair_rows(pm, g, row0, row_end, ablk0);
            const int x0 = nt * BN + h * COLS_PER_WARP;            // first column of this warp
            const int y = row0 + (int)rank * T::BM + q * 32;       // first row of this warp's 32
            // grouped: a slice's own bias; rows of the warp that TMA could
            // store past the slice's end go one by one (as scattered rows)
            const float *const bias = (GROUPED && args.bias) ? args.bias + (size_t)g * args.N : args.bias;
            const bool per_row = EPI && (args.scatter || (GROUPED && y + 32 > row_end));
            RowEpi re{1.0f, -1};
            if constexpr (EPI) {
                re = load_row_epi(args, y + lane, row_end);
                prefetch_bias(bias, args.N, x0, COLS_PER_WARP, lane);
            }
            if (!warp_wait(tfull0 + 8u * acc, acc_phase, wd, abort_flag, 4, lane))
                break;
            tc_fence_after_sync();
            const uint32_t t_acc = tmem + lane_off + (uint32_t)(acc * BN + h * COLS_PER_WARP);
            // chunk ch's 64 TMEM columns: both 32-column reads issued back to
            // back, completed by one tcgen05.wait::ld
            auto load_chunk = [&](int ch, uint32_t (&v0)[32], uint32_t (&v1)[32]) {
                tmem_ld_32x32b_x32(t_acc + ch * T::EPI_COLS, v0);
                tmem_ld_32x32b_x32(t_acc + ch * T::EPI_COLS + 32, v1);
            };
            // chunk ch's 64 FP32 columns -> alpha (bias, gamma) -> 32 BF16 pairs
            auto convert_chunk = [&](int ch, const uint32_t (&v0)[32], const uint32_t (&v1)[32],
                                     uint32_t (&pk)[32]) {
                if constexpr (EPI) {
                    convert64_epi(v0, v1, pk, scale, re, args, bias, x0 + ch * T::EPI_COLS);
                } else {
                    convert32(v0, pk, scale);
                    convert32(v1, pk + 16, scale);
                }
            };
            // one 64-column chunk from registers into a 128B-swizzled staging
            // buffer, once the store that last used the buffer has read it
            auto stage_out = [&](const uint32_t (&pk)[32], uint32_t sbuf) {
                if (lane == 0) {
                    if constexpr (T::EPI_BUFS == 1)
                        bulk_wait_group_read<0>();
                    else
                        bulk_wait_group_read<1>();
                }
                __syncwarp();
                const uint32_t row = sbuf + (uint32_t)lane * 128u;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(row + ((uint32_t)(c ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                                 pk[4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
            };
            auto store_chunk = [&](int ch, uint32_t sbuf) {
                const int x = x0 + ch * T::EPI_COLS;
                if (per_row) {
                    scatter_chunk(gbase + (sbuf - base), re.dst, args.d, args.N, x, lane);
                } else if (lane == 0) {
                    if (x < args.N && y < args.M)
                        tma_store_2d_hint(&tmD, sbuf, x, y, pol_d);   // D is not read again here
                    bulk_commit_group();
                }
            };
            auto release = [&]() {      // the accumulator is read out (tcgen05.wait::ld): the MMA may reuse it
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        mbar_arrive(tempty0 + 8u * acc);
                    else
                        mbar_arrive_remote_relaxed(mapa_shared(tempty0 + 8u * acc, lead));
                }
            };
            if constexpr (T::EPI_CHUNKS == 2) {
                // chunk 0 read and converted; chunk 1 read, then TMEM is
                // released at once -- staging both chunks, chunk 1's
                // conversion and both TMA stores overlap the next tile's MMAs
                uint32_t pk[32];
                {
                    uint32_t v0[32], v1[32];
                    load_chunk(0, v0, v1);
                    tmem_ld_wait();
                    convert_chunk(0, v0, v1, pk);
                }
                {
                    uint32_t v0[32], v1[32];
                    load_chunk(1, v0, v1);
                    tmem_ld_wait();
                    release();
                    stage_out(pk, ebuf);
                    store_chunk(0, ebuf);
                    convert_chunk(1, v0, v1, pk);
                }
                stage_out(pk, ebuf);
                store_chunk(1, ebuf);
            } else {
                // four chunks through two alternating buffers; TMEM is released
                // right after the last chunk's read, before its conversion
#pragma unroll 1
                for (int ch = 0; ch < T::EPI_CHUNKS; ++ch) {
                    uint32_t pk[32];
                    {
                        uint32_t v0[32], v1[32];
                        load_chunk(ch, v0, v1);
                        tmem_ld_wait();
                        if (ch == T::EPI_CHUNKS - 1)
                            release();
                        convert_chunk(ch, v0, v1, pk);
                    }
                    const uint32_t sbuf = ebuf + (uint32_t)(T::EPI_BUFS == 2 ? (ch & 1) : 0) * T::EPI_BUF_BYTES;
                    stage_out(pk, sbuf);
                    store_chunk(ch, sbuf);
                }
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
    cluster_sync_all();          // no CTA leaves while its peer may still touch it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, T::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Plans and launchers
// ---------------------------------------------------------------------------
template <Kind KIND, int BN, int STAGES, int NUM_ACC, bool PACKED = false>
static cudaError_t pair_launch_impl(const GemmMaps &maps, const GemmArgs &args, int grid,
                                    cudaStream_t stream)
{
    using T = PairTile<KIND, BN, STAGES, NUM_ACC, PACKED>;
    auto kern = has_epilogue(args) ? gemm_pair_kernel<KIND, BN, STAGES, NUM_ACC, true, PACKED>
                                   : gemm_pair_kernel<KIND, BN, STAGES, NUM_ACC, false, PACKED>;
    int smem = T::SMEM_BYTES;
    if (args.group_offs) {
        // the grouped instantiation: the 5-stage NVFP4 256-wide plan only
        if constexpr (KIND == Kind::NVFP4 && BN == 256 && STAGES == 5 && !PACKED) {
            kern = gemm_pair_kernel<KIND, BN, STAGES, NUM_ACC, true, PACKED, true>;
            smem += kPairGroupTableBytes;
        } else {
            return cudaErrorInvalidValue;
        }
    }
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(T::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T::CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = args.pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, maps.a, maps.b, maps.d, maps.sfa, maps.sfb, args);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <Kind KIND, int BN, int STAGES, int NUM_ACC, bool PACKED = false>
static int pair_clusters_impl()
{
    using T = PairTile<KIND, BN, STAGES, NUM_ACC, PACKED>;
    auto kern = gemm_pair_kernel<KIND, BN, STAGES, NUM_ACC, false, PACKED>;   // the EPI instantiation has the same footprint
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T::CLUSTER, 1, 1);
    cfg.blockDim = dim3(T::THREADS, 1, 1);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = T::CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void *)kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <Kind KIND, int BN, int STAGES, int NUM_ACC, bool PACKED = false>
static constexpr PlanInfo make_pair_plan(const char *name)
{
    using T = PairTile<KIND, BN, STAGES, NUM_ACC, PACKED>;
    // the TMEM-staged dense pair serves calls of kind NVFP4_BF16
    constexpr Kind kind = KIND == Kind::NVFP4_BF16_TMEM ? Kind::NVFP4_BF16 : KIND;
    return PlanInfo{name, kind, Family::PAIR, 2, T::TILE_M, BN, STAGES, NUM_ACC, T::K_BLOCK, T::SMEM_BYTES,
                    T::THREADS, T::TMEM_COLS, PACKED ? 1 : 0};
}

// The first plan of each kind and shape is the planner's; the shallower
// rings are there for the stage sweep (bsg_force_plan).
#define BSG_PAIR_PLANS(X)                                                    \
    X(Kind::NVFP4, 256, 5, 1, false, "nvfp4_tc2_256x256_s5_acc1")         \
    X(Kind::NVFP4, 128, 6, 2, false, "nvfp4_tc2_256x128_s6_acc2")         \
    X(Kind::FP8, 256, 6, 2, false, "fp8_tc2_256x256_s6_acc2")             \
    X(Kind::NVFP4, 256, 4, 1, false, "nvfp4_tc2_256x256_s4_acc1")         \
    X(Kind::NVFP4, 256, 3, 1, false, "nvfp4_tc2_256x256_s3_acc1")         \
    X(Kind::FP8, 256, 4, 2, false, "fp8_tc2_256x256_s4_acc2")             \
    X(Kind::NVFP4_BF16_TMEM, 256, 8, 1, false, "nvfp4bf16_tc2_256x256_s8_acc1_tmema") \
    X(Kind::NVFP4, 256, 5, 1, true, "nvfp4_tc2_256x256_s5_acc1_packed") \
    X(Kind::FP8, 512, 4, 1, false, "fp8_tc2_256x512_s4_acc1")

#define BSG_PAIR_INFO(K, BN, S, A, PK, NAME) make_pair_plan<K, BN, S, A, PK>(NAME),
static const PlanInfo kPairPlans[] = {BSG_PAIR_PLANS(BSG_PAIR_INFO)};
#undef BSG_PAIR_INFO

int pair_num_plans() { return (int)(sizeof(kPairPlans) / sizeof(kPairPlans[0])); }

const PlanInfo &pair_plan(int i) { return kPairPlans[i]; }

cudaError_t pair_launch(int id, const GemmMaps &maps, const GemmArgs &args, int grid,
                        cudaStream_t stream)
{
    int i = 0;
#define BSG_PAIR_LAUNCH(K, BN, S, A, PK, NAME)                              \
    if (id == i)                                                               \
        return pair_launch_impl<K, BN, S, A, PK>(maps, args, grid, stream); \
    ++i;
    BSG_PAIR_PLANS(BSG_PAIR_LAUNCH)
#undef BSG_PAIR_LAUNCH
    return cudaErrorInvalidValue;
}

int pair_max_clusters(int id)
{
    int i = 0;
#define BSG_PAIR_OCC(K, BN, S, A, PK, NAME)            \
    if (id == i)                                          \
        return pair_clusters_impl<K, BN, S, A, PK>();  \
    ++i;
    BSG_PAIR_PLANS(BSG_PAIR_OCC)
#undef BSG_PAIR_OCC
    return 0;
}

}  // namespace bsg
