// Skinny-M NVFP4 GEMM (up to 2 x 256 activation rows, large N x K weights):
// the memory-bound weight-streaming shape of a projection layer.
//
// A regular 128 x 256 output tiling gives such shapes only ceil(N/256) tiles
// per 128 rows -- 12 to 48 CTAs on a 152-SM GPU -- and every CTA walks all of
// K, so most SMs idle and the weights stream through a handful of them. This
// kernel instead
//   * swaps the operands: it computes D^T = (B * sB)(A * sA)^T, so 128 weight
//     rows are the MMA's M side and the (padded) activation rows its N side;
//     more activation rows than the tile holds (up to two tiles) run as a
//     third grid dimension, each CTA taking one half of the rows;
//   * splits K across a thread-block cluster of S CTAs (any S from 1 to 8,
//     chosen by the host so that the whole grid is resident at once and
//     fills the SMs) so that (N/128) * S CTAs stream disjoint weight bytes in
//     parallel;
//   * reduces the S partial accumulators inside the cluster, with no partials
//     in HBM and no cluster-wide barrier on the critical path: the tile's 128
//     weight rows are cut into 16 groups of 8, CTA o owning groups
//     [16 o / S, 16 (o + 1) / S). Every CTA pushes the rows it does not own
//     straight from TMEM into the owner's shared memory (st.async, 16 bytes
//     at a time, each completing bytes on the owner's mbarrier); the owner
//     sums the S terms of its rows in rank order (deterministic), stages them
//     as BF16 and writes its columns of D with 16-byte stores. Where shared
//     memory is short the receive area aliases the drained stage ring, and a
//     sender pushes only after every peer has said that its ring is free (one
//     relaxed remote arrive per peer once its MMAs have completed).
// The first stages' loads are issued by the initialising thread before the
// block-wide setup barrier, so HBM latency overlaps TMEM allocation.
// Everything else follows the persistent 1-SM kernel: TMA producer warp, one
// MMA thread (tcgen05.mma kind::mxf4nvf4 block_scale, FP32 accumulator in
// TMEM), four scale-writer warps (tcgen05.st, one per TMEM sub-partition),
// four epilogue warps.
#include <cuda_bf16.h>

#include "bsg_internal.h"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace bsg {

template <int M_PAD, int STAGES>
struct SkinnyTile {
    static constexpr int BW = 128;                        // weight rows per CTA (MMA M)
    static constexpr int ROW_BYTES = 128;
    static constexpr int K_BLOCK = 256;
    static constexpr int MMA_K_BYTES = 32;
    static constexpr int MMAS = ROW_BYTES / MMA_K_BYTES;
    static constexpr int W_BYTES = BW * ROW_BYTES;        // weights (MMA A operand)
    static constexpr int X_BYTES = M_PAD * ROW_BYTES;     // activations (MMA B operand)
    static constexpr int SF_BLOCK_BYTES = 2048;
    static constexpr int SFX_CHUNKS = (M_PAD + 127) / 128;
    static constexpr int SFW_BYTES = SF_BLOCK_BYTES;
    static constexpr int SFX_BYTES = SFX_CHUNKS * SF_BLOCK_BYTES;
    static constexpr int STAGE_BYTES = W_BYTES + X_BYTES + SFW_BYTES + SFX_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    // receive area: FP32 [sender rank][column / 4][owned row][column % 4];
    // owners hold 8 * ceil(16 / S) rows at most, so S senders fill at most
    // recv_rows(S) = S * 8 * ceil(16 / S) rows: 128 for S = 1, 2, 4, 8, 144
    // for S = 3, 6 and 160 for S = 5 (168 for S = 7, never used). The area
    // holds 160 rows where shared memory allows, else 144 (no S = 5). 32
    // lanes pushing or reading the same 4 columns of consecutive rows touch
    // 512 consecutive bytes
    static constexpr int recv_rows(int S) { return S * 8 * ((16 + S - 1) / S); }
    // output staging, BF16 [M_PAD][owned rows] (all 128 without a split),
    // placed after the receive area
    static constexpr int OUT_BYTES = M_PAD * BW * 2;
    static constexpr int NUM_BARS = 3 * STAGES + 4;
    static constexpr int BAR_BYTES = NUM_BARS * 8 + 16;
    // epilogue-variant operands, staged once per CTA: gamma and destination
    // row of the M_PAD activation rows, bias of the tile's BW weight rows
    static constexpr int EPI_BYTES = (2 * M_PAD + BW) * 4;
    // the receive and staging areas get shared memory of their own where it
    // fits beside the ring (peers may then push as soon as their own MMAs
    // are done); otherwise they alias the drained ring and a sender first
    // waits for every peer to report its ring free
    static constexpr int smem_own(int rows) { return 1024 + RING_BYTES + rows * M_PAD * 4 + OUT_BYTES + EPI_BYTES + BAR_BYTES; }
    static constexpr int area_alias(int rows)
    {
        return RING_BYTES > rows * M_PAD * 4 + OUT_BYTES ? RING_BYTES : rows * M_PAD * 4 + OUT_BYTES;
    }
    static constexpr int smem_alias(int rows) { return 1024 + area_alias(rows) + EPI_BYTES + BAR_BYTES; }
    static constexpr int RECV_ROWS = smem_alias(160) <= 232448 ? 160 : 144;
    static constexpr int RECV_BYTES = RECV_ROWS * M_PAD * 4;
    static constexpr bool OWN_RECV = smem_own(RECV_ROWS) <= 232448;
    static constexpr int RECV_OFF = OWN_RECV ? RING_BYTES : 0;
    static constexpr int AREA = OWN_RECV ? RING_BYTES + RECV_BYTES + OUT_BYTES : area_alias(RECV_ROWS);
    static constexpr int SMEM_BYTES = 1024 + AREA + EPI_BYTES + BAR_BYTES;
    // split counts the receive area holds (bit S set): S <= 8, S != 7
    static constexpr int SPLITS_MASK = (1 << 1) | (1 << 2) | (1 << 3) | (1 << 4) | (1 << 6) | (1 << 8) |
                                       (recv_rows(5) <= RECV_ROWS ? 1 << 5 : 0);
    static constexpr int SCALE_WARPS = 4;
    static constexpr int EPI_WARP0 = 2 + SCALE_WARPS;
    static constexpr int EPI_WARPS = 4;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    static constexpr int SFA_COLS = 4 * MMAS;                     // weights' scales
    static constexpr int SFB_COLS = 4 * SFX_CHUNKS * MMAS;        // activations' scales
    static constexpr int SF_COLS = SFA_COLS + SFB_COLS;
    static constexpr int TMEM_USED = M_PAD + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static constexpr uint32_t IDESC = idesc_nvfp4(BW, M_PAD);

    static_assert(M_PAD % 32 == 0 && M_PAD >= 32 && M_PAD <= 256, "activation tile");
    static_assert(RECV_BYTES + OUT_BYTES <= AREA - RECV_OFF, "receive and staging areas");
    static_assert(TMEM_USED <= 512, "TMEM: accumulator plus scales exceed 512 columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");
    static_assert(STAGE_BYTES % 1024 == 0, "stages must stay 1024-byte aligned (128B swizzle)");
};

// args: num_n_tiles = weight tiles (N/128), num_k_blocks = K/256 (whole K);
// the split count S is the cluster size (gridDim.y): 1 to 6 or 8, and <=
// num_k_blocks; gridDim.z is the number of M_PAD-row activation blocks.

// First weight row (of the tile's 128) owned by cluster rank o of S: the
// rows go in 16 groups of 8, rank o taking groups [16 o / S, 16 (o+1) / S).
__device__ __forceinline__ int skinny_own_lo(int o, int S) { return 8 * ((16 * o) / S); }

// Parts of one producer step (see the producer in gemm_skinny_kernel).
constexpr int kStepAll = 0, kStepWeights = 1, kStepRest = 2;

// Cluster rank that owns weight row n (the last rank whose first group is
// at or below n's group).
__device__ __forceinline__ int skinny_owner(int n, int S) { return (S * ((n >> 3) + 1) - 1) >> 4; }

// The owned block's reduction, spread over the epilogue's threads: item
// (cq, r) sums columns [4 cq, 4 cq + 4) of owned row r over the S partials in
// the receive area, in rank order, scales them and stages them as BF16
// [m][r] (row stride rpo) for the store. EPI: s_bias[r] is the bias of
// owned row r (an output column), s_gamma[m] the gamma of output row m.
template <bool EPI>
__device__ __forceinline__ void reduce_owned(const uint8_t *recv, __nv_bfloat16 *out, int S, int rpo,
                                             int live_cols, float alpha, int t, int nthreads, const float *s_gamma,
                                             const float *s_bias)
{
    const int items = (live_cols / 4) * rpo;
    const int slot_bytes = rpo * live_cols * 4;
    for (int idx = t; idx < items; idx += nthreads) {
        const uint8_t *p = recv + idx * 16;          // [cq][r] with r fastest: idx == cq * rpo + r
        // the S (<= 8) partials' loads all in flight, then summed in rank order
        float4 v[8];
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (s < S)
                v[s] = *reinterpret_cast<const float4 *>(p + s * slot_bytes);
        float4 a = v[0];
#pragma unroll
        for (int s = 1; s < 8; ++s)
            if (s < S) {
                a.x += v[s].x;
                a.y += v[s].y;
                a.z += v[s].z;
                a.w += v[s].w;
            }
        const int r = idx % rpo;
        const int m0 = (idx / rpo) * 4;
        if constexpr (EPI) {
            const float b = s_bias[r];
            out[(m0 + 0) * rpo + r] = __float2bfloat16_rn(fmaf(a.x, alpha, b) * s_gamma[m0 + 0]);
            out[(m0 + 1) * rpo + r] = __float2bfloat16_rn(fmaf(a.y, alpha, b) * s_gamma[m0 + 1]);
            out[(m0 + 2) * rpo + r] = __float2bfloat16_rn(fmaf(a.z, alpha, b) * s_gamma[m0 + 2]);
            out[(m0 + 3) * rpo + r] = __float2bfloat16_rn(fmaf(a.w, alpha, b) * s_gamma[m0 + 3]);
        } else {
            out[(m0 + 0) * rpo + r] = __float2bfloat16_rn(a.x * alpha);
            out[(m0 + 1) * rpo + r] = __float2bfloat16_rn(a.y * alpha);
            out[(m0 + 2) * rpo + r] = __float2bfloat16_rn(a.z * alpha);
            out[(m0 + 3) * rpo + r] = __float2bfloat16_rn(a.w * alpha);
        }
    }
}

// EPI: the epilogue-variant instantiation (bias, gamma, scattered rows).
template <int M_PAD, int STAGES, bool EPI>
__global__ void __launch_bounds__(SkinnyTile<M_PAD, STAGES>::THREADS, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const GemmArgs args)
{
    using T = SkinnyTile<M_PAD, STAGES>;
    if (threadIdx.x == 0) {              // before any parameter read: the descriptor fetches overlap it
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    float *const s_gamma = reinterpret_cast<float *>(gbase + T::AREA);   // [M_PAD]
    int *const s_dst = reinterpret_cast<int *>(s_gamma + M_PAD);          // [M_PAD]
    float *const s_bias = reinterpret_cast<float *>(s_dst + M_PAD);       // [BW]
    uint64_t *bars = reinterpret_cast<uint64_t *>(gbase + T::AREA + T::EPI_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t full0 = bar0;                       // [STAGES] operands -> MMA
    const uint32_t empty0 = full0 + 8u * STAGES;       // [STAGES] MMA done -> producer
    const uint32_t sfready0 = empty0 + 8u * STAGES;    // [STAGES] scales in TMEM -> MMA
    const uint32_t tfull = sfready0 + 8u * STAGES;     // accumulator complete -> epilogue
    const uint32_t drain_bar = tfull + 8u;
    const uint32_t peer_free = drain_bar + 8u;         // every peer's ring may be written
    const uint32_t rx = peer_free + 8u;                // the peers' rows have landed here
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + T::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Watchdog wd{args.status, args.timeout_ns};
    const int nt = blockIdx.x;                          // weight tile
    const int S = gridDim.y;                            // K split == cluster size
    const int split = blockIdx.y;
    const uint32_t rank = cluster_ctarank();
    const int kb0 = (int)((long long)args.num_k_blocks * split / S);
    const int kb1 = (int)((long long)args.num_k_blocks * (split + 1) / S);
    const int nkb = kb1 - kb0;
    const int m_off = blockIdx.z * M_PAD;               // first activation row of this CTA
    const int m_rows = min(M_PAD, args.M - m_off);      // activation rows it computes (>= 1)
    const int live_cols = min(M_PAD, (m_rows + 31) / 32 * 32);   // accumulator columns in use
    const int own_lo = skinny_own_lo((int)rank, S);     // weight rows this CTA owns: [own_lo, own_hi)
    const int rpo = skinny_own_lo((int)rank + 1, S) - own_lo;

    // Producer step i: weights, activations and both scale blocks of k-block
    // kb0 + i into ring stage i % STAGES, all counted on that stage's full
    // barrier (the scale writers wait on it too). `part`: the whole step
    // (kStepAll), or split around the wait for the previous grid when the
    // weights' codes are not written by it -- the barrier armed and the
    // weights' codes first (kStepWeights), the rest after (kStepRest).
    auto produce = [&](int i, int part) -> bool {
        const int stage = i % STAGES;
        const uint32_t phase = (uint32_t)(i / STAGES) & 1u;
        if (part != kStepRest && !mbar_wait(empty0 + 8u * stage, phase ^ 1u, wd, abort_flag, 1))
            return false;
        const int kb = kb0 + i;
        const uint32_t sw = base + stage * T::STAGE_BYTES;
        const uint32_t sx = sw + T::W_BYTES;
        const uint32_t ssw = sx + T::X_BYTES;
        const uint32_t ssx = ssw + T::SFW_BYTES;
        const uint32_t fb = full0 + 8u * stage;
        const int rb0 = m_off / 128;                      // first 128-row scale block of the activations
        const int nchunks = min(T::SFX_CHUNKS, args.sfx_row_blocks - rb0);
        if (part != kStepRest) {
            mbar_arrive_expect_tx(fb, T::W_BYTES + T::X_BYTES + T::SF_BLOCK_BYTES * (1 + nchunks));
            if (part == kStepWeights) {
                tma_load_2d(sw, &tmW, fb, kb * T::ROW_BYTES, nt * T::BW);
                return true;
            }
        }
        const size_t cb = (size_t)kb * 4u;
        // weights' scales (row block nt), activations' scales (row blocks rb0..)
        bulk_load(ssw, args.sfb + ((size_t)nt * args.sf_col_blocks + cb) * 512u, T::SF_BLOCK_BYTES, fb);
        for (int c = 0; c < nchunks; ++c)
            bulk_load(ssx + c * T::SF_BLOCK_BYTES, args.sfa + ((size_t)(rb0 + c) * args.sf_col_blocks + cb) * 512u,
                      T::SF_BLOCK_BYTES, fb);
        if (part == kStepAll)
            tma_load_2d(sw, &tmW, fb, kb * T::ROW_BYTES, nt * T::BW);
        tma_load_2d(sx, &tmX, fb, kb * T::ROW_BYTES, m_off);
        return true;
    };

    const int first = min(STAGES, nkb);
    bool producing = true;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
            mbar_init(sfready0 + 8u * s, T::SCALE_WARPS);
        }
        mbar_init(tfull, 1);
        mbar_init(drain_bar, 1);
        mbar_init(peer_free, S > 1 ? (uint32_t)(S - 1) : 1u);
        mbar_init(rx, 1);
        *abort_flag = 0;
        fence_mbar_init();               // initialised barriers: visible to the TMA unit and the peers
        if (args.pdl == 2) {
            // the weights' codes are not written by the previous grid: the
            // first stages' codes into the ring while it finishes (warming
            // L2 with later k-blocks too measured slower when the previous
            // grid streams weights of its own); their scales may be written
            // by it (a scale swizzle launched just before), so they wait
            // with the activations
            int armed = 0;
            while (armed < first && producing)
                if ((producing = produce(armed, kStepWeights)))
                    ++armed;
            griddep_wait();
            for (int i = 0; i < armed; ++i)
                produce(i, kStepRest);
        } else {
            griddep_wait();              // a dependent launch: the previous grid's writes are visible
            for (int i = 0; i < first && producing; ++i)
                producing = produce(i, kStepAll);
        }
        griddep_launch_dependents();     // the whole grid is resident: the next launch may set up
        if (S > 1)                       // the peers' rows, pushed with complete_tx
            mbar_arrive_expect_tx(rx, (uint32_t)((S - 1) * rpo * live_cols * 4));
    }
    __syncwarp();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (S > 1)
        cluster_arrive_relaxed();        // this CTA's barriers are initialised
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0)
            for (int i = first; i < nkb && producing; ++i)
                producing = produce(i, kStepAll);
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
                if (!mbar_wait(full0 + 8u * stage, phase, wd, abort_flag, 3) ||
                    !mbar_wait(sfready0 + 8u * stage, phase, wd, abort_flag, 5)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sw = base + stage * T::STAGE_BYTES;
                const uint32_t sx = sw + T::W_BYTES;
                const uint32_t sfa_t = tmem + (uint32_t)(M_PAD + stage * T::SF_COLS);
                const uint32_t sfb_t = sfa_t + T::SFA_COLS;
#pragma unroll
                for (int j = 0; j < T::MMAS; ++j)
                    mma_nvfp4(tmem, desc_kmajor_sw128(sw + T::MMA_K_BYTES * j),
                              desc_kmajor_sw128(sx + T::MMA_K_BYTES * j), T::IDESC, sfa_t + 4u * j,
                              sfb_t + 4u * j * T::SFX_CHUNKS, (i | j) != 0 ? 1u : 0u);
                tc_commit(empty0 + 8u * stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok && nkb > 0)
                tc_commit(tfull);
            tc_commit(drain_bar);
            mbar_wait_quiet(drain_bar, 0, wd.limit_ns);
        }
    } else if (warp < T::EPI_WARP0) {
        // ------------------------------------------------------------------
        // Scale writers: weights' scales as the MMA's A-side scales,
        // activations' as its B-side scales
        // ------------------------------------------------------------------
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        for (int i = 0; i < nkb; ++i) {
            if (!warp_wait(full0 + 8u * stage, phase, wd, abort_flag, 6, lane))
                break;
            const uint32_t ssw = base + stage * T::STAGE_BYTES + T::W_BYTES + T::X_BYTES;
            const uint32_t sfa_t = tmem + lane_off + (uint32_t)(M_PAD + stage * T::SF_COLS);
            store_stage_scales<T::SFX_CHUNKS>(sfa_t, sfa_t + T::SFA_COLS, ssw, ssw + T::SFW_BYTES, lane);
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
    } else {
        // ------------------------------------------------------------------
        // Epilogue: TMEM lane n (warp q = n / 32) holds weight row n of the
        // tile, column m its dot product with activation row m_off + m.
        // Receive area of the owner of rows [lo, lo + rpo): FP32 [sender
        // rank][column / 4][row - lo][column % 4], one slot of rpo *
        // live_cols floats per rank.
        // ------------------------------------------------------------------
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int n = q * 32 + lane;
        const int owner = skinny_owner(n, S);
        const int o_lo = skinny_own_lo(owner, S);
        const int o_rpo = skinny_own_lo(owner + 1, S) - o_lo;
        const int orow = n - o_lo;                      // row within the owner's share
        const int et = threadIdx.x - 32 * T::EPI_WARP0; // 0 .. 127
        const float alpha = args.alpha;
        uint8_t *const recv = gbase + T::RECV_OFF;
        __nv_bfloat16 *const out = reinterpret_cast<__nv_bfloat16 *>(recv + T::RECV_BYTES);
        if constexpr (EPI) {
            griddep_wait();
            // the epilogue operands into shared memory while the MMAs run:
            // gamma and destination row (-1: not written) of every
            // activation row, bias of the owned weight rows
            for (int m = et; m < M_PAD; m += 32 * T::EPI_WARPS) {
                s_gamma[m] = epi_gamma(args, m_off + m);
                int d = m < m_rows ? m_off + m : -1;
                if (args.scatter && m < m_rows) {
                    d = __ldg(args.scatter + m_off + m);
                    d = (d >= 0 && d < args.m_out) ? d : -1;
                }
                s_dst[m] = d;
            }
            for (int r = et; r < rpo; r += 32 * T::EPI_WARPS)
                s_bias[r] = epi_bias(args, nt * T::BW + own_lo + r);
            named_bar_sync(1, 32 * T::EPI_WARPS);
        }
        const bool have = nkb > 0 && warp_wait(tfull, 0, wd, abort_flag, 4, lane);
        if (have)
            tc_fence_after_sync();
        if (S == 1) {
            if (have) {
#pragma unroll 1
                for (int c0 = 0; c0 < live_cols; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem + lane_off + (uint32_t)c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if constexpr (EPI)
                            out[(c0 + i) * T::BW + n] = __float2bfloat16_rn(
                                fmaf(__uint_as_float(v[i]), alpha, s_bias[n]) * s_gamma[c0 + i]);
                        else
                            out[(c0 + i) * T::BW + n] = __float2bfloat16_rn(__uint_as_float(v[i]) * alpha);
                    }
                }
            }
        } else {
            cluster_wait();              // every CTA of the cluster has initialised its barriers
            bool may_push = true;
            if (!T::OWN_RECV) {
                if (have && warp == T::EPI_WARP0 && lane == 0)
                    for (int p = 0; p < S; ++p)  // this CTA's ring is drained: peers may push into it
                        if (p != (int)rank)
                            mbar_arrive_remote_relaxed(mapa_shared(peer_free, (uint32_t)p));
                may_push = warp_wait(peer_free, 0, wd, abort_flag, 7, lane);
            }
            // every row of the partial into its owner's slot for this rank:
            // the owned rows locally, the others pushed to their CTA
            const int slot_bytes = o_rpo * live_cols * 4;
            const uint32_t group_bytes = (uint32_t)o_rpo * 16u;
            if (have && may_push) {
                const uint32_t my_slot = smem_u32(recv) + (uint32_t)((int)rank * slot_bytes) + (uint32_t)orow * 16u;
                const uint32_t dst = mapa_shared(my_slot, (uint32_t)owner);
                const uint32_t recv_bar = mapa_shared(rx, (uint32_t)owner);
                float4 *const local = reinterpret_cast<float4 *>(recv + (int)rank * slot_bytes + orow * 16);
#pragma unroll 1
                for (int c0 = 0; c0 < live_cols; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem + lane_off + (uint32_t)c0, v);
                    tmem_ld_wait();
                    if (owner == (int)rank) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            local[(c0 / 4 + j) * o_rpo] =
                                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_async_v4(dst + (uint32_t)(c0 / 4 + j) * group_bytes, v[4 * j], v[4 * j + 1],
                                        v[4 * j + 2], v[4 * j + 3], recv_bar);
                    }
                }
            }
            const bool rows_in = warp_wait(rx, 0, wd, abort_flag, 8, lane);
            named_bar_sync(1, 32 * T::EPI_WARPS);        // the owned rows' local writes
            if (have && rows_in)
                reduce_owned<EPI>(recv, out, S, rpo, live_cols, alpha, et, 32 * T::EPI_WARPS, s_gamma, s_bias);
        }
        // this CTA's [m_rows x rpo] block of D (columns nt * 128 + own_lo ..)
        // from the BF16 staging (row stride rpo), in 16-byte pieces:
        // consecutive threads take consecutive pieces of one row; a
        // scattered row goes to row scatter[m], a dropped one nowhere
        named_bar_sync(1, 32 * T::EPI_WARPS);
        if (have) {
            const int pieces = rpo / 8;
            const int col0 = nt * T::BW + own_lo;
            for (int p = et; p < m_rows * pieces; p += 32 * T::EPI_WARPS) {
                const int m = p / pieces;
                const int col = col0 + 8 * (p - m * pieces);
                int d = m_off + m;
                if constexpr (EPI)
                    d = s_dst[m];
                if (d >= 0 && col < args.N)
                    *reinterpret_cast<uint4 *>(args.d + (size_t)d * (size_t)args.N + (size_t)col) =
                        *reinterpret_cast<const uint4 *>(out + m * rpo + (col - col0));
            }
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Plans and launchers
// ---------------------------------------------------------------------------
template <int M_PAD, int STAGES>
static cudaError_t skinny_launch_impl(const GemmMaps &maps, const GemmArgs &args, int splits, int halves,
                                      cudaStream_t stream)
{
    using T = SkinnyTile<M_PAD, STAGES>;
    auto kern = has_epilogue(args) ? gemm_skinny_kernel<M_PAD, STAGES, true> : gemm_skinny_kernel<M_PAD, STAGES, false>;
    cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), T::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)args.num_n_tiles, (unsigned)splits, (unsigned)halves);
    cfg.blockDim = dim3(T::THREADS, 1, 1);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)splits;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = args.pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, maps.b, maps.a, args);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <int M_PAD, int STAGES>
static int skinny_clusters_impl(int splits)
{
    using T = SkinnyTile<M_PAD, STAGES>;
    auto kern = gemm_skinny_kernel<M_PAD, STAGES, false>;   // the EPI instantiation has the same footprint
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, (unsigned)splits, 1);
    cfg.blockDim = dim3(T::THREADS, 1, 1);
    cfg.dynamicSmemBytes = T::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)splits;
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

template <int M_PAD, int STAGES>
static constexpr PlanInfo make_skinny_plan(const char *name)
{
    using T = SkinnyTile<M_PAD, STAGES>;
    return PlanInfo{name, Kind::NVFP4, Family::SKINNY, 1, M_PAD, T::BW, STAGES, 1, T::K_BLOCK,
                    T::SMEM_BYTES, T::THREADS, T::TMEM_COLS, 0, T::SPLITS_MASK};
}

// activation rows covered per CTA, stages. Kernels that allocate tensor
// memory were measured to run one CTA per SM whatever their shared memory
// (the occupancy query gives 1 even for 32 threads and no shared memory),
// so the 3-stage plans differ from the deeper ones only in ring depth.
#define BSG_SKINNY_PLANS(X)                                   \
    X(64, 3, "nvfp4_skinny_m64_s3")                           \
    X(64, 6, "nvfp4_skinny_m64_s6")                           \
    X(128, 3, "nvfp4_skinny_m128_s3")                         \
    X(256, 4, "nvfp4_skinny_m256_s4")

#define BSG_SKINNY_INFO(MP, S, NAME) make_skinny_plan<MP, S>(NAME),
static const PlanInfo kSkinnyPlans[] = {BSG_SKINNY_PLANS(BSG_SKINNY_INFO)};
#undef BSG_SKINNY_INFO

int skinny_num_plans() { return (int)(sizeof(kSkinnyPlans) / sizeof(kSkinnyPlans[0])); }

const PlanInfo &skinny_plan(int i) { return kSkinnyPlans[i]; }

cudaError_t skinny_launch(int id, const GemmMaps &maps, const GemmArgs &args, int splits, int halves,
                          cudaStream_t stream)
{
    int i = 0;
#define BSG_SKINNY_LAUNCH(MP, S, NAME)                                          \
    if (id == i)                                                               \
        return skinny_launch_impl<MP, S>(maps, args, splits, halves, stream); \
    ++i;
    BSG_SKINNY_PLANS(BSG_SKINNY_LAUNCH)
#undef BSG_SKINNY_LAUNCH
    return cudaErrorInvalidValue;
}

int skinny_max_clusters(int id, int splits)
{
    int i = 0;
#define BSG_SKINNY_OCC(MP, S, NAME)                    \
    if (id == i)                                      \
        return skinny_clusters_impl<MP, S>(splits);    \
    ++i;
    BSG_SKINNY_PLANS(BSG_SKINNY_OCC)
#undef BSG_SKINNY_OCC
    return 0;
}

}  // namespace bsg
