// Device helpers shared by the 1-SM and CTA-pair persistent GEMM kernels.
#pragma once

#include <cuda_bf16.h>

#include "bsg_internal.h"
#include "ptx.cuh"

namespace bsg {

// Tile id -> (m tile, n tile): groups of `raster_group` M tiles; inside a
// group the M tile varies fastest, so the CTAs resident at one time share a
// few A panels and a band of B panels in L2 ("Building the GEMM": tile
// rasterisation order permuted for memory locality).
__device__ __forceinline__ void raster_tile(int tile, const GemmArgs &a, int &mt, int &nt)
{
    const int per_group = a.raster_group * a.num_n_tiles;
    const int g = tile / per_group;
    const int first_m = g * a.raster_group;
    const int gm = min(a.raster_group, a.num_m_tiles - first_m);
    const int local = tile - g * per_group;
    mt = first_m + local % gm;
    nt = local / gm;
}

// Bounded wait with no status side effect, used only while draining.
__device__ __forceinline__ void mbar_wait_quiet(uint32_t bar, uint32_t parity,
                                                unsigned long long limit_ns)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > limit_ns)
            return;
}

// Lane 0 waits (bounded) and the verdict is broadcast, so the warp stays
// converged for the .sync.aligned tcgen05 instructions that follow. The other
// lanes are ordered after lane 0's acquiring wait by the warp barrier; they do
// not poll the mbarrier themselves (a per-lane poll that starts by reading
// the global timer was measured to add hundreds of cycles per wait, which on
// the scale writers' path cost the pair kernel ~10 %).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Watchdog &wd,
                                          volatile int *abort_flag, uint32_t site, int lane)
{
    int ok = 0;
    if (lane == 0)
        ok = mbar_wait(bar, parity, wd, abort_flag, site) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Writes one ring stage's NVFP4 block scales from shared memory into the
// calling warp's TMEM sub-partition (taddr carries the warp's lane base).
// The layout is the one the tensor core reads for a 128-row operand with one
// scale per 16 elements: for each 512-byte block of the tcgen05 scale layout
// (128 rows x 4 scales), lane r of every sub-partition holds the block's
// 16-byte line r -- rows r, r+32, r+64, r+96 -- in 4 consecutive columns.
// A stage holds 4 blocks of A's scales (16 columns at sfa) and 4 blocks per
// 128 rows of B's scales (16 * SFB_CHUNKS columns at sfb, K step major).
// Every one of the four sub-partitions needs its own copy, so four warps (one
// per sub-partition) each run this for every stage.
template <int SFB_CHUNKS>
__device__ __forceinline__ void store_stage_scales(uint32_t taddr_sfa, uint32_t taddr_sfb,
                                                   uint32_t ssfa, uint32_t ssfb, int lane)
{
    uint32_t a[16];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        ld_shared_v4(ssfa + 512u * j + 16u * lane, a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
    tmem_st_32x32b_x16(taddr_sfa, a);
    if constexpr (SFB_CHUNKS == 2) {
        uint32_t b[32];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int i = 4 * (2 * j + c);
                ld_shared_v4(ssfb + 2048u * c + 512u * j + 16u * lane, b[i], b[i + 1], b[i + 2], b[i + 3]);
            }
        tmem_st_32x32b_x32(taddr_sfb, b);
    } else {
        static_assert(SFB_CHUNKS == 1, "B tiles of 128 or 256 rows");
        uint32_t b[16];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            ld_shared_v4(ssfb + 512u * j + 16u * lane, b[4 * j], b[4 * j + 1], b[4 * j + 2], b[4 * j + 3]);
        tmem_st_32x32b_x16(taddr_sfb, b);
    }
}

}  // namespace bsg
