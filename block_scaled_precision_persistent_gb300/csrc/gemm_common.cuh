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
__device__ __forceinline__ void raster_tile(int tile, int raster_group, int num_m_tiles, int num_n_tiles, int &mt,
                                            int &nt)
{
    const int per_group = raster_group * num_n_tiles;
    const int g = tile / per_group;
    const int first_m = g * raster_group;
    const int gm = min(raster_group, num_m_tiles - first_m);
    const int local = tile - g * per_group;
    mt = first_m + local % gm;
    nt = local / gm;
}

__device__ __forceinline__ void raster_tile(int tile, const GemmArgs &a, int &mt, int &nt)
{
    raster_tile(tile, a.raster_group, a.num_m_tiles, a.num_n_tiles, mt, nt);
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

// ---------------------------------------------------------------------------
// Epilogue variants ("Triton #11171 - Why Two New NVFP4 Test Cases Produced
// Twelve Tensor-Memory Failures", sections on scatter, gamma and the shared
// bias route): D[dst(m)][n] = bf16(gamma[m] * (alpha * acc[m][n] + bias[n])).
// ---------------------------------------------------------------------------

// Per-row operands of computed row `row`: gamma (1 without one) and the row
// of D it is written to (-1: none -- a row at or past row_end (M, or the end
// of a grouped GEMM's slice), or a scatter index outside [0, m_out)).
struct RowEpi {
    float gamma;
    int dst;
};

__device__ __forceinline__ RowEpi load_row_epi(const GemmArgs &a, int row, int row_end)
{
    RowEpi e{1.0f, -1};
    if (row < row_end) {
        if (a.gamma)
            e.gamma = __ldg(a.gamma + row);
        e.dst = row;
        if (a.scatter) {
            const int d = __ldg(a.scatter + row);
            e.dst = (d >= 0 && d < a.m_out) ? d : -1;
        }
    }
    return e;
}

// Bias of output column n (-0 without one, or past N: adding -0 changes
// nothing) and gamma of output row m (1 without one, or past M).
__device__ __forceinline__ float epi_bias(const GemmArgs &a, int n)
{
    return (a.bias && n < a.N) ? __ldg(a.bias + n) : -0.0f;
}

__device__ __forceinline__ float epi_gamma(const GemmArgs &a, int m)
{
    return (a.gamma && m < a.M) ? __ldg(a.gamma + m) : 1.0f;
}

// The bias of columns [x0, x0 + ncols) into L1, 64 bytes per lane, issued
// before the accumulator wait: the epilogue's bias loads then hit L1 instead
// of waiting on L2 between the TMEM read and the TMEM release.
__device__ __forceinline__ void prefetch_bias(const float *bias, int N, int x0, int ncols, int lane)
{
    const int c = x0 + 16 * lane;
    if (bias && 16 * lane < ncols && c < N)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(bias + c));
}

// Bias of columns [col, col + 32) as 8 float4. bias + col is 16-byte
// aligned (bias is, col is a multiple of 32); every lane reads the same 128
// bytes. FULL: all 32 columns are below N (unconditional loads); otherwise
// columns at or past N read as -0 (never stored).
template <bool FULL>
__device__ __forceinline__ void load_bias32(const float *bias, int col, int N, float4 (&b)[8])
{
    const float4 *p = reinterpret_cast<const float4 *>(bias + col);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (FULL || col + 4 * j < N)
            b[j] = __ldg(p + j);
        else
            b[j] = make_float4(-0.0f, -0.0f, -0.0f, -0.0f);
    }
}

// 32 accumulator columns of one row -> 16 BF16 pairs of
// bf16(fma(acc, scale, bias[c]) * g), the multiply only with a gamma.
template <bool GAMMA>
__device__ __forceinline__ void convert32_bias(const uint32_t (&v)[32], uint32_t *pk, float scale, float g,
                                               const float4 (&b)[8])
{
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float x0 = fmaf(__uint_as_float(v[4 * j]), scale, b[j].x);
        float x1 = fmaf(__uint_as_float(v[4 * j + 1]), scale, b[j].y);
        float x2 = fmaf(__uint_as_float(v[4 * j + 2]), scale, b[j].z);
        float x3 = fmaf(__uint_as_float(v[4 * j + 3]), scale, b[j].w);
        if (GAMMA) {
            x0 *= g;
            x1 *= g;
            x2 *= g;
            x3 *= g;
        }
        pk[2 * j] = pack_bf16x2(x0, x1);
        pk[2 * j + 1] = pack_bf16x2(x2, x3);
    }
}

// 32 accumulator columns of one row -> 16 BF16 pairs of bf16(acc * scale).
__device__ __forceinline__ void convert32(const uint32_t (&v)[32], uint32_t *pk, float scale)
{
#pragma unroll
    for (int i = 0; i < 16; ++i)
        pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
}

// The epilogue-variant conversion of 64 accumulator columns of one row (two
// 32-column reads) starting at output column x; bias is the row's bias
// vector (a grouped GEMM's slice's), or null. Each case takes as few
// instructions per element as it can, on uniform branches:
//   no bias:  bf16(acc * (scale * gamma))           (gamma folded into the
//             row's scale: one multiply, as the plain epilogue)
//   bias:     bf16(fma(acc, scale, bias[c]) [* gamma])
// The FP32 evaluation order is the kernel's; it differs from the exact
// gamma * (alpha * acc + bias) only by FP32 rounding before the BF16 one.
__device__ __forceinline__ void convert64_epi(const uint32_t (&v0)[32], const uint32_t (&v1)[32], uint32_t (&pk)[32],
                                              float scale, const RowEpi &re, const GemmArgs &a, const float *bias,
                                              int x)
{
    if (!bias) {
        const float sg = scale * re.gamma;
        convert32(v0, pk, sg);
        convert32(v1, pk + 16, sg);
        return;
    }
    float4 b[8];
    const bool full = x + 64 <= a.N;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t(&v)[32] = h ? v1 : v0;
        if (full)
            load_bias32<true>(bias, x + 32 * h, a.N, b);
        else
            load_bias32<false>(bias, x + 32 * h, a.N, b);
        if (a.gamma)
            convert32_bias<true>(v, pk + 16 * h, scale, re.gamma, b);
        else
            convert32_bias<false>(v, pk + 16 * h, scale, 1.0f, b);
    }
}

// Scattered store of a warp's 32-row x 64-column BF16 chunk, staged with the
// 128-byte swizzle (row r's 16-byte piece c at r * 128 + ((c ^ (r % 8)) * 16)
// of sbuf) for columns [x, x + 64) of D. Four rows per step: each group of
// eight lanes reads one row's 128 bytes (conflict-free) and writes them to
// row dst(r) of D, so every group's store is one contiguous 128-byte run.
// `dst` is the calling lane's own row destination (-1: not written). Columns
// at or past N are skipped 8 at a time (N % 8 == 0).
__device__ __forceinline__ void scatter_chunk(const uint8_t *sbuf, int dst, uint16_t *D, int N, int x, int lane)
{
    const int c = lane & 7;
    const int col = x + 8 * c;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = 4 * it + (lane >> 3);
        const int d = __shfl_sync(0xffffffffu, dst, r);
        const uint4 val = *reinterpret_cast<const uint4 *>(sbuf + r * 128 + ((c ^ (r & 7)) << 4));
        if (d >= 0 && col < N)
            *reinterpret_cast<uint4 *>(D + (size_t)d * (size_t)N + (size_t)col) = val;
    }
}

// ---------------------------------------------------------------------------
// NVFP4 -> BF16 expansion: the A operand of the NVFP4 x dense-BF16 GEMM. An
// E2M1 value (at most 2 significant bits, |x| <= 6) times its E4M3 scale (at
// most 4 significant bits, 2^-9 .. 448) has at most 6 significant bits and
// lies in BF16's normal range, so the expanded operand is exact and the
// BF16 MMA computes the definition up to the FP32 accumulation order.
// ---------------------------------------------------------------------------

// Four E2M1 codes (nibbles 0..3 of x, x < 2^16, in element order) -> four
// BF16 values: elements 0, 1 in w01 and 2, 3 in w23 (low half first). The
// magnitudes 0 .5 1 1.5 2 3 4 6 are BF16 0x0000 0x3F00 0x3F80 0x3FC0 0x4000
// 0x4040 0x4080 0x40C0; byte permutes pick their low and high bytes by the
// code's three magnitude bits and a second pair interleaves them. The codes'
// sign bits (bits 3, 7, 11, 15 of x) are bit 7 of bytes 0, 1 of x << 4 and of
// x, so one more permute per word moves them to bits 15 and 31.
__device__ __forceinline__ void e2m1x4_to_bf16(uint32_t x, uint32_t &w01, uint32_t &w23)
{
    const uint32_t sel = x & 0x7777u;
    const uint32_t x4 = x << 4;
    uint32_t lo, hi, s01, s23;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0xC0800000u), "r"(0xC0804000u), "r"(sel));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x3F3F3F00u), "r"(0x40404040u), "r"(sel));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(w01) : "r"(lo), "r"(hi), "r"(0x5140u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(w23) : "r"(lo), "r"(hi), "r"(0x7362u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s01) : "r"(x), "r"(x4), "r"(0x0040u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s23) : "r"(x), "r"(x4), "r"(0x1050u));
    w01 |= s01 & 0x80008000u;
    w23 |= s23 & 0x80008000u;
}

// An E4M3 scale code (sign bit ignored: scales are unsigned) -> its BF16
// value in both halves. Normal codes map exponent e to e + 120 with the
// three mantissa bits on top; subnormals are m * 2^-9.
__device__ __forceinline__ uint32_t e4m3_to_bf16x2(uint32_t code)
{
    const uint32_t e = (code >> 3) & 15u, m = code & 7u;
    const float f = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0x1p-9f;
    const uint32_t b = __float_as_uint(f) >> 16;
    return b | (b << 16);
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// One row of a 64-element stage: 32 packed bytes of E2M1 codes at src
// (16-byte aligned; element 2i in the low nibble of byte i) and the row's
// four block scales (byte b of sc scales elements 16b..16b+15) -> 64 BF16 as
// 32 words, element 2w in the low half of word w.
__device__ __forceinline__ void expand_row_nvfp4_bf16(const uint8_t *src, uint32_t sc, uint32_t (&w)[32])
{
    const uint4 p0 = *reinterpret_cast<const uint4 *>(src);
    const uint4 p1 = *reinterpret_cast<const uint4 *>(src + 16);
    const uint32_t words[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t s2 = e4m3_to_bf16x2((sc >> (8 * (c >> 1))) & 0xFFu);
        uint32_t w0, w1, w2, w3;
        e2m1x4_to_bf16(words[c] & 0xFFFFu, w0, w1);
        e2m1x4_to_bf16(words[c] >> 16, w2, w3);
        w[4 * c] = mul_bf16x2(w0, s2);
        w[4 * c + 1] = mul_bf16x2(w1, s2);
        w[4 * c + 2] = mul_bf16x2(w2, s2);
        w[4 * c + 3] = mul_bf16x2(w3, s2);
    }
}

// Half a row: elements [32 hc, 32 hc + 32) of the stage's 64 (16 packed
// bytes at src + 16 hc, scale bytes 2 hc and 2 hc + 1 of sc) -> 16 words,
// element 2w in the low half of word w. The dense kernels give each half to
// its own warp, so that the expansion's latency per stage is halved.
__device__ __forceinline__ void expand_half_row_nvfp4_bf16(const uint8_t *src, uint32_t sc, int hc,
                                                           uint32_t (&w)[16])
{
    const uint4 p = *reinterpret_cast<const uint4 *>(src + 16 * hc);
    const uint32_t words[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t s2 = e4m3_to_bf16x2((sc >> (8 * (2 * hc + (c >> 1)))) & 0xFFu);
        uint32_t w0, w1, w2, w3;
        e2m1x4_to_bf16(words[c] & 0xFFFFu, w0, w1);
        e2m1x4_to_bf16(words[c] >> 16, w2, w3);
        w[4 * c] = mul_bf16x2(w0, s2);
        w[4 * c + 1] = mul_bf16x2(w1, s2);
        w[4 * c + 2] = mul_bf16x2(w2, s2);
        w[4 * c + 3] = mul_bf16x2(w3, s2);
    }
}

// Chunks [4 hc, 4 hc + 4) of row r (expanded half hc) into a 128B-swizzled
// K-major tile at shared address tile (see store_row_sw128).
__device__ __forceinline__ void store_half_row_sw128(const uint32_t (&w)[16], uint32_t tile, int r, int hc)
{
    const uint32_t row = tile + (uint32_t)r * 128u;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        st_shared_v4(row + ((uint32_t)((4 * hc + c) ^ (r & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                     w[4 * c + 3]);
}

// The expanded row r into a 128B-swizzled K-major tile at shared address
// tile: 16-byte chunk c (elements 8c..8c+7) at r * 128 + ((c ^ (r % 8)) *
// 16), the layout the MMA's shared-memory descriptor reads.
__device__ __forceinline__ void store_row_sw128(const uint32_t (&w)[32], uint32_t tile, int r)
{
    const uint32_t row = tile + (uint32_t)r * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        st_shared_v4(row + ((uint32_t)(c ^ (r & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
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
