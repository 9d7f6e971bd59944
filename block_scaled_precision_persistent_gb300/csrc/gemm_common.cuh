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

// k-blocks of the first tile's B that a 1-SM dependent launch whose B is not
// written by the previous kernel (GemmArgs::pdl == 2) warms in L2 before it
// waits for that kernel.
constexpr int kEarlyKBlocks = 8;

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
// NVFP4 -> BF16 / FP16 expansion: the A operand of the NVFP4 x dense GEMM.
// An E2M1 value (at most 2 significant bits, |x| <= 6) times its E4M3 scale
// (at most 4 significant bits, 2^-9 .. 448) has at most 6 significant bits
// and lies in the normal range of BF16 and of FP16, so the expanded operand
// is exact and the 16-bit MMA computes the definition up to the FP32
// accumulation order.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The sign bits of eight E2M1 codes (bits 3, 7, ..., 31 of x) at bits 15 and
// 31 of the four output words: sign bit 8i + 3 is bit 7 of byte i of x << 4,
// sign bit 8i + 7 bit 7 of byte i of x, so one byte permute per word moves
// them (the other bits are cleared by the caller's mask).
__device__ __forceinline__ void e2m1x8_signs(uint32_t x, uint32_t (&s)[4])
{
    const uint32_t x4 = x << 4;
    s[0] = prmt(x, x4, 0x0040u);
    s[1] = prmt(x, x4, 0x1050u);
    s[2] = prmt(x, x4, 0x2060u);
    s[3] = prmt(x, x4, 0x3070u);
}

// Eight E2M1 codes (nibble i of x is element i) -> eight BF16 values in four
// words, element 2w in the low half of word w. The magnitudes 0 .5 1 1.5 2 3
// 4 6 are BF16 0x0000 0x3F00 0x3F80 0x3FC0 0x4000 0x4040 0x4080 0x40C0; byte
// permutes pick their low and high bytes by the code's three magnitude bits
// (the selector nibbles; bit 3 of each is cleared, as it would select sign
// replication) and a second pair interleaves them.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t x, uint32_t (&w)[4])
{
    const uint32_t sel_lo = x & 0x7777u, sel_hi = (x >> 16) & 0x7777u;
    uint32_t s[4];
    e2m1x8_signs(x, s);
    const uint32_t lo_a = prmt(0xC0800000u, 0xC0804000u, sel_lo);
    const uint32_t hi_a = prmt(0x3F3F3F00u, 0x40404040u, sel_lo);
    const uint32_t lo_b = prmt(0xC0800000u, 0xC0804000u, sel_hi);
    const uint32_t hi_b = prmt(0x3F3F3F00u, 0x40404040u, sel_hi);
    w[0] = prmt(lo_a, hi_a, 0x5140u) | (s[0] & 0x80008000u);
    w[1] = prmt(lo_a, hi_a, 0x7362u) | (s[1] & 0x80008000u);
    w[2] = prmt(lo_b, hi_b, 0x5140u) | (s[2] & 0x80008000u);
    w[3] = prmt(lo_b, hi_b, 0x7362u) | (s[3] & 0x80008000u);
}

// Eight E2M1 codes -> eight FP16 values, laid out as e2m1x8_to_bf16. In FP16
// every magnitude (0x0000 0x3800 0x3C00 0x3E00 0x4000 0x4200 0x4400 0x4600)
// has a zero low byte, so one permute picks four high bytes and two more
// spread them into the halves.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t x, uint32_t (&w)[4])
{
    const uint32_t sel_lo = x & 0x7777u, sel_hi = (x >> 16) & 0x7777u;
    uint32_t s[4];
    e2m1x8_signs(x, s);
    const uint32_t hb_a = prmt(0x3E3C3800u, 0x46444240u, sel_lo);
    const uint32_t hb_b = prmt(0x3E3C3800u, 0x46444240u, sel_hi);
    w[0] = prmt(hb_a, 0u, 0x1404u) | (s[0] & 0x80008000u);
    w[1] = prmt(hb_a, 0u, 0x3424u) | (s[1] & 0x80008000u);
    w[2] = prmt(hb_b, 0u, 0x1404u) | (s[2] & 0x80008000u);
    w[3] = prmt(hb_b, 0u, 0x3424u) | (s[3] & 0x80008000u);
}

// Two E4M3 scale codes (bytes 0 and 1 of pair; sign bits ignored, scales are
// unsigned) -> their FP16 values, each broadcast to both halves of a word.
// Every E4M3 value is an FP16 value, so the hardware conversion is exact.
__device__ __forceinline__ void e4m3x2_to_f16x2(uint32_t pair, uint32_t &s0, uint32_t &s1)
{
    const uint16_t p = (uint16_t)(pair & 0x7F7Fu);
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(p));
    s0 = prmt(h, 0u, 0x1010u);
    s1 = prmt(h, 0u, 0x3232u);
}

// The same to BF16: E4M3 -> FP16 -> FP32 -> BF16, each step exact (an E4M3
// value has at most 4 significant bits and lies within every one of these
// types' normal range).
__device__ __forceinline__ void e4m3x2_to_bf16x2(uint32_t pair, uint32_t &s0, uint32_t &s1)
{
    const uint16_t p = (uint16_t)(pair & 0x7F7Fu);
    uint32_t h, b;
    float f0, f1;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(p));
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tcvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(f0), "=f"(f1)
        : "r"(h));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(b) : "f"(f1), "f"(f0));   // f1 to the upper half
    s0 = prmt(b, 0u, 0x1010u);
    s1 = prmt(b, 0u, 0x3232u);
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Half a row: elements [32 hc, 32 hc + 32) of the stage's 64 (16 packed
// bytes at src + 16 hc, scale bytes 2 hc and 2 hc + 1 of sc) -> 16 words of
// BF16 (F16 = false) or FP16 (F16 = true) pairs, element 2w in the low half
// of word w. Either product is exact: at most 6 significant bits, between
// 2^-10 and 2688 in magnitude. The dense kernels give each half to its own
// warp, so that the expansion's latency per stage is halved.
template <bool F16>
__device__ __forceinline__ void expand_half_row_nvfp4(const uint8_t *src, uint32_t sc, int hc, uint32_t (&w)[16])
{
    const uint4 p = *reinterpret_cast<const uint4 *>(src + 16 * hc);
    const uint32_t words[4] = {p.x, p.y, p.z, p.w};
    uint32_t s2[2];
    if constexpr (F16)
        e4m3x2_to_f16x2(sc >> (16 * hc), s2[0], s2[1]);
    else
        e4m3x2_to_bf16x2(sc >> (16 * hc), s2[0], s2[1]);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t v[4];
        if constexpr (F16)
            e2m1x8_to_f16(words[c], v);
        else
            e2m1x8_to_bf16(words[c], v);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[4 * c + i] = F16 ? mul_f16x2(v[i], s2[c >> 1]) : mul_bf16x2(v[i], s2[c >> 1]);
    }
}

// Chunks [4 hc, 4 hc + 4) of row r (expanded half hc) into a 128B-swizzled
// K-major tile at shared address tile: 16-byte chunk c (elements 8c..8c+7)
// of row r at r * 128 + ((c ^ (r % 8)) * 16), the layout the MMA's
// shared-memory descriptor reads.
__device__ __forceinline__ void store_half_row_sw128(const uint32_t (&w)[16], uint32_t tile, int r, int hc)
{
    const uint32_t row = tile + (uint32_t)r * 128u;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        st_shared_v4(row + ((uint32_t)((4 * hc + c) ^ (r & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                     w[4 * c + 3]);
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
