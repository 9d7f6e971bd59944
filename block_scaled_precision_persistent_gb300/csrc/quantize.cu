// Two-level NVFP4 quantisation of a BF16 matrix: the step in front of the
// block-scaled GEMM ("Triton #11171 - Why Two New NVFP4 Test Cases Produced
// Twelve Tensor-Memory Failures" names a shared NVFP4 quantisation there).
//
//   amax  = max |x| over the tensor
//   s_g   = 2688 / amax (448 * 6; 1 if amax == 0)
//   per 16-element block along K, bmax = max |x|:
//     scale = E4M3 (round to nearest even, saturating at 448) of (bmax / 6) * s_g
//     code  = E2M1 (round to nearest even, saturating at 6) of (x * s_g) / scale,
//             0 for every element of a block whose scale is 0
//
// The codes are defined with every float operation rounded once, in this
// order, so they are a function of the inputs alone. The kernel computes them
// with approximate reciprocals and checks, per block and per 8 elements, that
// both ends of a band around the approximation round to the same code; only
// where a rounding threshold lies inside the band does it compute the exact
// quotients (__fdiv_rn / __fmul_rn). Two launches: a global-amax reduction
// (one HBM read of X), then the quantiser (second read of X, writes codes and
// scales). X is read with 16-byte loads.
//
// Outputs: codes packed two per byte along K (element 2i in the low nibble),
// block scales directly in the tcgen05 block-scale layout the GEMM reads
// (rows padded to 128, scale columns to 4, 512-byte blocks of 128 rows x 4
// scales, byte (r % 32) * 16 + (r / 32) * 4 + c inside a block, padding zero)
// and, optionally, row-major.
#include <cuda_bf16.h>

#include "bsg_internal.h"
#include "ptx.cuh"

namespace bsg {

namespace {

constexpr int kAmaxThreads = 256;
constexpr int kQThreads = 256;
constexpr int kQRows = 128;                 // rows per quantiser CTA (one swizzled row block)
constexpr int kQBlocks = 16;                // 16-element blocks per row per CTA (four 4-column groups)
constexpr int kQPitch = 5;                  // words per staged row of scales (4 + 1, bank spread)

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// max |x| of the 8 BF16 values in a 16-byte vector
__device__ __forceinline__ float absmax8(uint4 v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(bf16_bits_to_float(w[i] & 0xFFFFu)));
        m = fmaxf(m, fabsf(bf16_bits_to_float(w[i] >> 16)));
    }
    return m;
}

// E4M3 code (round to nearest even, saturating at the largest finite 448)
__device__ __forceinline__ uint32_t e4m3_code(float v)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

// E4M3 codes of two values: the common code if they agree, else 0x100
__device__ __forceinline__ uint32_t e4m3_code2(float a, float b)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(a), "f"(b));
    const uint32_t lo = r & 0xFFu, hi = (uint32_t)r >> 8;
    return lo == hi ? lo : 0x100u;
}

// (d0, d1) = (a0 * b, a1 * b), each rounded to nearest: one paired FP32
// multiply
__device__ __forceinline__ void mul2_rn(float a0, float a1, float b, float &d0, float &d1)
{
    asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
        "mov.b64 pa, {%2, %3};\n\t"
        "mov.b64 pb, {%4, %4};\n\t"
        "mul.rn.f32x2 pd, pa, pb;\n\t"
        "mov.b64 {%0, %1}, pd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b));
}

// approximate reciprocal (within one unit in the last place)
__device__ __forceinline__ float rcp_approx(float v)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// value of a non-negative finite E4M3 code (exponent bias 7, 3 mantissa bits)
__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0u)
        return (float)m * 0.001953125f;                        // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));    // (1 + m/8) * 2^(e-7)
}

// four bytes of two E2M1 codes each (round to nearest even, saturating at
// 6); element 2i is the low nibble of byte i
__device__ __forceinline__ uint32_t e2m1_pack8(const float (&y)[8])
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
    return r;
}

// Exact codes where the fast path's band straddles an E2M1 rounding threshold
// (about 0.5 % of elements on BF16 data: exact ties are common). c_lo / c_hi: the 8 codes (4 bytes, 2 per byte) of the band's ends. Where a
// nibble differs, the two codes are neighbours and the threshold between them
// is mid = (m + m') / 2 with at most 3 significant bits; scale sv has at most
// 4, so mid * sv is exact, and t = RN(x * s_g) lies within a factor 1 +- 2^-20
// of it, so fma(-mid, sv, t) = t - mid * sv exactly (Sterbenz). Then
//   RN(t / sv) == mid  <=>  -ulp_below(mid)/2 <= (t - mid*sv)/sv <= ulp(mid)/2
// (mid has an even last mantissa bit, so the half-way cases round to it), in
// which case the E2M1 tie goes to the code with the even mantissa; otherwise
// the sign of t - mid*sv picks the code. No division.
__device__ __forceinline__ uint32_t e2m1_fix8(uint32_t c_lo, uint32_t c_hi, uint32_t w0, uint32_t w1, uint32_t w2,
                                               uint32_t w3, float s_g, float sv)
{
    uint32_t out = c_lo;
    uint32_t diff = c_lo ^ c_hi;
    while (diff != 0u) {                                    // usually one nibble
        const int e = (__ffs(diff) - 1) >> 2;
        diff &= ~(15u << (4 * e));
        const uint32_t a = (c_lo >> (4 * e)) & 15u, b = (c_hi >> (4 * e)) & 15u;
        const uint32_t ma = a & 7u, mb = b & 7u;
        const uint32_t lo_mag = min(ma, mb), hi_mag = max(ma, mb);   // neighbours
        // midpoint between E2M1 magnitudes lo_mag and lo_mag + 1:
        // .25 .75 1.25 1.75 (step .5), then 2.5 3.5, then 5
        const float mid = lo_mag < 4u ? 0.25f + 0.5f * (float)lo_mag
                                      : (lo_mag < 6u ? (float)lo_mag - 1.5f : 5.0f);
        // its unit in the last place above (2^(exponent - 23)) and below
        // (half of that when mid is a power of two: only .25)
        const uint32_t mb_bits = __float_as_uint(mid);
        const float ulp_up = __uint_as_float((mb_bits & 0x7F800000u) - (23u << 23));
        const float ulp_dn = (mb_bits & 0x007FFFFFu) ? ulp_up : 0.5f * ulp_up;
        const int wi = e >> 1;                              // selected without indexing (no local memory)
        const uint32_t word = wi == 0 ? w0 : wi == 1 ? w1 : wi == 2 ? w2 : w3;
        const float x = (e & 1) ? __uint_as_float(word & 0xFFFF0000u) : bf16_bits_to_float(word & 0xFFFFu);
        const float t = fabsf(__fmul_rn(x, s_g));
        const float d = fmaf(-mid, sv, t);                  // exact: t - mid * sv
        uint32_t mag;
        if (d <= 0.5f * ulp_up * sv && d >= -0.5f * ulp_dn * sv)
            mag = (lo_mag & 1u) ? hi_mag : lo_mag;          // RN(t / sv) == mid: tie to the even code
        else
            mag = d > 0.0f ? hi_mag : lo_mag;
        out = (out & ~(15u << (4 * e))) | (((a & 8u) | mag) << (4 * e));
    }
    return out;
}

__global__ void __launch_bounds__(kAmaxThreads)
    amax_kernel(const uint4 *__restrict__ x, size_t n_vec, unsigned int *__restrict__ amax_bits)
{
    float m = 0.0f;
    const size_t stride = (size_t)gridDim.x * kAmaxThreads;
    size_t i = (size_t)blockIdx.x * kAmaxThreads + threadIdx.x;
    for (; i + 3 * stride < n_vec; i += 4 * stride) {        // four 16-byte loads in flight
        const uint4 a = __ldg(x + i), b = __ldg(x + i + stride);
        const uint4 c = __ldg(x + i + 2 * stride), d = __ldg(x + i + 3 * stride);
        m = fmaxf(m, fmaxf(fmaxf(absmax8(a), absmax8(b)), fmaxf(absmax8(c), absmax8(d))));
    }
    for (; i < n_vec; i += stride)
        m = fmaxf(m, absmax8(__ldg(x + i)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float wmax[kAmaxThreads / 32];
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = wmax[0];
        for (int w = 1; w < kAmaxThreads / 32; ++w)
            b = fmaxf(b, wmax[w]);
        atomicMax(amax_bits, __float_as_uint(b));           // b >= 0: bit order is value order
    }
}

// One CTA: rows [128 y, +128) x 16-element blocks [16 x, +16).
// tiles: codes go to the tile-packed layout (16 KiB tiles of 128 rows x 128
// bytes, tile index row_block * K/256 + k_block, 16-byte chunk c of row r at
// chunk c ^ (r % 8)), and rows past `rows` of the last row block are written
// as zero codes; otherwise row-major rows of K/2 bytes.
__global__ void __launch_bounds__(kQThreads)
    quantize_kernel(const __nv_bfloat16 *__restrict__ X, int rows, int K, uint8_t *__restrict__ packed,
                    uint8_t *__restrict__ sf_swz, uint8_t *__restrict__ sf_rm, float *__restrict__ global,
                    int tiles)
{
    __shared__ uint32_t tile[kQRows * kQPitch];
    uint8_t *t8 = reinterpret_cast<uint8_t *>(tile);
    const int nb = K / 16;                          // scale columns
    const int ncb = (nb + 3) / 4;                   // 4-column groups (swizzled layout)
    const float amax = global[0];
    const float s_g = amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
    const float sg6 = s_g * 0.16666667163372039794921875f;      // s_g * RN(1/6), for the fast scale path
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        global[1] = s_g;

#pragma unroll 2
    for (int i = 0; i < kQRows * kQBlocks / kQThreads; ++i) {
        const int idx = threadIdx.x + kQThreads * i;
        const int r = idx / kQBlocks, cl = idx % kQBlocks;          // 16 consecutive threads: one row
        const int row = blockIdx.y * kQRows + r, cb = blockIdx.x * kQBlocks + cl;
        uint32_t scode = 0u;
        // byte 8 cb of row `row` in the tile-packed layout (8 bytes stay in
        // one 16-byte chunk; 16 consecutive threads fill one 128-byte row of a tile)
        const size_t tile_off = tiles ? (((size_t)blockIdx.y * (size_t)(K / 256) + (size_t)(cb >> 4)) * 128u + r) *
                                                128u + (size_t)((((cb & 15) >> 1) ^ (r & 7)) << 4) + 8u * (cb & 1)
                                      : 0;
        if (tiles && row >= rows && cb < nb)
            *reinterpret_cast<uint2 *>(packed + tile_off) = make_uint2(0u, 0u);
        if (row < rows && cb < nb) {
            const uint4 *src = reinterpret_cast<const uint4 *>(X + (size_t)row * (size_t)K + 16 * (size_t)cb);
            const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            // bmax: max |x| on BF16 pairs (exact)
            __nv_bfloat162 m2 = __habs2(*reinterpret_cast<const __nv_bfloat162 *>(&w[0]));
#pragma unroll
            for (int j = 1; j < 8; ++j)
                m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162 *>(&w[j])));
            const float bmax = fmaxf(__low2float(m2), __high2float(m2));
            // scale = E4M3(RN(RN(bmax / 6) * s_g)). bmax * (s_g / 6) is within a
            // few units in the last place of that value; where the E4M3 codes of
            // the band around it (x (1 -+ 2^-20)) agree, they are the code (no
            // E4M3 rounding threshold lies inside the band); otherwise the
            // value is computed exactly.
            const float sc = bmax * sg6;
            scode = e4m3_code2(sc * 0.99999904632568359375f, sc * 1.00000095367431640625f);
            if (scode > 0xFFu)                  // rare: an E4M3 threshold lies within the band
                scode = e4m3_code(__fmul_rn(__fdiv_rn(bmax, 6.0f), s_g));
            const float sv = e4m3_value(scode);
            uint2 out = make_uint2(0u, 0u);
            if (sv > 0.0f) {
                // code_k = E2M1(RN(RN(x_k * s_g) / sv)). x_k * s_g * approx(1 / sv)
                // is within ~2^-21 (relative) of that quotient, so the band
                // x_k * k * (1 -+ 2^-20), k = s_g / sv, contains it. Where both
                // ends of the band convert to the same codes, no E2M1 rounding
                // threshold lies inside it and every value in it -- the exact
                // quotient included -- has those codes. Where they differ (a
                // threshold or tie is that close), the quotient is computed
                // exactly.
                const float k = s_g * rcp_approx(sv);
                const float k_lo = k * 0.99999904632568359375f;   // 1 - 2^-20
                const float k_hi = k * 1.00000095367431640625f;   // 1 + 2^-20
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float lo[8], hi[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float xa = bf16_bits_to_float(w[4 * h + j] & 0xFFFFu);
                        const float xb = __uint_as_float(w[4 * h + j] & 0xFFFF0000u);
                        mul2_rn(xa, xb, k_lo, lo[2 * j], lo[2 * j + 1]);
                        mul2_rn(xa, xb, k_hi, hi[2 * j], hi[2 * j + 1]);
                    }
                    uint32_t c = e2m1_pack8(lo);
                    const uint32_t ch = e2m1_pack8(hi);
                    if (c != ch)                      // a threshold lies within the band
                        c = e2m1_fix8(c, ch, w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3], s_g, sv);
                    (h == 0 ? out.x : out.y) = c;
                }
            }
            *reinterpret_cast<uint2 *>(packed + (tiles ? tile_off : (size_t)row * (size_t)(K / 2) + 8 * (size_t)cb)) =
                out;
            if (sf_rm)
                sf_rm[(size_t)row * (size_t)nb + cb] = (uint8_t)scode;
        }
        t8[r * (kQPitch * 4) + cl] = (uint8_t)scode;              // zero for padding rows / columns
    }
    __syncthreads();

    // four 512-byte blocks of the swizzled layout: line l of group g holds
    // the 4-scale words of rows l, l+32, l+64, l+96
    const int g = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int cg = blockIdx.x * (kQBlocks / 4) + g;
    if (threadIdx.x < 4 * 32 && cg < ncb) {
        uint4 v;
        v.x = tile[(l + 0) * kQPitch + g];
        v.y = tile[(l + 32) * kQPitch + g];
        v.z = tile[(l + 64) * kQPitch + g];
        v.w = tile[(l + 96) * kQPitch + g];
        reinterpret_cast<uint4 *>(sf_swz + ((size_t)blockIdx.y * (size_t)ncb + (size_t)cg) * 512u)[l] = v;
    }
}

}  // namespace

cudaError_t launch_nvfp4_quantize(int rows, int K, const void *X, uint8_t *packed, uint8_t *sf_swz,
                                  uint8_t *sf_rm, float *global, int num_sms, cudaStream_t stream, bool tiles)
{
    cudaError_t e = cudaMemsetAsync(global, 0, sizeof(float), stream);
    if (e != cudaSuccess)
        return e;
    const size_t n_vec = (size_t)rows * (size_t)K / 8;        // 16-byte vectors of 8 BF16
    size_t blocks = (n_vec + kAmaxThreads - 1) / kAmaxThreads;
    const size_t cap = (size_t)num_sms * 8;
    if (blocks > cap)
        blocks = cap;
    amax_kernel<<<(unsigned)blocks, kAmaxThreads, 0, stream>>>(static_cast<const uint4 *>(X), n_vec,
                                                                reinterpret_cast<unsigned int *>(global));
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    const int nb = K / 16;
    dim3 grid((unsigned)((nb + kQBlocks - 1) / kQBlocks), (unsigned)((rows + kQRows - 1) / kQRows));
    quantize_kernel<<<grid, kQThreads, 0, stream>>>(static_cast<const __nv_bfloat16 *>(X), rows, K, packed,
                                                     sf_swz, sf_rm, global, tiles ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace bsg
