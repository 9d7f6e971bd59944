// Scale-layout prep: row-major E4M3 block scales uint8[rows][K/16] -> the
// tcgen05 block-scale layout that the persistent GEMM copies straight into
// shared memory with one bulk copy per 128 rows x 16 scales.
//
// "Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
// Failures", "Activation-scale swizzling forced the relevant persistent path":
// the persistent Blackwell kernel consumes scales rewritten in HBM into a
// Blackwell-specific layout. Layout (public PTX ISA, tcgen05 block scaling):
// rows padded to 128, scale columns padded to 4; 128x4 blocks of 512 bytes,
// row-block-major with the column block fastest; inside a block row r and
// column c go to byte (r%32)*16 + (r/32)*4 + c. Padding is zero.
//
// Each output 16-byte line holds the 4-byte column-block word of rows r0,
// r0+32, r0+64, r0+96, so the kernel is a permutation of 32-bit words: a CTA
// stages 128 rows x 128 scale columns in shared memory with coalesced reads
// (four 16-byte loads in flight per thread) and writes 32 contiguous
// 512-byte blocks. HBM-bound; bytes in = bytes out.
#include "bsg_internal.h"
#include "group.cuh"
#include "ptx.cuh"

namespace bsg {

constexpr int kSwzBlocksPerCta = 32;        // 4-column blocks per CTA (128 scale columns)
constexpr int kSwzThreads = 256;
constexpr int kSwzPitchWords = kSwzBlocksPerCta + 1;   // words per staged row + 1 (bank spread)

// GROUPED: the rows are E slices (offs, device); slice e is swizzled on its
// own from block row sb[e] on (group.cuh), and block rows past the slices'
// (grid y covers ceil(rows / 128) + E) are written as zeros.
// Two operands of the same K in one launch (not GROUPED): grid rows
// y >= nrb1 swizzle the second one (in2 -> out2, rows2 rows) from its block
// row y - nrb1.
template <bool GROUPED>
__global__ void __launch_bounds__(kSwzThreads)
    swizzle_scales_kernel(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int rows,
                          int cols, int ncb, int vec16, const int *offs, int E,
                          const uint8_t *__restrict__ in2, uint8_t *__restrict__ out2, int rows2, int nrb1)
{
    __shared__ uint32_t tile[128 * kSwzPitchWords];
    uint8_t *t8 = reinterpret_cast<uint8_t *>(tile);
    int rb = blockIdx.y;
    if (!GROUPED && rb >= nrb1) {
        rb -= nrb1;
        in = in2;
        out = out2;
        rows = rows2;
    }
    const int cb0 = blockIdx.x * kSwzBlocksPerCta;
    const int c0 = cb0 * 4;
    constexpr int span = kSwzBlocksPerCta * 4;   // 128 scale columns
    int row0 = rb * 128, row_end = rows;    // source rows of this block row: [row0, row_end)
    (void)E;
    if constexpr (GROUPED) {
        __shared__ int so[kMaxGroups + 1], sb[kMaxGroups + 1];
        if (threadIdx.x < 32)
            build_group_table(offs, E, rows, so, sb, threadIdx.x);
        __syncthreads();
        if (rb < sb[E]) {
            const int e = group_of_block(sb, E, rb);
            row0 = so[e] + (rb - sb[e]) * 128;
            row_end = so[e + 1];
        } else {
            row0 = row_end = 0;             // past the slices: zeros
        }
    }

    if (vec16) {
        // 16-byte loads (host-checked: 16-byte aligned base, cols % 16 == 0):
        // a 16-column segment of a row is then either wholly inside or wholly
        // past the matrix
        constexpr int kLoads = 128 * (span / 16) / kSwzThreads;   // 16-byte loads per thread
        static_assert(kLoads * kSwzThreads == 128 * (span / 16), "whole loads per thread");
        uint4 v[kLoads];
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {       // all loads in flight before the first shared store
            const int i = threadIdx.x + j * kSwzThreads;
            const int row = row0 + i / (span / 16), col = c0 + 16 * (i % (span / 16));
            v[j] = make_uint4(0u, 0u, 0u, 0u);
            if (row < row_end && col < cols)
                v[j] = __ldg(reinterpret_cast<const uint4 *>(in + (size_t)row * (size_t)cols + (size_t)col));
        }
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
            const int i = threadIdx.x + j * kSwzThreads;
            uint32_t *w = tile + (i / (span / 16)) * kSwzPitchWords + 4 * (i % (span / 16));
            w[0] = v[j].x;
            w[1] = v[j].y;
            w[2] = v[j].z;
            w[3] = v[j].w;
        }
    } else {
        for (int i = threadIdx.x; i < 128 * span; i += kSwzThreads) {
            const int r = i / span, b = i % span;
            const int row = row0 + r, col = c0 + b;
            uint8_t v = 0;
            if (row < row_end && col < cols)
                v = in[(size_t)row * (size_t)cols + (size_t)col];
            t8[r * (kSwzPitchWords * 4) + b] = v;
        }
    }
    __syncthreads();

    const int nblk = min(kSwzBlocksPerCta, ncb - cb0);
    for (int i = threadIdx.x; i < nblk * 32; i += kSwzThreads) {
        const int blk = i >> 5, r0 = i & 31;
        uint4 v;
        v.x = tile[(r0 + 0) * kSwzPitchWords + blk];
        v.y = tile[(r0 + 32) * kSwzPitchWords + blk];
        v.z = tile[(r0 + 64) * kSwzPitchWords + blk];
        v.w = tile[(r0 + 96) * kSwzPitchWords + blk];
        uint4 *dst = reinterpret_cast<uint4 *>(out + ((size_t)rb * (size_t)ncb + (size_t)(cb0 + blk)) * 512u);
        dst[r0] = v;
    }
}

cudaError_t launch_swizzle_scales(int rows, int K, const uint8_t *sf, uint8_t *out,
                                  cudaStream_t stream)
{
    const int cols = K / 16;
    const int ncb = (cols + 3) / 4;
    const int nrb = (rows + 127) / 128;
    dim3 grid((ncb + kSwzBlocksPerCta - 1) / kSwzBlocksPerCta, nrb);
    const int vec16 = (cols % 16) == 0 && (reinterpret_cast<uintptr_t>(sf) & 15u) == 0;
    swizzle_scales_kernel<false><<<grid, kSwzThreads, 0, stream>>>(sf, out, rows, cols, ncb, vec16, nullptr, 0,
                                                                   nullptr, nullptr, 0, nrb);
    return cudaGetLastError();
}

cudaError_t launch_swizzle_scales2(int rows_a, int rows_b, int K, const uint8_t *sfa, uint8_t *out_a,
                                   const uint8_t *sfb, uint8_t *out_b, cudaStream_t stream)
{
    const int cols = K / 16;
    const int ncb = (cols + 3) / 4;
    const int nrb_a = (rows_a + 127) / 128, nrb_b = (rows_b + 127) / 128;
    if ((long long)nrb_a + nrb_b > 65535)
        return cudaErrorInvalidConfiguration;
    dim3 grid((ncb + kSwzBlocksPerCta - 1) / kSwzBlocksPerCta, nrb_a + nrb_b);
    const int vec16 = (cols % 16) == 0 && (reinterpret_cast<uintptr_t>(sfa) & 15u) == 0 &&
                      (reinterpret_cast<uintptr_t>(sfb) & 15u) == 0;
    swizzle_scales_kernel<false><<<grid, kSwzThreads, 0, stream>>>(sfa, out_a, rows_a, cols, ncb, vec16, nullptr,
                                                                   0, sfb, out_b, rows_b, nrb_a);
    return cudaGetLastError();
}

cudaError_t launch_swizzle_scales_grouped(int E, int rows, int K, const int *offs, const uint8_t *sf,
                                          uint8_t *out, cudaStream_t stream)
{
    const int cols = K / 16;
    const int ncb = (cols + 3) / 4;
    const int nrb = (rows + 127) / 128 + E;     // bound on the slices' block rows
    dim3 grid((ncb + kSwzBlocksPerCta - 1) / kSwzBlocksPerCta, nrb);
    const int vec16 = (cols % 16) == 0 && (reinterpret_cast<uintptr_t>(sf) & 15u) == 0;
    swizzle_scales_kernel<true><<<grid, kSwzThreads, 0, stream>>>(sf, out, rows, cols, ncb, vec16, offs, E,
                                                                  nullptr, nullptr, 0, nrb);
    return cudaGetLastError();
}

// Tile-packed NVFP4 operand: tile (rb, kb) -- rows 128 rb .. +127, bytes
// 128 kb .. +127 of each -- stored whole at tile index rb * kblocks + kb,
// with the 128-byte swizzle applied inside (16-byte chunk c of row r at
// chunk c ^ (r % 8)) and rows past the end zero, so that one 16 KiB bulk
// copy into a 1024-byte-aligned buffer lands it as a 128B-swizzled
// tensor-map load would. One CTA per tile: 256 threads x four 16-byte
// chunks (loads coalesced along each row, stores along the tile).
__global__ void __launch_bounds__(256)
    pack_operand_kernel(const uint8_t *__restrict__ X, uint8_t *__restrict__ out, int rows, int width, int kblocks)
{
    const int kb = blockIdx.x, rb = blockIdx.y;
    uint8_t *const tile = out + ((size_t)rb * (size_t)kblocks + (size_t)kb) * 16384u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = threadIdx.x + 256 * j;           // chunk i of the tile's 1024: row i / 8, chunk i % 8
        const int r = i >> 3, c = i & 7;
        const int row = rb * 128 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < rows)
            v = __ldg(reinterpret_cast<const uint4 *>(X + (size_t)row * (size_t)width + (size_t)kb * 128u + c * 16));
        *reinterpret_cast<uint4 *>(tile + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
}

cudaError_t launch_pack_operand(int rows, int K, const uint8_t *X, uint8_t *out, cudaStream_t stream)
{
    const int kblocks = K / 256;
    const dim3 grid((unsigned)kblocks, (unsigned)((rows + 127) / 128));
    pack_operand_kernel<<<grid, 256, 0, stream>>>(X, out, rows, K / 2, kblocks);
    return cudaGetLastError();
}

// One thread waits, with the library's bounded wait, on an mbarrier that
// nothing arrives on: after `ns` it records the timeout and returns.
__global__ void watchdog_probe_kernel(unsigned int *status, unsigned long long ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        const Watchdog wd{status, ns};
        (void)mbar_wait(smem_u32(&bar), 0, wd, &abort_flag, 0xFu);
    }
}

cudaError_t launch_watchdog_probe(unsigned int *status, unsigned long long ns, cudaStream_t stream)
{
    watchdog_probe_kernel<<<1, 32, 0, stream>>>(status, ns);
    return cudaGetLastError();
}

}  // namespace bsg
