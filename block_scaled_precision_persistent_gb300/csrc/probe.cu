// Operand-ingress probe: how fast one SM can take bytes into its shared
// memory through the copy engine, with nothing else running. The tile
// kernels feed their tensor cores this way ("Together AI Ports
// ThunderKittens GEMM Kernels to NVIDIA Vera Rubin NVL72", introduction:
// loaders bring A and B into shared memory while one MMA warp drives the
// tensor cores), so this rate is a ceiling on their k-block period: a
// 256 x 256 NVFP4 pair tile needs 38,912 bytes per CTA and k-block.
//
// One CTA per SM; one thread keeps `stages` slots of two 16 KiB bulk copies
// (or, in the tensor-map form, two 128-row x 128-byte boxes)
// (global -> own shared memory) in flight over a source buffer, waiting on
// each slot's mbarrier before refilling it, and records its elapsed SM
// cycles. Every wait is bounded; a CTA whose wait runs out records the
// timeout status, lets its issued copies land, and returns.
#include "bsg_internal.h"
#include "ptx.cuh"

namespace bsg {

constexpr int kProbeChunk = 16384;
constexpr int kProbePerSlot = 2;
constexpr int kProbeSlotBytes = kProbeChunk * kProbePerSlot;
constexpr int kProbeMaxStages = 6;

__global__ void __launch_bounds__(32, 1)
    ingress_probe_kernel(const uint8_t *src, size_t src_bytes, int stages, int iters,
                         unsigned int *status, unsigned long long timeout_ns, unsigned long long *cycles)
{
    extern __shared__ __align__(1024) uint8_t slots[];
    __shared__ __align__(8) uint64_t bars[kProbeMaxStages];
    if (threadIdx.x != 0)
        return;
    for (int s = 0; s < stages; ++s)
        mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
    // each CTA starts at its own 1 KiB-aligned offset and wraps
    size_t off = ((size_t)blockIdx.x * 7919u * kProbeSlotBytes) % (src_bytes - kProbeSlotBytes);
    off -= off % 1024u;
    uint32_t phase = 0;
    const long long t0 = clock64();
    for (int it = 0; it < iters + stages; ++it) {
        const int s = it % stages;
        const uint32_t bar = smem_u32(&bars[s]);
        if (it >= stages) {
            const uint64_t w0 = global_timer_ns();
            while (!mbar_try_wait(bar, (phase >> s) & 1u)) {
                if (global_timer_ns() - w0 > timeout_ns) {
                    atomicCAS(status, 0u, (kStatusTimeout << 16) | 9u);
                    const uint64_t d0 = global_timer_ns();
                    while (global_timer_ns() - d0 < 200000ull) {
                    }
                    return;
                }
            }
            phase ^= 1u << s;
        }
        if (it < iters) {
            mbar_arrive_expect_tx(bar, kProbeSlotBytes);
#pragma unroll
            for (int c = 0; c < kProbePerSlot; ++c)
                bulk_load(smem_u32(slots + (size_t)s * kProbeSlotBytes + c * kProbeChunk), src + off + c * kProbeChunk,
                          kProbeChunk, bar);
            off += kProbeSlotBytes;
            if (off + kProbeSlotBytes > src_bytes)
                off = 0;
        }
    }
    cycles[blockIdx.x] = (unsigned long long)(clock64() - t0);
}

// The same with tensor-map copies shaped like the GEMM's operand tiles: each
// slot is two boxes of 128 rows x 128 bytes (128-byte swizzle) from a matrix
// of `rows` rows of `pitch` bytes, walking along the rows (K) first.
__global__ void __launch_bounds__(32, 1)
    tma_ingress_probe_kernel(const __grid_constant__ CUtensorMap tm, int xtiles, int ytiles, int stages, int iters,
                             unsigned int *status, unsigned long long timeout_ns, unsigned long long *cycles)
{
    extern __shared__ __align__(1024) uint8_t slots[];
    __shared__ __align__(8) uint64_t bars[kProbeMaxStages];
    if (threadIdx.x != 0)
        return;
    for (int s = 0; s < stages; ++s)
        mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
    int xt = 0, yt = (int)((blockIdx.x * 7u) % (unsigned)ytiles);
    uint32_t phase = 0;
    const long long t0 = clock64();
    for (int it = 0; it < iters + stages; ++it) {
        const int s = it % stages;
        const uint32_t bar = smem_u32(&bars[s]);
        if (it >= stages) {
            const uint64_t w0 = global_timer_ns();
            while (!mbar_try_wait(bar, (phase >> s) & 1u)) {
                if (global_timer_ns() - w0 > timeout_ns) {
                    atomicCAS(status, 0u, (kStatusTimeout << 16) | 10u);
                    const uint64_t d0 = global_timer_ns();
                    while (global_timer_ns() - d0 < 200000ull) {
                    }
                    return;
                }
            }
            phase ^= 1u << s;
        }
        if (it < iters) {
            mbar_arrive_expect_tx(bar, kProbeSlotBytes);
            tma_load_2d(smem_u32(slots + (size_t)s * kProbeSlotBytes), &tm, bar, xt * 128, yt * 128);
            tma_load_2d(smem_u32(slots + (size_t)s * kProbeSlotBytes + kProbeChunk), &tm, bar, xt * 128,
                        ((yt + 1) % ytiles) * 128);
            if (++xt == xtiles) {
                xt = 0;
                yt = (yt + 2) % ytiles;
            }
        }
    }
    cycles[blockIdx.x] = (unsigned long long)(clock64() - t0);
}

cudaError_t launch_tma_ingress_probe(const CUtensorMap &tm, int xtiles, int ytiles, int stages, int iters, int ctas,
                                     unsigned int *status, unsigned long long timeout_ns, unsigned long long *cycles,
                                     cudaStream_t stream)
{
    const int smem = stages * kProbeSlotBytes;
    cudaError_t e = cudaFuncSetAttribute(tma_ingress_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    tma_ingress_probe_kernel<<<ctas, 32, smem, stream>>>(tm, xtiles, ytiles, stages, iters, status, timeout_ns,
                                                         cycles);
    return cudaGetLastError();
}

cudaError_t launch_ingress_probe(const uint8_t *src, size_t src_bytes, int stages, int iters, int ctas,
                                 unsigned int *status, unsigned long long timeout_ns, unsigned long long *cycles,
                                 cudaStream_t stream)
{
    const int smem = stages * kProbeSlotBytes;
    cudaError_t e = cudaFuncSetAttribute(ingress_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    ingress_probe_kernel<<<ctas, 32, smem, stream>>>(src, src_bytes, stages, iters, status, timeout_ns, cycles);
    return cudaGetLastError();
}

int probe_slot_bytes() { return kProbeSlotBytes; }
int probe_max_stages() { return kProbeMaxStages; }

}  // namespace bsg
