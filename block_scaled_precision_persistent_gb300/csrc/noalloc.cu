// nvfp4_gemm_noalloc: the NVFP4 GEMM with row-major scales, for callers that
// cannot allocate device memory. nvfp4_gemm swizzles the scales into a
// workspace it grows with cudaMalloc; this entry point swizzles them into a
// fixed array that lives in the library's own module instead, so it never
// calls cudaMalloc, cudaFree or any allocating routine.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits. Host code cannot use its name as
// a device address (on the host the name is only a stand-in), so the address
// is looked up once per device with cudaGetSymbolAddress and passed to the
// kernels as a plain pointer.
#include <cstdint>
#include <mutex>

#include "bsg_internal.h"
#include "bsgemm.h"

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)BSG_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

}  // namespace

// Scratch for the two swizzled scale sets of one call (A's, then B's).
static __device__ __align__(256) uint8_t g_bsg_noalloc_scratch[BSG_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_scratch_mu;
uint8_t *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on
// the first call for that device (with that device current).
int scratch_on_current_device(uint8_t **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return BSG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bsg_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return BSG_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<uint8_t *>(p);
    }
    *out = g_scratch_addr[dev];
    return BSG_OK;
}

size_t round_up_256(size_t x) { return (x + 255u) & ~(size_t)255u; }

}  // namespace

extern "C" int nvfp4_gemm_noalloc(int M, int N, int K, const void *A, const void *sfA,
                                  const void *B, const void *sfB, float alpha, void *D,
                                  bsg_stream_t stream)
{
    // the same checks as nvfp4_gemm, before anything touches the scratch
    // array or launches: a bad call returns the same status and runs nothing
    int rc = bsg::validate_nvfp4_call(M, N, K, A, sfA, B, sfB, D);
    if (rc != BSG_OK)
        return rc;
    const size_t bytes_a = round_up_256(nvfp4_swizzled_scale_bytes(M, K));
    const size_t bytes_b = round_up_256(nvfp4_swizzled_scale_bytes(N, K));
    if (bytes_a + bytes_b > kNoallocScratchBytes)
        return BSG_ERR_EXCEEDS_SCRATCH;
    uint8_t *scratch = nullptr;
    if ((rc = scratch_on_current_device(&scratch)) != BSG_OK)
        return rc;
    // Every byte of both swizzled regions (padding included) is rewritten by
    // the swizzle, so the previous call's contents never leak into this one.
    // Both regions fit the scratch, so their block rows fit one launch's grid.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bsg::launch_swizzle_scales2(M, N, K, static_cast<const uint8_t *>(sfA), scratch,
                                    static_cast<const uint8_t *>(sfB), scratch + bytes_a, s) != cudaSuccess)
        return BSG_ERR_CUDA;
    rc = nvfp4_gemm_swizzled(M, N, K, A, scratch, B, scratch + bytes_a, alpha, D, stream);
    bsg::add_launches(1);   // the swizzle, after the GEMM's own count was set
    return rc;
}
