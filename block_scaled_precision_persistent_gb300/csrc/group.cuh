// Slice table of a grouped (ragged, routed) GEMM, built on the device from
// the routing offsets, so that no host synchronisation is needed
// ("Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
// Tensor-Memory Failures", section "Ragged mode added routing rather than a
// plain matrix": routed activation rows form slices, each multiplied by the
// dense right-hand side of its own slice).
#pragma once

#include <cstdint>

namespace bsg {

// Largest number of slices a grouped call takes (the table lives in shared
// memory: two int32 arrays of kMaxGroups + 1 entries).
constexpr int kMaxGroups = 1024;
constexpr int kGroupTableBytes = 2 * (kMaxGroups + 1) * 4;

// One warp fills, for offs[0..E] (device, int32):
//   so[e] = min(M, max(0, offs[0], ..., offs[e]))   e = 0..E
//     the slice boundaries, clamped to a nondecreasing sequence in [0, M]
//     (valid offsets -- offs[0] = 0, nondecreasing, offs[E] = M -- are kept
//     as they are; any others can then neither read nor write out of bounds)
//   sb[e] = sum_{e' < e} ceil((so[e'+1] - so[e']) / 128)   e = 0..E
//     the first 128-row block of slice e: one GEMM tile row of 128 rows and
//     one block row of the per-slice swizzled scales each
// Each lane owns a run of consecutive entries; two warp scans (max, then
// sum) join the runs. The caller synchronises before other warps read.
__device__ __forceinline__ void build_group_table(const int *offs, int E, int M, int *so, int *sb, int lane)
{
    const int n = E + 1;
    const int per = (n + 31) / 32;
    const int lo = min(lane * per, n), hi = min(lo + per, n);
    // boundaries: prefix max, clamped
    int run = 0;
    for (int i = lo; i < hi; ++i)
        run = max(run, __ldg(offs + i));
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl = max(incl, v);
    }
    int excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0)
        excl = 0;
    run = excl;
    for (int i = lo; i < hi; ++i) {
        run = max(run, __ldg(offs + i));
        so[i] = min(run, M);
    }
    __syncwarp();
    // 128-row blocks: entry i (i >= 1) adds slice i - 1
    int sum = 0;
    for (int i = max(lo, 1); i < hi; ++i)
        sum += (so[i] - so[i - 1] + 127) / 128;
    int isum = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, isum, d);
        if (lane >= d)
            isum += v;
    }
    run = isum - sum;
    for (int i = lo; i < hi; ++i) {
        if (i >= 1)
            run += (so[i] - so[i - 1] + 127) / 128;
        sb[i] = run;
    }
    __syncwarp();
}

// After build_group_table: one warp fills, for the boundaries so[0..E],
//   sp[e] = sum_{e' < e} ceil((so[e'+1] - so[e']) / rows)   e = 0..E
// the first block of `rows` rows of slice e (the CTA pair's 256-row tile
// rows). The caller synchronises before other warps read.
__device__ __forceinline__ void build_block_prefix(const int *so, int E, int rows, int *sp, int lane)
{
    const int n = E + 1;
    const int per = (n + 31) / 32;
    const int lo = min(lane * per, n), hi = min(lo + per, n);
    int sum = 0;
    for (int i = max(lo, 1); i < hi; ++i)
        sum += (so[i] - so[i - 1] + rows - 1) / rows;
    int isum = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, isum, d);
        if (lane >= d)
            isum += v;
    }
    int run = isum - sum;
    for (int i = lo; i < hi; ++i) {
        if (i >= 1)
            run += (so[i] - so[i - 1] + rows - 1) / rows;
        sp[i] = run;
    }
    __syncwarp();
}

// The slice that block row b (0 <= b < sb[E]) belongs to: the largest e with
// sb[e] <= b (empty slices share their sb with the next one and are skipped).
__device__ __forceinline__ int group_of_block(const int *sb, int E, int b)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sb[mid] <= b)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

}  // namespace bsg
