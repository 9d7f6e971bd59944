// Internal host/device interface between the C ABI (api.cu) and the kernel
// translation units. Not part of the public header.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsg {

// NVFP4: block-scaled E2M1 x E2M1; FP8: E4M3 x E4M3; NVFP4_BF16: block-scaled
// E2M1 activations x dense BF16 (or, with GemmArgs::b_f16, FP16) weights. NVFP4_BF16_TMEM is not a kind of
// call but a kernel variant of NVFP4_BF16 (the expanded A staged in tensor
// memory instead of shared memory); its plans report kind NVFP4_BF16.
enum class Kind : int { NVFP4 = 0, FP8 = 1, NVFP4_BF16 = 2, NVFP4_BF16_TMEM = 3 };

// Kernel families: persistent 1-SM tiles, persistent CTA-pair tiles, and the
// swap-AB split-K kernel for skinny M.
enum class Family : int { TC1 = 0, PAIR = 1, SKINNY = 2 };

// Everything a persistent GEMM launch needs besides its tensor maps.
struct GemmArgs {
    int M, N, K;
    int num_m_tiles, num_n_tiles, num_k_blocks;
    int raster_group;          // M tiles per rasterisation group
    int sf_col_blocks;         // NVFP4: 4-scale column blocks per 128-row block (K/64)
    int sfb_row_blocks;        // NVFP4: 128-row blocks of the swizzled B scales
    int sfx_row_blocks;        // skinny NVFP4: 128-row blocks of the swizzled A scales
    const uint8_t *sfa;        // NVFP4: swizzled A scales
    const uint8_t *sfb;        // NVFP4: swizzled B scales
    float alpha;
    const float *sA;           // FP8 per-tensor scales (device, may be null)
    const float *sB;
    unsigned int *status;      // device status word
    unsigned long long timeout_ns;
    // Fused epilogue variants, read only by the kernels instantiated with
    // EPI = true: D[dst(m)][n] = bf16(gamma[m] * (alpha * acc[m][n] + bias[n]))
    const float *bias;         // [N] FP32 added to every row, or null
    const float *gamma;        // [M] FP32 per-row multiplier, or null
    const int *scatter;        // [M] row of D that computed row m goes to, or null
    uint16_t *d;               // D (BF16 bits, row pitch N) for the scattered stores
    int m_out;                 // rows of D when scattered
    // Grouped (ragged) GEMM, read only by the GROUPED instantiation: A's
    // rows are num_groups slices by group_offs (device int32[E+1]); slice e
    // multiplies B rows [e*N, e*N + N), whose swizzled scales start
    // e * sfb_group_bytes bytes into sfb, and adds bias + e*N
    int num_groups;
    const int *group_offs;
    size_t sfb_group_bytes;
    // K-ragged (inner-expert) GEMM, read only by the KGROUPED instantiation:
    // group_offs (device int32[E+1]) splits K instead of M, and slice e
    // writes rows [e*M, e*M + M) of D with bias + e*N
    int k_grouped;
    // tile-packed operands (PACKED pair plans): 16 KiB tiles of 128 rows x
    // 128 bytes, 128B-swizzled inside, at tile index row_block * K/256 + kb
    const uint8_t *a_packed;
    const uint8_t *b_packed;
    // NVFP4 x dense kind: B holds FP16 values (A is expanded to FP16 and the
    // MMA runs kind::f16 with F16 operands) instead of BF16
    int b_f16;
    // launch with programmatic stream serialisation (the kernel's prologue
    // may overlap the previous kernel on the stream): 0 off, 1 on, 2 on and
    // B's codes are not written by the previous kernel, so the skinny-M and
    // 1-SM kernels start reading their first k-blocks of B before waiting
    int pdl;
};

// Kernel instantiations: the plain epilogue, the epilogue variants, the
// grouped GEMM and the K-ragged GEMM (both always with the variants'
// epilogue).
enum KernelMode : int { kModePlain = 0, kModeEpi = 1, kModeGrouped = 2, kModeKGrouped = 3 };

// True when a call needs the epilogue-variant kernels.
inline bool has_epilogue(const GemmArgs &a) { return a.bias || a.gamma || a.scatter; }

// One compiled persistent-kernel configuration.
struct PlanInfo {
    const char *name;
    Kind kind;
    Family family;
    int cta_group;             // 1: one SM per tile; 2: a CTA pair shares one tile
    int tile_m, bn;            // output tile of one scheduling unit (CTA or pair);
                               // skinny: max activation rows, weight rows per CTA
    int stages;                // smem ring depth
    int num_acc;               // TMEM accumulator buffers
    int k_block;               // K elements per ring stage
    int smem_bytes;            // dynamic shared memory per CTA
    int threads;
    int tmem_cols;
    int packed = 0;            // 1: reads tile-packed operands (nvfp4_gemm_packed only)
    int splits_mask = 0;       // skinny plans: bit S set for each K split the kernel takes
};

// Most slices the CTA-pair plan's grouped mode takes (its slice table sits
// in the shared memory left beside the ring).
constexpr int kPairMaxGroups = 256;

// Encoded tensor maps of one call (sfa / sfb only for CTA-pair NVFP4 plans).
struct GemmMaps {
    CUtensorMap a, b, d, sfa, sfb;
};

// Plan registry: the 1-SM plans (gemm_persistent.cu), then the CTA-pair plans
// (gemm_pair.cu), then the skinny plans (gemm_skinny.cu).
int num_plans();
const PlanInfo &plan_info(int id);
int find_plan(const char *name);

// Launch plan `id` with `grid` CTAs (a multiple of 2 for pair plans).
cudaError_t launch_gemm(int id, const GemmMaps &maps, const GemmArgs &args, int grid,
                        cudaStream_t stream);

// Largest number of CTAs of plan `id` that are co-resident on the current
// device (clusters x 2 for pair plans, SMs for 1-SM plans); 0 on error.
int max_resident_ctas(int id, int num_sms);

// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes), and the
// shared-memory carveout to its maximum, on the current device, once per
// (device, kernel, bytes): the attributes belong to the device's context,
// and setting them again on every launch cost host time.
cudaError_t set_max_dynamic_smem(const void *kern, int bytes);

int tc1_num_plans();
const PlanInfo &tc1_plan(int i);
cudaError_t tc1_launch(int i, const GemmMaps &maps, const GemmArgs &args, int grid,
                       cudaStream_t stream);
int pair_num_plans();
const PlanInfo &pair_plan(int i);
cudaError_t pair_launch(int i, const GemmMaps &maps, const GemmArgs &args, int grid,
                        cudaStream_t stream);
int pair_max_clusters(int i);
int skinny_num_plans();
const PlanInfo &skinny_plan(int i);
// Grid: weight tiles x splits (one cluster of `splits` CTAs per weight tile
// and activation block) x halves (activation blocks of tile_m rows); maps.d
// is not read (D is written with plain stores).
cudaError_t skinny_launch(int i, const GemmMaps &maps, const GemmArgs &args, int splits, int halves,
                          cudaStream_t stream);
// Thread-block clusters of `splits` CTAs of skinny plan i that fit on the
// device at once (0 if the query fails).
int skinny_max_clusters(int i, int splits);

// The checks nvfp4_gemm makes before it launches anything, in its order:
// arguments, 16-byte alignment, then the current device (compute 10.3).
// Resets the calling thread's launch count (bsg_last_launch_count).
int validate_nvfp4_call(int M, int N, int K, const void *A, const void *sfA, const void *B, const void *sfB,
                        void *D);
// Adds n to the calling thread's launch count.
void add_launches(int n);

// Scale-layout prep kernel. Returns a cudaError_t.
cudaError_t launch_swizzle_scales(int rows, int K, const uint8_t *sf, uint8_t *out,
                                  cudaStream_t stream);

// Per-slice scale-layout prep of a grouped A (offs: device int32[E+1]);
// out holds (ceil(rows / 128) + E) block rows.
// Both operands' scales of one GEMM (same K) in one launch.
cudaError_t launch_swizzle_scales2(int rows_a, int rows_b, int K, const uint8_t *sfa, uint8_t *out_a,
                                   const uint8_t *sfb, uint8_t *out_b, cudaStream_t stream);
cudaError_t launch_swizzle_scales_grouped(int E, int rows, int K, const int *offs, const uint8_t *sf,
                                          uint8_t *out, cudaStream_t stream);

// Two-level NVFP4 quantisation: memset of global[0], amax kernel, quantiser.
cudaError_t launch_nvfp4_quantize(int rows, int K, const void *X, uint8_t *packed, uint8_t *sf_swz,
                                  uint8_t *sf_rm, float *global, int num_sms, cudaStream_t stream,
                                  bool tiles = false);

// Tile-packed NVFP4 operand (swizzle.cu): rows x K/2 bytes -> 16 KiB tiles
// of 128 rows x 128 bytes, 128B-swizzled inside, rows padded to 128.
cudaError_t launch_pack_operand(int rows, int K, const uint8_t *X, uint8_t *out, cudaStream_t stream);

// Watchdog probe: waits on an mbarrier nothing arrives on.
cudaError_t launch_watchdog_probe(unsigned int *status, unsigned long long ns,
                                  cudaStream_t stream);

// Operand-ingress probe (probe.cu): `ctas` CTAs, one per SM, each keeping
// `stages` slots of probe_slot_bytes() of bulk copies in flight for `iters`
// refills; cycles[i] = CTA i's elapsed SM cycles.
cudaError_t launch_ingress_probe(const uint8_t *src, size_t src_bytes, int stages, int iters, int ctas,
                                 unsigned int *status, unsigned long long timeout_ns, unsigned long long *cycles,
                                 cudaStream_t stream);
cudaError_t launch_tma_ingress_probe(const CUtensorMap &tm, int xtiles, int ytiles, int stages, int iters, int ctas,
                                     unsigned int *status, unsigned long long timeout_ns, unsigned long long *cycles,
                                     cudaStream_t stream);
int probe_slot_bytes();
int probe_max_stages();

}  // namespace bsg
