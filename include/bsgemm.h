/*
 * bsgemm.h -- C ABI of the block-scaled low-precision GEMM library for one
 * GB300 GPU (sm_103a).
 *
 *     D = alpha * (A (.) sA) (B (.) sB)^T,   FP32 accumulation, BF16 output
 *
 * The operation is the NVFP4 / FP8 GEMM of "Together AI Ports ThunderKittens
 * GEMM Kernels to NVIDIA Vera Rubin NVL72" (introduction; "Building the
 * GEMM"): a tcgen05 tensor-core MMA that reads its operands from shared memory,
 * accumulates in tensor memory and consumes one E4M3 scale per 16 K-elements
 * (NVFP4) or per-tensor FP32 scales (FP8). The scale-layout prep call follows
 * "Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
 * Failures", "Activation-scale swizzling forced the relevant persistent path":
 * the persistent kernel reads scales in a layout rewritten in HBM beforehand.
 *
 * Conventions shared by every entry point
 *  - All matrix arguments are DEVICE pointers on the current CUDA device,
 *    owned by the caller. The library never frees or retains them.
 *  - Row-major everywhere. A is [M][K], B is [N][K] (so the GEMM contracts
 *    the contiguous K dimension of both), D is [M][N] BF16.
 *  - NVFP4 operand rows hold E2M1 codes packed two per byte along K: element
 *    2i in bits 0..3 of byte i, element 2i+1 in bits 4..7 (A: uint8[M][K/2]).
 *  - Row-major NVFP4 scales: uint8[rows][K/16], one E4M3 code per 16
 *    consecutive K-elements; scales are read as unsigned (the sign bit must be
 *    clear) and must not be NaN.
 *  - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *    NULL = legacy default stream). No call synchronises except
 *    bsg_get_device_status.
 *  - Every function returns a bsg_status code; no exception crosses the ABI.
 *    Argument errors are detected on the host before anything is launched.
 *  - Sizes: M, N >= 1; N % 8 == 0 (16-byte BF16 rows for the TMA store);
 *    NVFP4: K % 256 == 0; FP8: K % 128 == 0. Base pointers must be 16-byte
 *    aligned.
 *  - A GPU-side wait that exceeds the watchdog limit (default 1 s per wait)
 *    makes the kernel record BSG_ERR_DEVICE_TIMEOUT in a device status word
 *    and return instead of hanging; read it with bsg_get_device_status.
 */
#ifndef BSGEMM_H
#define BSGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BSG_API __attribute__((visibility("default")))
#else
#define BSG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *bsg_stream_t;

typedef enum bsg_status {
    BSG_OK = 0,
    BSG_ERR_INVALID_ARG = 1,        /* null pointer, bad size or multiple     */
    BSG_ERR_MISALIGNED = 2,         /* a base pointer is not 16-byte aligned  */
    BSG_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute 10.3     */
    BSG_ERR_NO_PLAN = 4,            /* forced plan unknown or unfit for shape */
    BSG_ERR_CUDA = 5,               /* a CUDA runtime / driver call failed    */
    BSG_ERR_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait ran out        */
    BSG_ERR_OUT_OF_MEMORY = 7,      /* workspace allocation failed            */
    BSG_ERR_EXCEEDS_SCRATCH = 8     /* nvfp4_gemm_noalloc: scales do not fit
                                       in its fixed scratch array            */
} bsg_status;

/* Size of the fixed device scratch array used by nvfp4_gemm_noalloc.      */
#define BSG_NOALLOC_SCRATCH_BYTES (16u << 20)

/* ---------------------------------------------------------------------------
 * NVFP4 GEMM with row-major scales.
 *   A   : uint8[M][K/2]  E2M1 codes, two per byte
 *   sfA : uint8[M][K/16] E4M3 block scales, row-major
 *   B   : uint8[N][K/2]
 *   sfB : uint8[N][K/16]
 *   D   : bf16[M][N]; D = bf16_rn(alpha * sum_k a*sA * b*sB), FP32 accumulate
 * Swizzles sfA and sfB into a library-owned per-device workspace (grown on
 * demand with cudaMalloc; pre-size it with bsg_reserve_workspace before any
 * stream capture), then runs nvfp4_gemm_swizzled. Calls on different streams
 * of one device share that workspace and must not overlap in time.
 * ------------------------------------------------------------------------- */
BSG_API int nvfp4_gemm(int M, int N, int K,
               const void *A, const void *sfA,
               const void *B, const void *sfB,
               float alpha, void *D, bsg_stream_t stream);

/* Same GEMM with scales already in the swizzled layout produced by
 * nvfp4_swizzle_scales (sfA_swz: nvfp4_swizzled_scale_bytes(M, K) bytes,
 * sfB_swz: nvfp4_swizzled_scale_bytes(N, K) bytes). Allocates nothing.     */
BSG_API int nvfp4_gemm_swizzled(int M, int N, int K,
                        const void *A, const void *sfA_swz,
                        const void *B, const void *sfB_swz,
                        float alpha, void *D, bsg_stream_t stream);

/* ---------------------------------------------------------------------------
 * Tile-packed NVFP4 operands (this library's own layout, made to be loaded
 * by one contiguous 16 KiB bulk copy per tile instead of a tensor-map box:
 * the per-SM ingest rate of contiguous copies is the higher one on sm_103a).
 * Tile (rb, kb) holds rows 128 rb .. 128 rb + 127 and bytes 128 kb ..
 * 128 kb + 127 of each row of a row-major uint8[rows][K/2] operand, stored
 * at byte offset (rb * K/256 + kb) * 16384; inside a tile, byte c of row r
 * sits at r * 128 + ((c / 16) XOR (r % 8)) * 16 + c % 16 (the 128-byte
 * swizzle); rows past `rows` are zero.
 *
 * nvfp4_packed_operand_bytes: size of that layout, rows padded to 128
 *   (0 for rows < 1 or K not a positive multiple of 256). Host only.
 * nvfp4_pack_operand: X uint8[rows][K/2] (device, 16-byte aligned) ->
 *   out (device, 16-byte aligned, nvfp4_packed_operand_bytes(rows, K)
 *   bytes). Bit-exact byte permutation; one launch on `stream`. Requires
 *   ceil(rows / 128) <= 65535.
 * nvfp4_gemm_packed: the GEMM of nvfp4_gemm_swizzled with A and B given in
 *   the packed layout (A_packed: nvfp4_packed_operand_bytes(M, K) bytes,
 *   B_packed: nvfp4_packed_operand_bytes(N, K)), scales in the swizzled
 *   layout. Always runs the plan "nvfp4_tc2_256x256_s5_acc1_packed" (a
 *   forced plan does not apply; that plan cannot be forced on the other
 *   entries). Same size and alignment rules and result as
 *   nvfp4_gemm_swizzled; allocates nothing.
 * nvfp4_gemm_packed_ex: the same with the epilogue variants of
 *   nvfp4_gemm_ex (bias, gamma, scatter, m_out: same meaning, layouts and
 *   checks).
 * ------------------------------------------------------------------------- */
BSG_API size_t nvfp4_packed_operand_bytes(int rows, int K);
BSG_API int nvfp4_pack_operand(int rows, int K, const void *X, void *out, bsg_stream_t stream);
BSG_API int nvfp4_gemm_packed(int M, int N, int K,
                      const void *A_packed, const void *sfA_swz,
                      const void *B_packed, const void *sfB_swz,
                      float alpha, void *D, bsg_stream_t stream);
BSG_API int nvfp4_gemm_packed_ex(int M, int N, int K,
                         const void *A_packed, const void *sfA_swz,
                         const void *B_packed, const void *sfB_swz, float alpha,
                         const float *bias, const float *gamma, const int32_t *scatter,
                         int m_out, void *D, bsg_stream_t stream);

/* Scale-layout prep: row-major uint8[rows][K/16] -> the tcgen05 block-scale
 * layout: rows padded to a multiple of 128, K/16 padded to a multiple of 4,
 * 128x4 blocks of 512 bytes ordered row-block-major with the column block
 * fastest; inside a block, (r, c) -> byte (r%32)*16 + (r/32)*4 + c. Padding
 * is written as zero. Requires K % 16 == 0; sf_swz must hold
 * nvfp4_swizzled_scale_bytes(rows, K) bytes. Bit-exact byte permutation.  */
BSG_API int nvfp4_swizzle_scales(int rows, int K, const void *sf, void *sf_swz,
                         bsg_stream_t stream);

/* Both operands' scales of one GEMM in one launch: sfA uint8[M][K/16] ->
 * sfA_swz, sfB uint8[N][K/16] -> sfB_swz, each exactly as
 * nvfp4_swizzle_scales would write it. Requires M, N >= 1, K % 16 == 0,
 * 16-byte aligned outputs. (Where ceil(M/128) + ceil(N/128) exceeds 65535
 * the two operands take one launch each.) nvfp4_gemm uses it.           */
BSG_API int nvfp4_swizzle_scales2(int M, int N, int K, const void *sfA, void *sfA_swz,
                                  const void *sfB, void *sfB_swz, bsg_stream_t stream);

/* Size in bytes of the swizzled layout (0 for invalid sizes). Host only.  */
BSG_API size_t nvfp4_swizzled_scale_bytes(int rows, int K);

/* ---------------------------------------------------------------------------
 * Two-level NVFP4 quantisation of a BF16 matrix (the step in front of the
 * GEMM: "Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
 * Tensor-Memory Failures" names a shared NVFP4 quantisation; the scheme is
 * this library's reading of it):
 *   amax  = max |x| over the matrix;  s_g = 2688 / amax (1 if amax == 0)
 *   per 16 consecutive K elements, bmax = max |x|:
 *     scale = E4M3 nearest-even (saturating at 448) of (bmax / 6) * s_g
 *     code  = E2M1 nearest-even (saturating at 6) of (x * s_g) / scale
 *             (0 where scale is 0), every step in FP32 rounded once
 * so that D = A_q B_q^T / (s_gA s_gB): pass alpha = 1 / (s_gA * s_gB) to the
 * GEMM.
 *   X           : bf16[rows][K] row-major, device, 16-byte aligned
 *   packed      : uint8[rows][K/2] out (element 2i in the low nibble), 16-byte aligned
 *   sf_swz      : uint8[nvfp4_swizzled_scale_bytes(rows, K)] out, the layout
 *                 nvfp4_gemm_swizzled reads (padding written zero), 16-byte aligned
 *   sf_rowmajor : uint8[rows][K/16] out, or NULL
 *   global      : float[2] device out: global[0] = amax, global[1] = s_g; 8-byte aligned
 * Requires rows >= 1, K % 16 == 0, finite inputs. Stream-ordered: one
 * 4-byte memset and two kernels; allocates nothing.                       */
BSG_API int nvfp4_quantize(int rows, int K, const void *X, void *packed, void *sf_swz,
                           void *sf_rowmajor, float *global, bsg_stream_t stream);

/* The same quantisation with the codes written in the tile-packed operand
 * layout that nvfp4_gemm_packed reads (see nvfp4_pack_operand), so that
 * activations need no separate packing pass: packed_tiles holds
 * nvfp4_packed_operand_bytes(rows, K) bytes (16-byte aligned), and the
 * padding rows of its last row block are written as zero codes. Scales,
 * global and every other argument as nvfp4_quantize. Requires K % 256 == 0
 * (BSG_ERR_INVALID_ARG otherwise).                                         */
BSG_API int nvfp4_quantize_tiles(int rows, int K, const void *X, void *packed_tiles, void *sf_swz,
                                 void *sf_rowmajor, float *global, bsg_stream_t stream);

/* NVFP4 GEMM with row-major scales that allocates nothing. The pages have no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc -- for instance a runtime that has handed all device memory to
 * its own pool allocator, or code running where a device allocation is not
 * allowed (a host callback, a loop with a no-allocation rule).
 *   Arguments, layouts, result and error codes are those of nvfp4_gemm,
 *   checked in the same order before anything is launched or written.
 *   Scratch: the swizzled scales of A and B go to one file-scope device
 *   array of BSG_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU which loads
 *   the library holds until the process exits. A call needs
 *   round256(nvfp4_swizzled_scale_bytes(M, K)) +
 *   round256(nvfp4_swizzled_scale_bytes(N, K)) bytes of it (for example
 *   M = N = 8192 at K = 16384); larger requests return
 *   BSG_ERR_EXCEEDS_SCRATCH before anything is launched.
 *   Set-up: the first call on a device looks up the array's device address
 *   with cudaGetSymbolAddress (with that device current); make that first
 *   call before any stream capture.
 *   Sharing: all calls share the one array, which keeps the last call's
 *   contents. Each call rewrites every byte it reads, so nothing needs
 *   clearing, but calls whose work overlaps on the GPU (different streams)
 *   race on the array and must be serialised by the caller.
 *   bsg_last_launch_count() afterwards counts the swizzle and the GEMM.    */
BSG_API int nvfp4_gemm_noalloc(int M, int N, int K,
                               const void *A, const void *sfA,
                               const void *B, const void *sfB,
                               float alpha, void *D, bsg_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 E4M3 GEMM with per-tensor FP32 scales.
 *   A : uint8[M][K] E4M3, B : uint8[N][K] E4M3, D : bf16[M][N]
 *   sA, sB: DEVICE pointers to one float each, or NULL for 1.0
 *   D = bf16_rn(alpha * sA * sB * sum_k a*b), FP32 accumulate
 * ------------------------------------------------------------------------- */
BSG_API int fp8_gemm(int M, int N, int K,
             const void *A, const float *sA,
             const void *B, const float *sB,
             float alpha, void *D, bsg_stream_t stream);

/* ---------------------------------------------------------------------------
 * Fused epilogue variants: shared bias, per-row gamma, scattered output rows
 * ("Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
 * Tensor-Memory Failures", sections "Scatter changes where output rows are
 * written", "Gamma adds a per-row scaling input" and "The ordinary variants
 * also exercise the shared bias route": the NVFP4 x dense matmul plus bias,
 * optional gamma, optional scatter). Reading of the order (the pages list
 * the steps, not a formula):
 *     D[dst(m)][n] = bf16_rn( gamma[m] * (alpha * acc[m][n] + bias[n]) )
 * computed in FP32 in the GEMM's epilogue (one FMA, one multiply, one
 * rounding to BF16); acc as for nvfp4_gemm_swizzled / fp8_gemm (for FP8,
 * alpha stands for alpha * sA * sB).
 *   bias    : DEVICE float[N], 16-byte aligned, or NULL (no bias)
 *   gamma   : DEVICE float[M], 4-byte aligned, or NULL (gamma = 1)
 *   scatter : DEVICE int32[M], 4-byte aligned, or NULL (dst(m) = m). Computed
 *             row m is written to row scatter[m] of D; an index outside
 *             [0, m_out) -- e.g. -1 for a padding row -- writes nothing.
 *             Indices must be distinct (two rows sent to one destination:
 *             which one lands is unspecified). Rows of D that no index
 *             names are left as they were.
 *   m_out   : rows of D (D is bf16[m_out][N], row pitch N, 16-byte aligned).
 *             Without scatter m_out must equal M; with it m_out >= 1.
 * Other arguments, layouts and errors as nvfp4_gemm_swizzled / fp8_gemm;
 * allocates nothing. With bias, gamma and scatter all NULL the call is
 * exactly nvfp4_gemm_swizzled / fp8_gemm. Only the scatter indices are
 * range-checked (on the GPU, per row); the caller guarantees the lengths.
 * ------------------------------------------------------------------------- */
BSG_API int nvfp4_gemm_ex(int M, int N, int K,
                          const void *A, const void *sfA_swz,
                          const void *B, const void *sfB_swz,
                          float alpha, const float *bias, const float *gamma,
                          const int32_t *scatter, int m_out, void *D, bsg_stream_t stream);

BSG_API int fp8_gemm_ex(int M, int N, int K,
                        const void *A, const float *sA,
                        const void *B, const float *sB,
                        float alpha, const float *bias, const float *gamma,
                        const int32_t *scatter, int m_out, void *D, bsg_stream_t stream);

/* ---------------------------------------------------------------------------
 * NVFP4 x dense-BF16 / dense-FP16 GEMM ("Triton #11171 - Why Two New NVFP4
 * Test Cases Produced Twelve Tensor-Memory Failures", opening: an
 * NVFP4-scaled activation times a dense BF16 or FP16 operand, with the
 * shared bias route and the optional gamma and scatter):
 *   D[dst(m)][n] = bf16_rn( gamma[m] * (alpha * sum_k a(m,k) sA(m,k/16) * b(n,k) + bias[n]) )
 *   A       : uint8[M][K/2] E2M1 codes (element 2i in the low nibble)
 *   sfA_swz : A's E4M3 block scales in the swizzled layout (nvfp4_swizzle_scales)
 *   B       : nvfp4_dense_gemm: bf16[N][K]; nvfp4_dense_f16_gemm: IEEE
 *             binary16 [N][K]; row-major (K contiguous), plain values
 *   bias, gamma, scatter, m_out, D: as nvfp4_gemm_ex (D is BF16 in both)
 * The codes times their scales are exact in BF16 and in FP16 (at most 6
 * significant bits, magnitudes 2^-10 .. 2688), so the kernel expands A to
 * B's type and runs the 16-bit tensor core; the sum is FP32. Requires K % 64 == 0, N % 8 == 0, 16-byte aligned
 * A, sfA_swz, B, D. One launch; allocates nothing.
 * ------------------------------------------------------------------------- */
BSG_API int nvfp4_dense_gemm(int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                             float alpha, const float *bias, const float *gamma, const int32_t *scatter,
                             int m_out, void *D, bsg_stream_t stream);

BSG_API int nvfp4_dense_f16_gemm(int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                                 float alpha, const float *bias, const float *gamma, const int32_t *scatter,
                                 int m_out, void *D, bsg_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped (ragged, routed) NVFP4 GEMM -- the MoE expert matmul ("Triton
 * #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
 * Failures", section "Ragged mode added routing rather than a plain matrix":
 * routed activation rows form slices, and each slice is multiplied by the
 * dense right-hand side of its own slice):
 *   for each slice e in [0, E) and offs[e] <= m < offs[e+1]:
 *     D[dst(m)][n] = bf16_rn( gamma[m] * (alpha * sum_k a(m,k) sA * b_e(n,k) sB_e + bias[e][n]) )
 * with dst / gamma / scatter / m_out exactly as nvfp4_gemm_ex.
 *   A       : uint8[M][K/2], rows grouped by slice (slice e = rows offs[e] .. offs[e+1]-1)
 *   sfA_swz : A's scales in the per-slice layout of nvfp4_swizzle_scales_grouped
 *   B       : uint8[E][N][K/2], the slices' right-hand sides
 *   sfB_swz : E swizzled scale sets of N rows, each nvfp4_swizzled_scale_bytes(N, K)
 *             bytes, back to back (nvfp4_swizzle_scales on the [E*N][K/16] matrix
 *             gives exactly this when N % 128 == 0)
 *   offs    : DEVICE int32[E+1], 4-byte aligned: offs[0] = 0, nondecreasing,
 *             offs[E] = M. Read on the GPU (no host synchronisation). Any other
 *             sequence is clamped there to a nondecreasing one in [0, M], so
 *             that nothing is read or written out of bounds; its result is
 *             unspecified.
 *   bias    : DEVICE float[E][N], 16-byte aligned, or NULL
 * 1 <= E <= 1024 slices; slices may be empty. Sizes, alignment and errors as
 * nvfp4_gemm_ex. One launch; allocates nothing. Plans: with many tiles and
 * E <= 256, the CTA pair with one 256-row tile row per 256 rows of a slice;
 * otherwise the 1-SM plans with 128-row tile rows. A forced CTA-pair plan
 * with E > 256 gives BSG_ERR_NO_PLAN.
 * ------------------------------------------------------------------------- */
BSG_API int nvfp4_grouped_gemm(int E, int M, int N, int K,
                               const void *A, const void *sfA_swz,
                               const void *B, const void *sfB_swz,
                               const int32_t *offs, float alpha,
                               const float *bias, const float *gamma,
                               const int32_t *scatter, int m_out, void *D, bsg_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped (routed) NVFP4 x dense GEMM: the pages' ragged mode with a dense
 * BF16 (nvfp4_dense_grouped_gemm) or FP16 (nvfp4_dense_f16_grouped_gemm)
 * right-hand side ("Triton #11171 - Why Two New NVFP4 Test Cases Produced
 * Twelve Tensor-Memory Failures", section "Ragged mode added routing rather
 * than a plain matrix", and its opening for the dense operand):
 *   for each slice e in [0, E) and offs[e] <= m < offs[e+1]:
 *     D[dst(m)][n] = bf16_rn( gamma[m] * (alpha * sum_k a(m,k) sA(m,k/16) * b_e(n,k) + bias[e][n]) )
 *   A       : uint8[M][K/2] E2M1 codes, rows grouped by slice
 *   sfA_swz : A's scales in the per-slice layout of nvfp4_swizzle_scales_grouped
 *   B       : 16-bit [E][N][K] row-major (K contiguous), plain values
 *   offs, bias ([E][N]), gamma, scatter, m_out, D: as nvfp4_grouped_gemm
 * Requires K % 64 == 0, N % 8 == 0, 16-byte aligned A, sfA_swz, B, D and a
 * 4-byte aligned offs; 1 <= E <= 1024, slices may be empty. One launch;
 * allocates nothing. Runs only the plans that stage the expanded A in tensor
 * memory and leave room for the slice table (a forced plan otherwise gives
 * BSG_ERR_NO_PLAN).
 * ------------------------------------------------------------------------- */
BSG_API int nvfp4_dense_grouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz,
                                     const void *B, const int32_t *offs, float alpha, const float *bias,
                                     const float *gamma, const int32_t *scatter, int m_out, void *D,
                                     bsg_stream_t stream);

BSG_API int nvfp4_dense_f16_grouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz,
                                         const void *B, const int32_t *offs, float alpha, const float *bias,
                                         const float *gamma, const int32_t *scatter, int m_out, void *D,
                                         bsg_stream_t stream);

/* ---------------------------------------------------------------------------
 * Inner-expert (K-ragged) NVFP4 x dense GEMM: the pages' K-ragged variant
 * with a BF16 (nvfp4_dense_kgrouped_gemm) or FP16 (..._f16_...) right-hand
 * side ("Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
 * Tensor-Memory Failures", section "Why `pad_a` represents the K-ragged
 * boundary": the ragged dimension is A's K, padded per slice). K is split
 * into E slices at koffs and slice e gives its own output:
 *   D[e][m][n] = bf16_rn( gamma[m] * (alpha * sum_{k in slice e} a(m,k) sA(m,k/16) * b(n,k) + bias[e][n]) )
 *   A       : uint8[M][K/2] E2M1 codes; sfA_swz: its scales, swizzled over all of K
 *   B       : 16-bit [N][K] row-major, plain values
 *   koffs   : DEVICE int32[E+1], 4-byte aligned: koffs[0] = 0, nondecreasing,
 *             koffs[E] = K, each a multiple of 64 (the caller pads every
 *             slice to whole 64-element blocks, with zero codes in A).
 *             Read on the GPU; other sequences are clamped there to a
 *             nondecreasing one in [0, K] (nothing is read or written out of
 *             bounds; the result is unspecified). An empty slice gives
 *             D[e] = bf16(gamma * (0 + bias[e])).
 *   bias    : DEVICE float[E][N], 16-byte aligned, or NULL
 *   gamma   : DEVICE float[M], 4-byte aligned, or NULL
 *   D       : bf16[E][M][N], 16-byte aligned
 * Requires K % 64 == 0, N % 8 == 0, 16-byte aligned A, sfA_swz, B, D;
 * 1 <= E <= 1024. One launch; allocates nothing. Plans as
 * nvfp4_dense_grouped_gemm.
 * ------------------------------------------------------------------------- */
BSG_API int nvfp4_dense_kgrouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz,
                                      const void *B, const int32_t *koffs, float alpha, const float *bias,
                                      const float *gamma, void *D, bsg_stream_t stream);

BSG_API int nvfp4_dense_f16_kgrouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz,
                                          const void *B, const int32_t *koffs, float alpha, const float *bias,
                                          const float *gamma, void *D, bsg_stream_t stream);

/* Scale layout of a grouped A: row-major uint8[M][K/16] scales -> the
 * swizzled layout of nvfp4_swizzle_scales applied to each slice on its own,
 * slice e starting at 128-row block row sum_{e'<e} ceil(rows_e' / 128), so
 * that every 128-row tile of one slice reads one block row. offs as for
 * nvfp4_grouped_gemm (device, read on the GPU). sf_swz must hold
 * nvfp4_grouped_scale_bytes(E, M, K) bytes, 16-byte aligned; block rows past
 * the slices' are written as zeros. Requires M >= 1, K % 16 == 0, 1 <= E <=
 * 1024. Bit-exact byte permutation.                                        */
BSG_API int nvfp4_swizzle_scales_grouped(int E, int M, int K, const int32_t *offs, const void *sf,
                                         void *sf_swz, bsg_stream_t stream);

/* Bytes of the grouped layout: (ceil(M/128) + E) block rows of 128 rows x
 * K/16 (padded to 4) scales -- a bound on any split of M rows into E
 * slices (0 for invalid sizes). Host only.                                 */
BSG_API size_t nvfp4_grouped_scale_bytes(int E, int M, int K);

/* ---------------------------------------------------------------------------
 * Runtime control
 * ------------------------------------------------------------------------- */

/* Grow the nvfp4_gemm scale workspace of `device` to at least `bytes`.    */
BSG_API int bsg_reserve_workspace(int device, size_t bytes);

/* Synchronise `stream`, then return and clear the device status word of the
 * current device: BSG_OK, BSG_ERR_DEVICE_TIMEOUT (a bounded wait ran out) or
 * BSG_ERR_CUDA (the stream reported an error).                            */
BSG_API int bsg_get_device_status(bsg_stream_t stream);

/* Raw status word of the last bsg_get_device_status call on this thread:
 * 0, or (BSG_ERR_DEVICE_TIMEOUT << 16) | wait-site id.                    */
BSG_API uint32_t bsg_last_status_word(void);

/* Per-wait watchdog limit in nanoseconds used by later launches (0 restores
 * the default of 1e9).                                                    */
BSG_API int bsg_set_watchdog_ns(uint64_t ns);

/* Programmatic dependent launch for later GEMM launches (1 on, 0 off, the
 * default): each kernel's prologue (barrier set-up, tensor-memory
 * allocation, descriptor prefetch) may then overlap the end of the previous
 * kernel on the same stream; every kernel still waits for that kernel's
 * completion before its first dependent global access, so results do not
 * change. 2: on, and the caller promises that the previous kernel on the
 * stream does not write B's codes (the weights of an inference chain whose
 * previous kernel produced the activations): the skinny-M kernel then loads
 * its first ring stages of B's codes, and the 1-SM tile kernel warms L2 with
 * the first k-blocks of its first tile's B codes, before that wait. B's
 * scales, A and everything else still wait; the other kernels behave as
 * with 1. A chain that breaks the promise reads stale weights. Returns
 * BSG_ERR_INVALID_ARG for other values. Process-wide.                      */
BSG_API int bsg_set_pdl(int on);

/* Tuning lever: M tiles per rasterisation group of the tile kernels (the
 * tile order walks the group's M tiles fastest, so that the CTAs resident at
 * one time share a band of B in L2) for later launches; 0 restores the
 * default of 16. 1 <= m_tiles <= 1024. Process-wide.                       */
BSG_API int bsg_set_raster_group(int m_tiles);

/* Tuning lever: K splits of the skinny-M kernel (the thread-block cluster
 * that shares one weight tile) for later launches: 1 to 6 or 8, or 0
 * (the default) to let each call choose the split whose busiest SM streams
 * the fewest k-blocks. A forced split that the plan's receive area cannot
 * hold (5 with 256 activation rows) or that leaves the grid unable to be
 * resident at once makes those calls return BSG_ERR_NO_PLAN. Process-wide;
 * BSG_ERR_INVALID_ARG for other values.                                    */
BSG_API int bsg_set_skinny_splits(int splits);

/* Launch a one-thread probe that waits, with the library's bounded wait, on
 * an mbarrier that nothing ever arrives on. After `ns` nanoseconds it records
 * BSG_ERR_DEVICE_TIMEOUT in the status word and returns: a test of the
 * watchdog that faults and hangs nothing.                                 */
BSG_API int bsg_watchdog_selftest(uint64_t ns, bsg_stream_t stream);

/* Operand-ingress probe: the rate at which one SM takes bytes into its
 * shared memory through the copy engine with nothing else running -- the
 * ceiling on a tile kernel's k-block period, whose loaders bring A, B and
 * their scales into shared memory ("Together AI Ports ThunderKittens GEMM
 * Kernels to NVIDIA Vera Rubin NVL72", introduction).
 *   src_bytes : source buffer size (>= 128 KiB; >= 2 MiB with tensor_boxes);
 *               32 MiB keeps it in L2
 *   stages    : 1..6 slots of 32 KiB copies in flight per SM
 *   tensor_boxes : 0 = contiguous 16 KiB bulk copies; 1 = tensor-map copies
 *               of 128-row x 128-byte boxes (128-byte swizzle) from rows of
 *               8192 bytes, the pattern of the GEMMs' NVFP4 operand tiles
 *   bytes_per_cycle_per_sm : out, bytes per SM clock cycle, averaged over SMs
 *   total_gbs : out (may be NULL), bytes of all SMs per second
 * One CTA per SM, 4000 refills per slot, after one untimed pass. Blocking:
 * allocates and frees its own buffers and stream, so it is a measurement
 * routine, not one for a hot path. A wait that runs out returns
 * BSG_ERR_DEVICE_TIMEOUT (and leaves the status word set, as the GEMMs do). */
BSG_API int bsg_measure_ingress(size_t src_bytes, int stages, int tensor_boxes, double *bytes_per_cycle_per_sm,
                                double *total_gbs);

/* Force the planner to one named plan for later calls (NULL or "" = choose
 * automatically). Unknown names return BSG_ERR_NO_PLAN.                    */
BSG_API int bsg_force_plan(const char *name);

/* Name of the plan the planner picks for a shape on a GPU with `num_sms`
 * SMs; kind 0 = NVFP4, 1 = FP8, 2 = NVFP4 x dense BF16. Host only (no GPU
 * needed).                                                                 */
BSG_API int bsg_select_plan(int kind, int M, int N, int K, int num_sms,
                    char *name, size_t name_len);

/* Number of kernel launches the last GEMM call on this thread issued
 * (swizzle passes included).                                               */
BSG_API int bsg_last_launch_count(void);

/* Plan name of the last GEMM kernel launched on this thread ("" before any;
 * a static string owned by the library).                                   */
BSG_API const char *bsg_last_plan_name(void);

/* Human-readable name of a status code.                                    */
BSG_API const char *bsg_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* BSGEMM_H */
