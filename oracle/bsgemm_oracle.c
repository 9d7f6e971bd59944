/*
 * CPU oracle for the block-scaled low-precision GEMM
 *
 *     D = alpha * (A (.) sA) (B (.) sB)^T      (FP32 accumulate, BF16 output)
 *
 * TEST INFRASTRUCTURE. This is the plain, slow, obviously correct definition
 * that the CUDA library is checked against. Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg load it; the library never does.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it follows:
 *  - "Together AI Ports ThunderKittens GEMM Kernels to NVIDIA Vera Rubin
 *    NVL72", introduction and "Building the GEMM": NVFP4 and FP8 GEMMs whose
 *    tensor-core MMA consumes block scaling factors beside the operands.
 *  - The operation itself: A and B hold E2M1 codes packed two per byte along
 *    K, one E4M3 scale per 16 consecutive K elements, an FP32 global alpha,
 *    FP32 accumulation and BF16 output; the FP8 variant takes E4M3 operands
 *    with per-tensor FP32 scales.
 *  - "Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
 *    Tensor-Memory Failures", section "The matrix also compared Triton with a
 *    reference implementation": the GPU output is compared with a reference
 *    implementation under a format-specific tolerance.
 *  - "Triton #11171 ...": a shared NVFP4 quantisation step in front of the
 *    GEMM; written out here as the two-level scheme described above
 *    bso_nvfp4_quantize.
 *  - Element formats (the pages name them but do not define them): E2M1 as in
 *    the OCP Microscaling Formats (MX) v1.0 specification (FP4 element type),
 *    E4M3 as in the OCP 8-bit Floating Point (OFP8) specification ("E4M3",
 *    no infinities, S.1111.111 is NaN).
 *
 * Readings where the sources are silent:
 *  - element 2i of a packed row sits in bits 0..3 of byte i, element 2i+1 in
 *    bits 4..7;
 *  - T (the magnitude sum in the tolerance) includes the scales and alpha, so
 *    it is in output units;
 *  - the sum runs in double in natural k order, block by block; it is rounded
 *    once, to BF16 with round-to-nearest-even.
 *
 * Parity pins for every function here live in tests/test_oracle.py.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Element decoders                                                          */
/* ------------------------------------------------------------------------ */

/* E2M1 (4 bits): sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Exponent field 0 is subnormal: value = mantissa * 0.5.
 * Otherwise value = 2^(e-1) * (1 + m/2).                                    */
double bso_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double v;
#ifdef BSO_MUTANT_E2M1_BIAS0
    /* planted mistake for the negative-control tests: exponent bias 0 */
    v = (e == 0) ? m * 0.5 : ldexp(1.0 + m * 0.5, (int)e);
#else
    v = (e == 0) ? m * 0.5 : ldexp(1.0 + m * 0.5, (int)e - 1);
#endif
#ifdef BSO_MUTANT_E2M1_NOSIGN
    s = 0;
#endif
    return s ? -v : v;
}

/* E4M3 (8 bits): sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0.
 * Exponent field 0 is subnormal: value = m/8 * 2^-6. S.1111.111 is NaN;
 * there are no infinities, so S.1111.110 = 448 is the largest magnitude.   */
double bso_e4m3(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double v;
    if (e == 15u && m == 7u)
        return NAN;
#ifdef BSO_MUTANT_E4M3_BIAS8
    v = (e == 0) ? ldexp((double)m, -10) : ldexp(1.0 + m / 8.0, (int)e - 8);
#else
    v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, (int)e - 7);
#endif
    return s ? -v : v;
}

/* Round a double to BF16 (8 exponent bits, bias 127, 7 fraction bits) with
 * round-to-nearest, ties-to-even, in ONE rounding step. Returns the bits.
 * Values whose rounded magnitude reaches 2^128 become infinities.           */
uint16_t bso_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);

    int e2;
    (void)frexp(a, &e2);          /* a in [2^(e2-1), 2^e2)                  */
    int lead = e2 - 1;            /* exponent of the leading bit            */
    int ulp_exp = (lead < -126 ? -126 : lead) - 7;  /* BF16 spacing here    */
    double q = ldexp(a, -ulp_exp);                  /* exact (power of two) */

    /* explicit round-half-to-even of q to an integer */
    double fl = floor(q);
    double frac = q - fl;         /* exact: q < 2^9 in magnitude            */
    double r = fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
        r = fl + 1.0;

    if (lead < -126) {
        /* subnormal range: r counts units of 2^-133, 0..128; r == 128 is
         * the smallest normal, whose bit pattern is also 128.              */
        return (uint16_t)(sign | (uint16_t)r);
    }
    /* normal range: r in [128, 256]; 256 carries into the exponent         */
    if (r == 256.0) {
        r = 128.0;
        lead += 1;
    }
    int ef = lead + 127;
    if (ef >= 255)
        return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)(ef << 7) | (uint16_t)(r - 128.0));
}

/* ------------------------------------------------------------------------ */
/* Packed-operand access                                                     */
/* ------------------------------------------------------------------------ */

/* K-th E2M1 code of a packed row (two codes per byte along K).
 * Swapping the nibble order of BOTH operands permutes k inside each pair the
 * same way for A and B and leaves every dot product unchanged; the order is
 * observable only when the two operands disagree, which is what the planted
 * variant below does (A read high-nibble-first, B low-nibble-first).       */
static unsigned nib(const uint8_t *row, int k)
{
    uint8_t byte = row[k >> 1];
    return (k & 1) ? (byte >> 4) : (byte & 15u);
}

static unsigned nib_a(const uint8_t *row, int k)
{
#ifdef BSO_MUTANT_SWAP_NIBBLES_A
    return nib(row, k ^ 1);
#else
    return nib(row, k);
#endif
}

/* ------------------------------------------------------------------------ */
/* Threaded driver: output rows are split evenly across threads             */
/* ------------------------------------------------------------------------ */

typedef struct {
    int kind;                     /* 0 = NVFP4, 1 = FP8, 2 = NVFP4 x BF16, 3 = NVFP4 x FP16 */
    int M, N, K;
    const uint8_t *A, *sfA, *B, *sfB;
    double scale;                 /* alpha (NVFP4) or alpha*sA*sB (FP8)       */
    const float *bias;            /* [N] added per output column, or NULL    */
    const float *gamma;           /* [M] per-row multiplier, or NULL         */
    const int32_t *rows;
    int nrows;
    const int32_t *cols;
    int ncols;
    double *S, *T;
    uint16_t *D;
    int r0, r1;                   /* this worker's output-row range          */
    double e2m1_tab[16];
    double e4m3_tab[256];
} job_t;

/* One output element of the NVFP4 GEMM, by the definition:
 *   S = alpha * sum_b  e4m3(sfA[i][b]) * e4m3(sfB[j][b])
 *                    * sum_{t<16} e2m1(A[i][16b+t]) * e2m1(B[j][16b+t])
 *   T = |alpha| * sum_b |sA*sB| * sum_t |a*b|                              */
static void nvfp4_element(const job_t *jb, int i, int j, double *S, double *T)
{
    const int K = jb->K, nb = K / 16;
    const uint8_t *ra = jb->A + (size_t)i * (size_t)(K / 2);
    const uint8_t *rb = jb->B + (size_t)j * (size_t)(K / 2);
    const uint8_t *sa = jb->sfA + (size_t)i * (size_t)nb;
    const uint8_t *sb = jb->sfB + (size_t)j * (size_t)nb;
    double s = 0.0, t = 0.0;
#ifdef BSO_MUTANT_DROP_LAST_BLOCK
    for (int b = 0; b < nb - 1; ++b) {
#else
    for (int b = 0; b < nb; ++b) {
#endif
        double blk = 0.0, blk_abs = 0.0;
        for (int u = 0; u < 16; ++u) {
            int k = 16 * b + u;
#ifdef BSO_MUTANT_TRANSPOSE_B
            /* reads B as if it were stored [K][N] (square shapes only) */
            double p = jb->e2m1_tab[nib_a(ra, k)]
                       * jb->e2m1_tab[nib(jb->B + (size_t)k * (size_t)(K / 2), j)];
            (void)rb;
#else
            double p = jb->e2m1_tab[nib_a(ra, k)] * jb->e2m1_tab[nib(rb, k)];
#endif
            blk += p;
            blk_abs += fabs(p);
        }
#ifdef BSO_MUTANT_DROP_SFB
        double sc = jb->e4m3_tab[sa[b]];
        (void)sb;
#else
        double sc = jb->e4m3_tab[sa[b]] * jb->e4m3_tab[sb[b]];
#endif
        s += sc * blk;
        t += fabs(sc) * blk_abs;
    }
    *S = jb->scale * s;
    *T = fabs(jb->scale) * t;
}

/* One output element of the FP8 GEMM:
 *   S = alpha*sA*sB * sum_k e4m3(A[i][k]) * e4m3(B[j][k])                  */
static void fp8_element(const job_t *jb, int i, int j, double *S, double *T)
{
    const int K = jb->K;
    const uint8_t *ra = jb->A + (size_t)i * (size_t)K;
    const uint8_t *rb = jb->B + (size_t)j * (size_t)K;
    double s = 0.0, t = 0.0;
    for (int k = 0; k < K; ++k) {
        double p = jb->e4m3_tab[ra[k]] * jb->e4m3_tab[rb[k]];
        s += p;
        t += fabs(p);
    }
    *S = jb->scale * s;
    *T = fabs(jb->scale) * t;
}

/* Epilogue variants ("Triton #11171 ...", section "The ordinary variants
 * also exercise the shared bias route" and the two sections before it):
 * the matmul result gets the shared bias added, is multiplied by the per-row
 * gamma, and (outside this function) its row is written to a scattered
 * position. Reading: bias is indexed by output column j, gamma by logical
 * output row i, bias comes before gamma:
 *     S' = gamma[i] * (S + bias[j]),   T' = |gamma[i]| * (T + |bias[j]|)
 * Both are FP32 inputs widened exactly to double; still one rounding.      */
static void epilogue(const job_t *jb, int i, int j, double *S, double *T)
{
    if (jb->bias) {
#ifdef BSO_MUTANT_EPI_BIAS_BY_ROW
        double b = (double)jb->bias[i < jb->N ? i : 0];
#else
        double b = (double)jb->bias[j];
#endif
#ifdef BSO_MUTANT_EPI_GAMMA_FIRST
        if (jb->gamma) {
            *S *= (double)jb->gamma[i];
            *T *= fabs((double)jb->gamma[i]);
        }
        *S += b;
        *T += fabs(b);
        return;
#else
        *S += b;
        *T += fabs(b);
#endif
    }
    if (jb->gamma) {
        double g = (double)jb->gamma[i];
        *S *= g;
        *T *= fabs(g);
    }
}

/* IEEE binary16 bit pattern -> its exact value: sign, 5 exponent bits (bias
 * 15, field 0 subnormal: m * 2^-24), 10 fraction bits; field 31 is Inf/NaN. */
static double f16_value(uint16_t h)
{
    const int sgn = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
#ifdef BSO_MUTANT_F16_BIAS16
        v = ldexp(1024.0 + (double)m, e - 26);
#else
        v = ldexp(1024.0 + (double)m, e - 25);
#endif
    return sgn ? -v : v;
}

/* BF16 bit pattern -> its exact value (BF16 is the top half of binary32). */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One output element of the NVFP4 x dense GEMM: A block-scaled E2M1, B plain
 * BF16 (kind 2) or FP16 (kind 3) values (uint16 bit patterns, [N][K]):
 *   S = alpha * sum_b sA[i][b] * sum_t e2m1(A[i][16b+t]) * B[j][16b+t]    */
static void dense_element(const job_t *jb, int i, int j, double *S, double *T)
{
    const int K = jb->K, nb = K / 16;
    const uint8_t *ra = jb->A + (size_t)i * (size_t)(K / 2);
    const uint8_t *sa = jb->sfA + (size_t)i * (size_t)nb;
    const uint16_t *rb = (const uint16_t *)(const void *)jb->B + (size_t)j * (size_t)K;
    double s = 0.0, t = 0.0;
    for (int b = 0; b < nb; ++b) {
        double blk = 0.0, blk_abs = 0.0;
        for (int u = 0; u < 16; ++u) {
            int k = 16 * b + u;
            double p = jb->e2m1_tab[nib_a(ra, k)] * (jb->kind == 3 ? f16_value(rb[k]) : bf16_value(rb[k]));
            blk += p;
            blk_abs += fabs(p);
        }
#ifdef BSO_MUTANT_DENSE_DROP_SFA
        double sc = 1.0;
        (void)sa;
#else
        double sc = jb->e4m3_tab[sa[b]];
#endif
        s += sc * blk;
        t += fabs(sc) * blk_abs;
    }
    *S = jb->scale * s;
    *T = fabs(jb->scale) * t;
}

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    for (int r = jb->r0; r < jb->r1; ++r) {
        int i = jb->rows ? jb->rows[r] : r;
        for (int c = 0; c < jb->ncols; ++c) {
            int j = jb->cols ? jb->cols[c] : c;
            double S, T;
            if (jb->kind == 0)
                nvfp4_element(jb, i, j, &S, &T);
            else if (jb->kind == 1)
                fp8_element(jb, i, j, &S, &T);
            else
                dense_element(jb, i, j, &S, &T);   /* kinds 2 and 3 */
            epilogue(jb, i, j, &S, &T);
            size_t o = (size_t)r * (size_t)jb->ncols + (size_t)c;
            if (jb->S) jb->S[o] = S;
            if (jb->T) jb->T[o] = T;
            if (jb->D) jb->D[o] = bso_bf16_rne(S);
        }
    }
    return NULL;
}

static int run(job_t *proto, int nthreads)
{
    for (int c = 0; c < 16; ++c)
        proto->e2m1_tab[c] = bso_e2m1((unsigned)c);
    for (int c = 0; c < 256; ++c)
        proto->e4m3_tab[c] = bso_e4m3((unsigned)c);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > proto->nrows)
        nthreads = proto->nrows > 0 ? proto->nrows : 1;
    if (nthreads > 1024)
        nthreads = 1024;
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -2;
    }
    int started = 0;
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = *proto;
        jobs[w].r0 = (int)((long long)proto->nrows * w / nthreads);
        jobs[w].r1 = (int)((long long)proto->nrows * (w + 1) / nthreads);
        if (nthreads == 1 || pthread_create(&th[w], NULL, worker, &jobs[w]) != 0) {
            worker(&jobs[w]);
            th[w] = 0;
        } else {
            ++started;
        }
    }
    for (int w = 0; w < nthreads; ++w)
        if (th[w])
            pthread_join(th[w], NULL);
    (void)started;
    free(jobs);
    free(th);
    return 0;
}

static int check_sel(const int32_t *sel, int n, int lim)
{
    if (!sel)
        return 0;
    for (int q = 0; q < n; ++q)
        if (sel[q] < 0 || sel[q] >= lim)
            return -1;
    return 0;
}

/* NVFP4 GEMM over the selected rows x cols of D (rows/cols NULL = all).
 * A: uint8[M][K/2], sfA: uint8[M][K/16] row-major E4M3, B: uint8[N][K/2],
 * sfB: uint8[N][K/16]; bias float[N] and gamma float[M] may be NULL (see
 * epilogue above). Outputs are [nrows][ncols]; any may be NULL.
 * Returns 0, or -1 for bad sizes.                                          */
int bso_nvfp4_gemm(int M, int N, int K, const uint8_t *A, const uint8_t *sfA,
                   const uint8_t *B, const uint8_t *sfB, float alpha,
                   const float *bias, const float *gamma,
                   const int32_t *rows, int nrows, const int32_t *cols, int ncols,
                   double *S, double *T, uint16_t *D, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (K % 16) != 0)
        return -1;
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    if (check_sel(rows, nrows, M) || check_sel(cols, ncols, N))
        return -1;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 0;
    jb.M = M; jb.N = N; jb.K = K;
    jb.A = A; jb.sfA = sfA; jb.B = B; jb.sfB = sfB;
    jb.scale = (double)alpha;
    jb.bias = bias; jb.gamma = gamma;
    jb.rows = rows; jb.nrows = nrows; jb.cols = cols; jb.ncols = ncols;
    jb.S = S; jb.T = T; jb.D = D;
    return run(&jb, nthreads);
}

/* FP8 GEMM: A uint8[M][K] E4M3, B uint8[N][K] E4M3; the effective multiplier
 * is the exact double product alpha * sA * sB of the three FP32 values.    */
int bso_fp8_gemm(int M, int N, int K, const uint8_t *A, const uint8_t *B,
                 float alpha, float sA, float sB,
                 const float *bias, const float *gamma,
                 const int32_t *rows, int nrows, const int32_t *cols, int ncols,
                 double *S, double *T, uint16_t *D, int nthreads)
{
    if (M < 0 || N < 0 || K < 0)
        return -1;
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    if (check_sel(rows, nrows, M) || check_sel(cols, ncols, N))
        return -1;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 1;
    jb.M = M; jb.N = N; jb.K = K;
    jb.A = A; jb.B = B;
    jb.scale = (double)alpha * (double)sA * (double)sB;
    jb.bias = bias; jb.gamma = gamma;
    jb.rows = rows; jb.nrows = nrows; jb.cols = cols; jb.ncols = ncols;
    jb.S = S; jb.T = T; jb.D = D;
    return run(&jb, nthreads);
}

/* NVFP4 x dense-BF16 GEMM ("Triton #11171 - Why Two New NVFP4 Test Cases
 * Produced Twelve Tensor-Memory Failures", opening: an NVFP4-scaled
 * activation times a dense BF16 or FP16 operand): A: uint8[M][K/2] E2M1
 * codes with sfA: uint8[M][K/16] E4M3 block scales, B: uint16[N][K] bit
 * patterns, each a plain BF16 value (b_f16 = 0) or IEEE binary16 value
 * (b_f16 = 1); bias / gamma as bso_nvfp4_gemm. The sum runs
 * in double block by block (each product a * sA * b has at most 2 + 4 + 11
 * significant bits, so it is exact), then the epilogue, then one BF16
 * rounding.                                                                 */
int bso_nvfp4_dense_gemm(int M, int N, int K, const uint8_t *A, const uint8_t *sfA, const uint16_t *B,
                         int b_f16, float alpha, const float *bias, const float *gamma,
                         const int32_t *rows, int nrows, const int32_t *cols, int ncols,
                         double *S, double *T, uint16_t *D, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || (K % 16) != 0)
        return -1;
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    if (check_sel(rows, nrows, M) || check_sel(cols, ncols, N))
        return -1;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = b_f16 ? 3 : 2;
    jb.M = M; jb.N = N; jb.K = K;
    jb.A = A; jb.sfA = sfA; jb.B = (const uint8_t *)(const void *)B;
    jb.scale = (double)alpha;
    jb.bias = bias; jb.gamma = gamma;
    jb.rows = rows; jb.nrows = nrows; jb.cols = cols; jb.ncols = ncols;
    jb.S = S; jb.T = T; jb.D = D;
    return run(&jb, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Scale-factor layout consumed by the block-scaled tensor-core MMA          */
/* ------------------------------------------------------------------------ */

/* "Triton #11171 ...", section "Activation-scale swizzling forced the
 * relevant persistent path": the persistent Blackwell kernel reads the scales
 * in a Blackwell-specific layout rewritten in HBM. The layout used here is the
 * tcgen05 block-scale-factor layout of the public PTX ISA: rows are padded to
 * a multiple of 128 and scale columns (K/16) to a multiple of 4; the padded
 * matrix is cut into 128 x 4 blocks of 512 bytes, ordered row-block-major
 * with the column-block index fastest; inside a block, row r and column c go
 * to byte (r % 32) * 16 + (r / 32) * 4 + c. Padding bytes are zero.        */
size_t bso_swizzled_scale_bytes(int rows, int K)
{
    if (rows < 0 || K < 0 || (K % 16) != 0)
        return 0;
    size_t pr = ((size_t)rows + 127u) / 128u * 128u;
    size_t pc = ((size_t)(K / 16) + 3u) / 4u * 4u;
    return pr * pc;
}

int bso_swizzle_scales(int rows, int K, const uint8_t *in, uint8_t *out)
{
    if (rows < 0 || K < 0 || (K % 16) != 0)
        return -1;
    const int cols = K / 16;
    const int pr = (rows + 127) / 128 * 128;
    const int pc = (cols + 3) / 4 * 4;
    const int ncb = pc / 4;
    for (int r = 0; r < pr; ++r) {
        for (int c = 0; c < pc; ++c) {
            size_t blk = (size_t)(r / 128) * (size_t)ncb + (size_t)(c / 4);
            int rr = r % 128;
#ifdef BSO_MUTANT_SWIZZLE_ROWMAJOR_BLOCK
            size_t off = blk * 512u + (size_t)rr * 4u + (size_t)(c % 4);
#else
            size_t off = blk * 512u + (size_t)(rr % 32) * 16u + (size_t)(rr / 32) * 4u
                         + (size_t)(c % 4);
#endif
            out[off] = (r < rows && c < cols) ? in[(size_t)r * (size_t)cols + (size_t)c] : 0u;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped (ragged, routed) NVFP4 GEMM                                        */
/* ------------------------------------------------------------------------ */

/* "Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
 * Tensor-Memory Failures", section "Ragged mode added routing rather than a
 * plain matrix": routed activation rows form expert slices, and each slice
 * is multiplied by the dense right-hand side of its own slice. Written out:
 * the rows of A are grouped into E consecutive slices, slice e being rows
 * [offs[e], offs[e+1]); for those rows
 *     S[i][j] = alpha * sum_b sA[i][b] sB_e[j][b] sum_t a(i, 16b+t) b_e(j, 16b+t)
 * followed by the epilogue of bso_nvfp4_gemm with bias_e = bias + e*N and
 * gamma[i]. That is: each slice is an ordinary NVFP4 GEMM of its own.
 *   A: uint8[M][K/2], sfA: uint8[M][K/16]   (rows grouped by slice)
 *   B: uint8[E][N][K/2], sfB: uint8[E][N][K/16]
 *   offs: int32[E+1] with offs[0] = 0, nondecreasing, offs[E] = M
 *   bias: float[E][N] or NULL; gamma: float[M] or NULL
 * Outputs are [M][N] in row order; any may be NULL. Returns 0, or -1 for
 * bad sizes or offsets.                                                     */
int bso_nvfp4_grouped_gemm(int E, int M, int N, int K, const uint8_t *A, const uint8_t *sfA,
                           const uint8_t *B, const uint8_t *sfB, const int32_t *offs, float alpha,
                           const float *bias, const float *gamma, double *S, double *T, uint16_t *D,
                           int nthreads)
{
    if (E < 1 || M < 0 || N < 0 || K < 0 || (K % 16) != 0 || !offs)
        return -1;
    if (offs[0] != 0 || offs[E] != M)
        return -1;
    for (int e = 0; e < E; ++e)
        if (offs[e + 1] < offs[e])
            return -1;
    const size_t arow = (size_t)(K / 2), srow = (size_t)(K / 16);
    for (int e = 0; e < E; ++e) {
        const int r0 = offs[e], rows = offs[e + 1] - offs[e];
        if (rows == 0)
            continue;
#ifdef BSO_MUTANT_GROUP_SHIFT
        const int be = (e + 1) % E;      /* planted: the next slice's right-hand side */
#else
        const int be = e;
#endif
        const size_t o = (size_t)r0 * (size_t)N;
        int rc = bso_nvfp4_gemm(rows, N, K, A + (size_t)r0 * arow, sfA + (size_t)r0 * srow,
                                B + (size_t)be * (size_t)N * arow, sfB + (size_t)be * (size_t)N * srow,
                                alpha, bias ? bias + (size_t)e * (size_t)N : NULL,
                                gamma ? gamma + r0 : NULL, NULL, 0, NULL, 0,
                                S ? S + o : NULL, T ? T + o : NULL, D ? D + o : NULL, nthreads);
        if (rc != 0)
            return rc;
    }
    return 0;
}

/* Scale layout of a grouped A: the swizzled layout above, applied to each
 * slice on its own, the slices' 128-row blocks concatenated in slice order
 * -- slice e starts at 128-row block sum_{e'<e} ceil(rows_e' / 128), so
 * every tile of 128 rows of one slice reads one block row. The buffer holds
 * (ceil(M/128) + E) block rows (an upper bound of the sum, since sizes
 * are not known on the host); block rows past the slices' are zero.       */
size_t bso_grouped_scale_bytes(int E, int M, int K)
{
    if (E < 1 || M < 0 || K < 0 || (K % 16) != 0)
        return 0;
    size_t pc = ((size_t)(K / 16) + 3u) / 4u * 4u;
    return ((size_t)(M + 127) / 128u + (size_t)E) * 128u * pc;
}

int bso_swizzle_scales_grouped(int E, int M, int K, const int32_t *offs, const uint8_t *in, uint8_t *out)
{
    if (E < 1 || M < 0 || K < 0 || (K % 16) != 0 || !offs || offs[0] != 0 || offs[E] != M)
        return -1;
    for (int e = 0; e < E; ++e)
        if (offs[e + 1] < offs[e])
            return -1;
    const size_t cols = (size_t)(K / 16);
    const size_t block_row_bytes = 128u * ((cols + 3u) / 4u * 4u);
    memset(out, 0, bso_grouped_scale_bytes(E, M, K));
    size_t brow = 0;
    for (int e = 0; e < E; ++e) {
        const int rows = offs[e + 1] - offs[e];
        if (bso_swizzle_scales(rows, K, in + (size_t)offs[e] * cols, out + brow * block_row_bytes) != 0)
            return -1;
        brow += ((size_t)rows + 127u) / 128u;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Two-level NVFP4 quantisation: BF16 -> E2M1 codes + E4M3 block scales      */
/* ------------------------------------------------------------------------ */

/* "Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
 * Tensor-Memory Failures" names a shared NVFP4 quantisation step in front of
 * the block-scaled GEMM; the pages give no formula. The scheme written out
 * here is the plainest reading:
 *
 *   amax  = max |x| over the whole tensor                    (exact)
 *   s_g   = 2688 / amax   (448 * 6; 1 when amax == 0)         (FP32, rounded once)
 *   per block of 16 consecutive elements along K:
 *     bmax  = max |x| over the block                         (exact)
 *     sc    = (bmax / 6) * s_g                               (FP32, two roundings, this order)
 *     scale = nearest E4M3 (ties to even), saturated at 448  (positive, sign bit 0)
 *     if scale decodes to 0: every code of the block is 0
 *     else code_k = nearest E2M1 (ties to even), saturated at 6, of
 *                   (x_k * s_g) / scale                      (FP32, two roundings, this order)
 *                   with the sign of that quotient (so a tiny negative gives -0, code 8)
 *
 * so that the largest |x| of the tensor lands on 6 * 448. Each decision that
 * picks a code is taken in FP32 with every operation rounded once, in the
 * order above: the precision of the GPU kernel, so that both sides decide
 * ties identically. Inputs must be finite. Element 2i of a row goes to the
 * low nibble of byte i, as everywhere in this file.                         */

/* Nearest E4M3 code (ties to the even code) of v >= 0, saturated at 448:
 * binary search over the positive finite codes 0x00..0x7E, whose decoded
 * values rise with the code. */
static unsigned e4m3_nearest(float v)
{
    if (!(v > 0.0f))
        return 0u;
#ifdef BSO_MUTANT_Q_E4M3_CEIL
    for (unsigned c = 0; c < 0x7Fu; ++c)
        if (bso_e4m3(c) >= (double)v)
            return c;
    return 0x7Eu;
#endif
    if ((double)v >= bso_e4m3(0x7Eu))
        return 0x7Eu;
    unsigned lo = 0u, hi = 0x7Eu;            /* decode(lo) <= v < decode(hi) */
    while (hi - lo > 1u) {
        unsigned mid = (lo + hi) / 2u;
        if (bso_e4m3(mid) <= (double)v)
            lo = mid;
        else
            hi = mid;
    }
    double dl = (double)v - bso_e4m3(lo), dh = bso_e4m3(hi) - (double)v;
    if (dl < dh)
        return lo;
    if (dh < dl)
        return hi;
    return (lo & 1u) ? hi : lo;              /* tie: the code with an even mantissa */
}

/* Nearest E2M1 code (ties to the even code) of y, saturated at +-6; the
 * sign bit is the sign of y (so -0.0 and tiny negatives give code 8). */
static unsigned e2m1_nearest(float y)
{
    const unsigned s = signbit(y) ? 8u : 0u;
    const double m = fabs((double)y);
    unsigned best = 0u;
    double bd = -1.0;
    for (unsigned c = 0; c < 8u; ++c) {
        double d = fabs(bso_e2m1(c) - m);
#ifdef BSO_MUTANT_Q_TIES_AWAY
        if (bd < 0.0 || d < bd || (d == bd && bso_e2m1(c) > bso_e2m1(best))) {
#else
        if (bd < 0.0 || d < bd || (d == bd && (c & 1u) == 0u && (best & 1u) != 0u)) {
#endif
            best = c;
            bd = d;
        }
    }
    return s | best;
}

static float bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* X: BF16 bit patterns uint16[rows][K]; outputs packed uint8[rows][K/2],
 * row-major scales uint8[rows][K/16], and the tensor's amax and s_g. */
int bso_nvfp4_quantize(int rows, int K, const uint16_t *X, uint8_t *packed, uint8_t *sf,
                       float *amax_out, float *sg_out)
{
    if (rows < 0 || K < 16 || (K % 16) != 0)
        return -1;
    float amax = 0.0f;
    for (size_t i = 0; i < (size_t)rows * (size_t)K; ++i) {
        float a = fabsf(bf16_to_float(X[i]));
        if (a > amax)
            amax = a;
    }
    const float s_g = amax > 0.0f ? 2688.0f / amax : 1.0f;
    *amax_out = amax;
    *sg_out = s_g;
    const int nb = K / 16;
    for (int r = 0; r < rows; ++r) {
        const uint16_t *xr = X + (size_t)r * (size_t)K;
        uint8_t *pr = packed + (size_t)r * (size_t)(K / 2);
        for (int b = 0; b < nb; ++b) {
            float bmax = 0.0f;
            for (int k = 0; k < 16; ++k) {
                float a = fabsf(bf16_to_float(xr[16 * b + k]));
                if (a > bmax)
                    bmax = a;
            }
            const float sc = (bmax / 6.0f) * s_g;
            const unsigned scode = e4m3_nearest(sc);
            sf[(size_t)r * (size_t)nb + (size_t)b] = (uint8_t)scode;
            const float sv = (float)bso_e4m3(scode);
            unsigned codes[16];
            for (int k = 0; k < 16; ++k) {
                if (sv == 0.0f) {
                    codes[k] = 0u;
                    continue;
                }
#ifdef BSO_MUTANT_Q_NO_SG
                const float y = bf16_to_float(xr[16 * b + k]) / sv;
#else
                const float y = (bf16_to_float(xr[16 * b + k]) * s_g) / sv;
#endif
                codes[k] = e2m1_nearest(y);
            }
            for (int k = 0; k < 16; k += 2) {
#ifdef BSO_MUTANT_Q_SWAP_NIBBLES
                pr[8 * b + k / 2] = (uint8_t)(codes[k + 1] | (codes[k] << 4));
#else
                pr[8 * b + k / 2] = (uint8_t)(codes[k] | (codes[k + 1] << 4));
#endif
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Freivalds' check of a whole product without forming it                   */
/* ------------------------------------------------------------------------ */

/* R. Freivalds, "Probabilistic machines can use less running time" (IFIP
 * Congress 1977): a correct D = alpha * Adeq Bdeq^T satisfies, for every
 * vector x of length N,
 *     D x = alpha * Adeq (Bdeq^T x),
 * and the right-hand side costs O((M + N) K) instead of the product's
 * O(M N K). So every element of a full-size result (16384^3: hours of the
 * element-wise definition above) enters a check that takes seconds. Adeq /
 * Bdeq hold the decoded elements times their block scales (NVFP4) or the
 * decoded E4M3 elements (FP8, whose per-tensor scales fold into `scale`).
 *
 * For each of the nv vectors x_q (int8[nv][N]) this returns
 *     v_q[k]   = sum_j bdeq[j][k] * x_q[j]
 *     y[q][i]  = scale * sum_k adeq[i][k] * v_q[k]
 *     g[q][i]  = |scale| * sum_k |adeq[i][k]| * |v_q[k]|
 * and, for the tolerance, per row i
 *     tsum[i]  = |scale| * sum_k |adeq[i][k]| * sum_j |bdeq[j][k]|
 *              = sum_j T[i][j]            (T of the element-wise oracle)
 *     t2[i]    = scale^2 * (sum_k adeq[i][k]^2) * (sum_j sum_k bdeq[j][k]^2)
 *              >= sum_j T[i][j]^2         (Cauchy-Schwarz on each T[i][j])
 * Exactness: NVFP4 elements are multiples of 2^-10 below 2^12 in magnitude,
 * E4M3 ones multiples of 2^-9 below 2^9; with |x| <= 127 and N < 2^20 every
 * v_q[k] and every sum_j |bdeq[j][k]| is an integer multiple of that unit
 * below 2^53 of them, so exact in double whatever the summation order. y,
 * tsum and t2 carry the rounding of a K-term double sum; g bounds y's.     */

typedef struct {
    int kind;                     /* 0 = NVFP4, 1 = FP8 */
    int is_b;                     /* decoding B (the first phase)          */
    int N, K, nv;
    const uint8_t *X, *sfX;       /* the operand of this phase             */
    const int8_t *x;              /* [nv][N] (B phase)                     */
    const double *v, *w;          /* [nv][K], [K]   (A phase)              */
    double scale;
    double *pv, *pw, *pb2;        /* B phase: this worker's partial sums   */
    double *y, *g, *tsum, *a2;    /* A phase outputs, [nv][M] / [M]        */
    int M;
    int r0, r1;
    double e2m1_tab[16];
    double e4m3_tab[256];
} fv_job_t;

/* Row r of an operand, decoded with its block scales into out[K]. */
static void fv_decode_row(const fv_job_t *jb, int r, double *out)
{
    const int K = jb->K;
    if (jb->kind == 0) {
        const uint8_t *row = jb->X + (size_t)r * (size_t)(K / 2);
        const uint8_t *sf = jb->sfX + (size_t)r * (size_t)(K / 16);
#ifdef BSO_MUTANT_FV_DROP_SFB
        if (jb->is_b) {
            for (int k = 0; k < K; ++k)
                out[k] = jb->e2m1_tab[nib(row, k)];
            return;
        }
#endif
        for (int k = 0; k < K; ++k)
            out[k] = jb->e2m1_tab[nib(row, k)] * jb->e4m3_tab[sf[k / 16]];
    } else {
        const uint8_t *row = jb->X + (size_t)r * (size_t)K;
        for (int k = 0; k < K; ++k)
            out[k] = jb->e4m3_tab[row[k]];
    }
}

/* B phase: rows [r0, r1) of B into this worker's partial v, w, b2. */
static void *fv_b_worker(void *arg)
{
    fv_job_t *jb = (fv_job_t *)arg;
    const int K = jb->K, nv = jb->nv;
    double *row = (double *)malloc(sizeof(double) * (size_t)K);
    if (!row)
        return (void *)1;
    for (int j = jb->r0; j < jb->r1; ++j) {
        fv_decode_row(jb, j, row);
        for (int k = 0; k < K; ++k) {
#ifdef BSO_MUTANT_FV_TSUM_SIGNED
            jb->pw[k] += row[k];
#else
            jb->pw[k] += fabs(row[k]);
#endif
            *jb->pb2 += row[k] * row[k];
        }
        for (int q = 0; q < nv; ++q) {
#ifdef BSO_MUTANT_FV_X_REVERSED
            const double xq = (double)jb->x[(size_t)q * (size_t)jb->N + (size_t)(jb->N - 1 - j)];
#else
            const double xq = (double)jb->x[(size_t)q * (size_t)jb->N + (size_t)j];
#endif
            double *vq = jb->pv + (size_t)q * (size_t)K;
            if (xq != 0.0)
                for (int k = 0; k < K; ++k)
                    vq[k] += row[k] * xq;
        }
    }
    free(row);
    return NULL;
}

/* A phase: rows [r0, r1) of A against the finished v and w. */
static void *fv_a_worker(void *arg)
{
    fv_job_t *jb = (fv_job_t *)arg;
    const int K = jb->K, nv = jb->nv, M = jb->M;
    double *row = (double *)malloc(sizeof(double) * (size_t)K);
    if (!row)
        return (void *)1;
    for (int i = jb->r0; i < jb->r1; ++i) {
        fv_decode_row(jb, i, row);
        double t = 0.0, s2 = 0.0;
        for (int k = 0; k < K; ++k) {
            t += fabs(row[k]) * jb->w[k];
            s2 += row[k] * row[k];
        }
        jb->tsum[i] = fabs(jb->scale) * t;
        jb->a2[i] = s2;
        for (int q = 0; q < nv; ++q) {
            const double *vq = jb->v + (size_t)q * (size_t)K;
            double s = 0.0, a = 0.0;
            for (int k = 0; k < K; ++k) {
                s += row[k] * vq[k];
                a += fabs(row[k]) * fabs(vq[k]);
            }
            jb->y[(size_t)q * (size_t)M + (size_t)i] = jb->scale * s;
            jb->g[(size_t)q * (size_t)M + (size_t)i] = fabs(jb->scale) * a;
        }
    }
    free(row);
    return NULL;
}

/* Runs `fn` over rows [0, rows) split across nthreads copies of proto. */
static int fv_run(fv_job_t *proto, int rows, int nthreads, void *(*fn)(void *), fv_job_t **jobs_out,
                  int *njobs)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > rows)
        nthreads = rows > 0 ? rows : 1;
    if (nthreads > 256)
        nthreads = 256;
    fv_job_t *jobs = (fv_job_t *)calloc((size_t)nthreads, sizeof(fv_job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int *started = (int *)calloc((size_t)nthreads, sizeof(int));
    *jobs_out = NULL;
    *njobs = 0;
    if (!jobs || !th || !started) {
        free(jobs);
        free(th);
        free(started);
        return -2;
    }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].r0 = (int)((long long)rows * t / nthreads);
        jobs[t].r1 = (int)((long long)rows * (t + 1) / nthreads);
    }
    if (fn == fv_b_worker) {
        const size_t nvk = (size_t)proto->nv * (size_t)proto->K;
        for (int t = 0; t < nthreads; ++t) {
            jobs[t].pv = (double *)calloc(nvk + (size_t)proto->K + 1u, sizeof(double));
            if (!jobs[t].pv)
                rc = -2;
            else {
                jobs[t].pw = jobs[t].pv + nvk;
                jobs[t].pb2 = jobs[t].pw + proto->K;
            }
        }
    }
    if (rc == 0) {
        for (int t = 0; t < nthreads; ++t)
            started[t] = nthreads > 1 && pthread_create(&th[t], NULL, fn, &jobs[t]) == 0;
        for (int t = 0; t < nthreads; ++t) {
            void *ret = NULL;
            if (started[t])
                pthread_join(th[t], &ret);
            else
                ret = fn(&jobs[t]);
            if (ret)
                rc = -2;
        }
    }
    free(th);
    free(started);
    *jobs_out = jobs;
    *njobs = nthreads;
    return rc;
}

static int fv_check(fv_job_t *proto, int M, const uint8_t *A, const uint8_t *sfA, const uint8_t *B,
                    const uint8_t *sfB, double *y, double *g, double *tsum, double *t2, int nthreads)
{
    for (int c = 0; c < 16; ++c)
        proto->e2m1_tab[c] = bso_e2m1((unsigned)c);
    for (int c = 0; c < 256; ++c)
        proto->e4m3_tab[c] = bso_e4m3((unsigned)c);
    const int K = proto->K, nv = proto->nv, N = proto->N;
    const size_t nvk = (size_t)nv * (size_t)K;
    double *v = (double *)calloc(nvk + (size_t)K, sizeof(double));
    double *a2 = (double *)calloc((size_t)(M > 0 ? M : 1), sizeof(double));
    if (!v || !a2) {
        free(v);
        free(a2);
        return -2;
    }
    double *w = v + nvk;
    double b2 = 0.0;

    /* B phase: partial sums per worker, added afterwards (exact: see above) */
    proto->X = B;
    proto->sfX = sfB;
    proto->is_b = 1;
    fv_job_t *jobs = NULL;
    int nj = 0;
    int rc = fv_run(proto, N, nthreads, fv_b_worker, &jobs, &nj);
    for (int t = 0; t < nj; ++t) {
        if (jobs[t].pv) {
            for (size_t u = 0; u < nvk; ++u)
                v[u] += jobs[t].pv[u];
            for (int k = 0; k < K; ++k)
                w[k] += jobs[t].pw[k];
            b2 += *jobs[t].pb2;
            free(jobs[t].pv);
        }
    }
    free(jobs);
    if (rc != 0) {
        free(v);
        free(a2);
        return rc;
    }

    /* A phase */
    proto->X = A;
    proto->sfX = sfA;
    proto->is_b = 0;
    proto->v = v;
    proto->w = w;
    proto->y = y;
    proto->g = g;
    proto->tsum = tsum;
    proto->a2 = a2;
    proto->M = M;
    rc = fv_run(proto, M, nthreads, fv_a_worker, &jobs, &nj);
    free(jobs);
    if (rc == 0)
        for (int i = 0; i < M; ++i)
            t2[i] = proto->scale * proto->scale * a2[i] * b2;
    free(v);
    free(a2);
    return rc;
}

/* NVFP4: A uint8[M][K/2], sfA uint8[M][K/16], B uint8[N][K/2], sfB
 * uint8[N][K/16] (row-major scales); x int8[nv][N]; outputs y, g [nv][M],
 * tsum, t2 [M]. Returns 0, -1 for bad sizes, -2 if memory ran out.        */
int bso_nvfp4_freivalds(int M, int N, int K, const uint8_t *A, const uint8_t *sfA, const uint8_t *B,
                        const uint8_t *sfB, float alpha, const int8_t *x, int nv, double *y, double *g,
                        double *tsum, double *t2, int nthreads)
{
    if (M < 1 || N < 1 || K < 16 || (K % 16) != 0 || nv < 1 || N >= (1 << 20))
        return -1;
    fv_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 0;
    jb.N = N;
    jb.K = K;
    jb.nv = nv;
    jb.x = x;
    jb.scale = (double)alpha;
    return fv_check(&jb, M, A, sfA, B, sfB, y, g, tsum, t2, nthreads);
}

/* FP8: A uint8[M][K], B uint8[N][K] E4M3; the multiplier is the double
 * product alpha * sA * sB, as in bso_fp8_gemm.                              */
int bso_fp8_freivalds(int M, int N, int K, const uint8_t *A, const uint8_t *B, float alpha, float sA, float sB,
                      const int8_t *x, int nv, double *y, double *g, double *tsum, double *t2, int nthreads)
{
    if (M < 1 || N < 1 || K < 1 || nv < 1 || N >= (1 << 20))
        return -1;
    fv_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 1;
    jb.N = N;
    jb.K = K;
    jb.nv = nv;
    jb.x = x;
    jb.scale = (double)alpha * (double)sA * (double)sB;
    return fv_check(&jb, M, A, NULL, B, NULL, y, g, tsum, t2, nthreads);
}
