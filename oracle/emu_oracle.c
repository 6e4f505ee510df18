/*
 * emu_oracle.c -- plain CPU oracle for FP32 GEMM emulated with BF16x9 and TF32x3.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (cited by title and section):
 *   [Blog] "Unlocking Tensor Core performance for machine-learning interatomic
 *          potentials" (NVIDIA technical blog), sections
 *          "How Tensor Core FP32 bridges the hardware gap" (Fig. 1, Fig. 2, Eq. 1),
 *          "TF32x3 on Ampere GPUs", "Limitations and decision criteria".
 *   [TC models] "Accurate Models of NVIDIA Tensor Cores", sections
 *          "Methodology" and "Results".
 *
 * What is computed, step by step, in the order the blog describes it:
 *   1. split each FP32 operand into low-precision components
 *        BF16x9: three scaled BF16 components            ([Blog] Fig. 1)
 *        TF32x3: a leading and a residual TF32 component  ([Blog] Fig. 2)
 *   2. form the selected cross products of components (exact in FP32)
 *   3. accumulate them in FP32
 *        BF16x9: along the five anti-diagonal bands i+j = 0..4, then recombine
 *                with the scale factors                    ([Blog] Fig. 1)
 *        TF32x3: hi*hi + hi*lo + lo*hi, lo*lo dropped       ([Blog] Eq. 1)
 * a model of the tensor cores that carry out step 3 on the GPU, for bit-level
 * comparison ([TC models] "Methodology", "Results"):
 *   - one block FMA per tensor-core instruction (16 BF16 or 8 TF32 products
 *     and an FP32 accumulator input), 2 extra alignment bits, truncation;
 *   - the emulated GEMM through that model in the order this repository's
 *     kernel issues its work (oracle_gemm_tc);
 * and the plain definitions the method is judged against:
 *   - the float64 GEMM (products and sums in binary64, sequential in k);
 *   - the native FP32 SGEMM (sequential round-to-nearest fmaf over k), the
 *     "native FP32" accuracy the blog compares against
 *     ([Blog] "Limitations and decision criteria").
 *
 * Readings where the blog is silent (each is listed with its reason in the
 * design notes of the repository):
 *   - BF16x9 scale: 2^8 per component level; 8 is the BF16 significand width,
 *     so the three components cover the 24-bit FP32 significand exactly.
 *   - BF16x9 rounding of each component: toward zero (keep the top 16 bits of
 *     the FP32 word).  The split is then exact for every finite FP32 value.
 *   - TF32x3 rounding: hi = nearest TF32 (ties to even), lo = nearest TF32 of
 *     the exact residual a - hi.  A second variant takes hi by truncation
 *     (TF32X3_HI_RZ), which is what a tensor core does when it ignores the
 *     low 13 bits of an FP32 container.
 *   - Band accumulation: one FP32 round-to-nearest sum per band, sequential in
 *     k, adding the band's products in (i, j) order with i ascending; then
 *     recombination smallest band first.  A second variant keeps one FP32 sum
 *     and adds, for each k, bands 4 down to 0 into it.
 *   - alpha/beta/bias: C = fmaf(alpha, acc, beta * C_old) + bias; beta == 0
 *     never reads C_old.
 *
 * Pins: every function in this file is checked on the CPU against something
 * other than itself (exact rational arithmetic, closed forms, hand-derived
 * golden values, brute force on tiny inputs; tests/test_oracle_*.py), and
 * planted mistakes in each one are caught (tests/test_oracle_mutations.py).
 * None is unpinned.
 *
 * Matrices are row-major.  op(A) is M x K: A[m*lda + k] when transA == 0,
 * A[k*lda + m] when transA == 1.  op(B) is K x N: B[k*ldb + n] when
 * transB == 0, B[n*ldb + k] when transB == 1.  C is M x N with leading
 * dimension ldc.  The row list `rows` (NULL = all rows) lets a caller
 * evaluate a sample of the output rows of a large problem.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared [-fopenmp].  Contraction
 * must stay off: every multiply and add below is meant to round separately,
 * and fmaf is written where a fused operation is meant.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <limits.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* bit helpers                                                              */
/* ------------------------------------------------------------------------ */
static inline uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline float float_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* Round toward zero to BF16: keep sign, exponent and the top 7 fraction bits. */
static inline float bf16_rz(float x) { return float_of(bits_of(x) & 0xFFFF0000u); }

/* Round to nearest, ties to even, to TF32 (10 fraction bits).  Inf and NaN
 * pass through unchanged; a finite value beyond the largest TF32 number
 * rounds to infinity, as IEEE rounding to a narrower format does. */
static inline float tf32_rn(float x)
{
    uint32_t u = bits_of(x);
    if ((u & 0x7F800000u) == 0x7F800000u) return x;
    uint32_t keep_lsb = (u >> 13) & 1u;
    u += 0x00000FFFu + keep_lsb;
    return float_of(u & 0xFFFFE000u);
}

/* Round toward zero to TF32. */
static inline float tf32_rz(float x) { return float_of(bits_of(x) & 0xFFFFE000u); }

/* ------------------------------------------------------------------------ */
/* Step 1: splits                                                           */
/* ------------------------------------------------------------------------ */

/* BF16x9 split of one value into three scaled BF16 components
 * ([Blog] Fig. 1: "each FP32 operand is split into three scaled BF16
 * components"):  a = c0 + 2^-8 c1 + 2^-16 c2.
 *   c0 = RZ_bf16(a)
 *   c1 = RZ_bf16(2^8 (a - c0))
 *   c2 = 2^8 (2^8 (a - c0) - c1)       -- at most 8 significant bits, so BF16
 * Each subtraction is exact (the subtrahend is a leading part of the
 * minuend) and each scaling by 2^8 is exact. */
static inline void split3(float a, float *c0, float *c1, float *c2)
{
    float a0 = bf16_rz(a);
    float r1 = (a - a0) * 256.0f;
    float a1 = bf16_rz(r1);
    float a2 = (r1 - a1) * 256.0f;
    *c0 = a0; *c1 = a1; *c2 = a2;
}

/* TF32x3 split ([Blog] Fig. 2: a leading TF32 component and a residual TF32
 * component, no scale factor). */
enum { TF32X3_HI_RN = 0, TF32X3_HI_RZ = 1 };
static inline void split2(float a, int variant, float *hi, float *lo)
{
    float h = (variant == TF32X3_HI_RZ) ? tf32_rz(a) : tf32_rn(a);
    *hi = h;
    *lo = tf32_rn(a - h);
}

ORACLE_API void oracle_split_bf16x9(const float *a, int64_t n,
                                    uint16_t *s0, uint16_t *s1, uint16_t *s2)
{
    for (int64_t i = 0; i < n; ++i) {
        float c0, c1, c2;
        split3(a[i], &c0, &c1, &c2);
        s0[i] = (uint16_t)(bits_of(c0) >> 16);
        s1[i] = (uint16_t)(bits_of(c1) >> 16);
        s2[i] = (uint16_t)(bits_of(c2) >> 16);
    }
}

/* The low 16 bits of every FP32 word written here are zero when the split is
 * exact; the caller checks that, which is why the words are returned whole. */
ORACLE_API void oracle_split_bf16x9_f32(const float *a, int64_t n,
                                        float *c0, float *c1, float *c2)
{
    for (int64_t i = 0; i < n; ++i) split3(a[i], &c0[i], &c1[i], &c2[i]);
}

ORACLE_API void oracle_split_tf32x3(const float *a, int64_t n, int variant,
                                    float *hi, float *lo)
{
    for (int64_t i = 0; i < n; ++i) split2(a[i], variant, &hi[i], &lo[i]);
}

/* ------------------------------------------------------------------------ */
/* operand packing: op(A) as M x K rows, op(B)^T as N x K rows              */
/* (a copy, no arithmetic; it only makes the k loops below contiguous)      */
/* ------------------------------------------------------------------------ */
static float *pack_opA(int transA, int64_t M, int64_t K, const float *A, int64_t lda)
{
    float *p = (float *)malloc(sizeof(float) * (size_t)(M > 0 ? M : 1) * (size_t)(K > 0 ? K : 1));
    if (!p) return NULL;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            p[m * K + k] = transA ? A[k * lda + m] : A[m * lda + k];
    return p;
}

static float *pack_opBt(int transB, int64_t N, int64_t K, const float *B, int64_t ldb)
{
    float *p = (float *)malloc(sizeof(float) * (size_t)(N > 0 ? N : 1) * (size_t)(K > 0 ? K : 1));
    if (!p) return NULL;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            p[n * K + k] = transB ? B[n * ldb + k] : B[k * ldb + n];
    return p;
}

static inline int64_t row_at(const int64_t *rows, int64_t r) { return rows ? rows[r] : r; }

/* C = fmaf(alpha, acc, beta*C_old) + bias, in FP32.  beta == 0 never reads C_old. */
static inline float epilogue_f32(float acc, float alpha, float beta, const float *Cold_elem,
                                 const float *bias_elem)
{
    float bc = (beta != 0.0f) ? beta * (*Cold_elem) : 0.0f;
    float c = fmaf(alpha, acc, bc);
    if (bias_elem) c = c + *bias_elem;
    return c;
}

/* ------------------------------------------------------------------------ */
/* Plain definitions                                                         */
/* ------------------------------------------------------------------------ */

/* float64 GEMM: C64 = alpha * (op(A) op(B)) + beta * C_old + bias, every
 * product and sum in binary64, sequential in k.  Output rows follow `rows`
 * (C64 has nrows x N entries, row-major, leading dimension N). */
ORACLE_API int oracle_gemm_f64(int transA, int transB, int64_t M, int64_t N, int64_t K,
                               double alpha, const float *A, int64_t lda,
                               const float *B, int64_t ldb,
                               double beta, const float *Cold, int64_t ldc,
                               const float *bias,
                               const int64_t *rows, int64_t nrows, double *C64)
{
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    if (!pa || !pb) { free(pa); free(pb); return -1; }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            const float *ar = pa + m * K, *br = pb + n * K;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += (double)ar[k] * (double)br[k];
            double c = alpha * s;
            if (beta != 0.0) c += beta * (double)Cold[m * ldc + n];
            if (bias) c += (double)bias[n];
            C64[r * N + n] = c;
        }
    }
    free(pa); free(pb);
    return 0;
}

/* The denominator of the normwise error: D = |alpha| (|op(A)| |op(B)|)
 * + |beta| |C_old| + |bias|, in binary64. */
ORACLE_API int oracle_gemm_absdenom_f64(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                        double alpha, const float *A, int64_t lda,
                                        const float *B, int64_t ldb,
                                        double beta, const float *Cold, int64_t ldc,
                                        const float *bias,
                                        const int64_t *rows, int64_t nrows, double *D)
{
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    if (!pa || !pb) { free(pa); free(pb); return -1; }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            const float *ar = pa + m * K, *br = pb + n * K;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += fabs((double)ar[k]) * fabs((double)br[k]);
            double d = fabs(alpha) * s;
            if (beta != 0.0) d += fabs(beta) * fabs((double)Cold[m * ldc + n]);
            if (bias) d += fabs((double)bias[n]);
            D[r * N + n] = d;
        }
    }
    free(pa); free(pb);
    return 0;
}

/* Native FP32 SGEMM: acc = fmaf(a_k, b_k, acc) for k = 0..K-1 in order,
 * then the FP32 epilogue.  C has nrows x N entries (leading dimension N). */
ORACLE_API int oracle_sgemm_f32(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                float alpha, const float *A, int64_t lda,
                                const float *B, int64_t ldb,
                                float beta, const float *Cold, int64_t ldc,
                                const float *bias,
                                const int64_t *rows, int64_t nrows, float *C)
{
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    if (!pa || !pb) { free(pa); free(pb); return -1; }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            const float *ar = pa + m * K, *br = pb + n * K;
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) acc = fmaf(ar[k], br[k], acc);
            C[r * N + n] = epilogue_f32(acc, alpha, beta, Cold + m * ldc + n,
                                        bias ? bias + n : NULL);
        }
    }
    free(pa); free(pb);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Steps 2-3: BF16x9                                                         */
/* ------------------------------------------------------------------------ */
enum { BF16X9_FIVE_BANDS = 0, BF16X9_ONE_ACCUMULATOR = 1 };

/* Split every element of an n-vector into its three scaled BF16 components,
 * stored as three planes. */
static float *split3_planes(const float *x, int64_t n)
{
    float *p = (float *)malloc(sizeof(float) * 3 * (size_t)(n > 0 ? n : 1));
    if (!p) return NULL;
    for (int64_t i = 0; i < n; ++i) split3(x[i], &p[i], &p[n + i], &p[2 * n + i]);
    return p;
}

/* BF16x9 emulated GEMM ([Blog] Fig. 1).
 *   Products: P_ij(k) = a_i(k) * b_j(k), BF16 x BF16, exact in FP32.
 *   Band b = i + j carries the scale 2^-8b.
 *   FIVE_BANDS (the plain reading of "accumulated in FP32 along the five
 *   anti-diagonal bands"): S_b = sum over k of the band's products, one FP32
 *   round-to-nearest sum per band, the products of band b added in order of
 *   ascending i; then acc = S_4 2^-32 + S_3 2^-24 + S_2 2^-16 + S_1 2^-8 + S_0,
 *   added smallest band first, in FP32.
 *   ONE_ACCUMULATOR: one FP32 sum; for each k the scaled products are added
 *   band 4 first, down to band 0.
 * bands_out (optional, 5 x nrows x N): the band sums S_0..S_4 (FIVE_BANDS). */
ORACLE_API int oracle_gemm_bf16x9(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                  float alpha, const float *A, int64_t lda,
                                  const float *B, int64_t ldb,
                                  float beta, const float *Cold, int64_t ldc,
                                  const float *bias, int variant,
                                  const int64_t *rows, int64_t nrows,
                                  float *C, float *bands_out)
{
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    float *sa = pa ? split3_planes(pa, M * K) : NULL;
    float *sb = pb ? split3_planes(pb, N * K) : NULL;
    if (!pa || !pb || !sa || !sb) { free(pa); free(pb); free(sa); free(sb); return -1; }
    const int64_t MK = M * K, NK = N * K;
    /* scale of band b: 2^-8b */
    const float band_scale[5] = { 1.0f, 0x1p-8f, 0x1p-16f, 0x1p-24f, 0x1p-32f };
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            const float *a[3] = { sa + m * K, sa + MK + m * K, sa + 2 * MK + m * K };
            const float *b[3] = { sb + n * K, sb + NK + n * K, sb + 2 * NK + n * K };
            float acc;
            if (variant == BF16X9_ONE_ACCUMULATOR) {
                acc = 0.0f;
                for (int64_t k = 0; k < K; ++k)
                    for (int band = 4; band >= 0; --band)
                        for (int i = 0; i <= 2; ++i) {
                            int j = band - i;
                            if (j < 0 || j > 2) continue;
                            float p = a[i][k] * b[j][k];          /* exact */
                            acc = acc + p * band_scale[band];     /* scale exact */
                        }
            } else {
                float S[5] = { 0.0f, 0.0f, 0.0f, 0.0f, 0.0f };
                for (int64_t k = 0; k < K; ++k)
                    for (int band = 0; band <= 4; ++band)
                        for (int i = 0; i <= 2; ++i) {
                            int j = band - i;
                            if (j < 0 || j > 2) continue;
                            S[band] = S[band] + a[i][k] * b[j][k];
                        }
                if (bands_out)
                    for (int band = 0; band < 5; ++band)
                        bands_out[(int64_t)band * nrows * N + r * N + n] = S[band];
                acc = S[4] * band_scale[4];
                acc = acc + S[3] * band_scale[3];
                acc = acc + S[2] * band_scale[2];
                acc = acc + S[1] * band_scale[1];
                acc = acc + S[0];
            }
            C[r * N + n] = epilogue_f32(acc, alpha, beta, Cold + m * ldc + n,
                                        bias ? bias + n : NULL);
        }
    }
    free(pa); free(pb); free(sa); free(sb);
    return 0;
}

/* BF16x6 (a comparator, not on the blog's pages): the same split and the same
 * per-band FP32 sums as BF16x9, keeping only bands 0, 1 and 2 (six of the
 * nine products; the four products of bands 3 and 4 are dropped).  Sums in
 * k order, recombined smallest band first: acc = S_2 2^-16 + S_1 2^-8 + S_0. */
ORACLE_API int oracle_gemm_bf16x6(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                  float alpha, const float *A, int64_t lda,
                                  const float *B, int64_t ldb,
                                  float beta, const float *Cold, int64_t ldc,
                                  const float *bias, const int64_t *rows, int64_t nrows, float *C)
{
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    float *sa = pa ? split3_planes(pa, M * K) : NULL;
    float *sb = pb ? split3_planes(pb, N * K) : NULL;
    if (!pa || !pb || !sa || !sb) { free(pa); free(pb); free(sa); free(sb); return -1; }
    const int64_t MK = M * K, NK = N * K;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            const float *a[3] = { sa + m * K, sa + MK + m * K, sa + 2 * MK + m * K };
            const float *b[3] = { sb + n * K, sb + NK + n * K, sb + 2 * NK + n * K };
            float S[3] = { 0.0f, 0.0f, 0.0f };
            for (int64_t k = 0; k < K; ++k)
                for (int band = 0; band <= 2; ++band)
                    for (int i = 0; i <= band; ++i) {
                        int j = band - i;
                        S[band] = S[band] + a[i][k] * b[j][k];
                    }
            float acc = S[2] * 0x1p-16f;
            acc = acc + S[1] * 0x1p-8f;
            acc = acc + S[0];
            C[r * N + n] = epilogue_f32(acc, alpha, beta, Cold + m * ldc + n, bias ? bias + n : NULL);
        }
    }
    free(pa); free(pb); free(sa); free(sb);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Steps 2-3: TF32x3                                                         */
/* ------------------------------------------------------------------------ */

/* TF32x3 emulated GEMM ([Blog] Fig. 2 and Eq. 1):
 *   a b ~= a_hi b_hi + a_hi b_lo + a_lo b_hi   (a_lo b_lo dropped)
 * Each product of two TF32 values (11-bit significands) is exact in FP32.
 * One FP32 round-to-nearest sum over k; for each k the three products are
 * added smallest first: a_lo b_hi, a_hi b_lo, a_hi b_hi.
 * terms_out (optional, 3 x nrows x N): the three separate sums over k of
 * a_hi b_hi, a_hi b_lo and a_lo b_hi, each accumulated in FP32 in k order. */
ORACLE_API int oracle_gemm_tf32x3(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                  float alpha, const float *A, int64_t lda,
                                  const float *B, int64_t ldb,
                                  float beta, const float *Cold, int64_t ldc,
                                  const float *bias, int split_variant,
                                  const int64_t *rows, int64_t nrows,
                                  float *C, float *terms_out)
{
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    float *ha = (float *)malloc(sizeof(float) * 2 * (size_t)(M * K > 0 ? M * K : 1));
    float *hb = (float *)malloc(sizeof(float) * 2 * (size_t)(N * K > 0 ? N * K : 1));
    if (!pa || !pb || !ha || !hb) { free(pa); free(pb); free(ha); free(hb); return -1; }
    const int64_t MK = M * K, NK = N * K;
    for (int64_t i = 0; i < MK; ++i) split2(pa[i], split_variant, &ha[i], &ha[MK + i]);
    for (int64_t i = 0; i < NK; ++i) split2(pb[i], split_variant, &hb[i], &hb[NK + i]);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            const float *ahi = ha + m * K, *alo = ha + MK + m * K;
            const float *bhi = hb + n * K, *blo = hb + NK + n * K;
            float acc = 0.0f, t_hh = 0.0f, t_hl = 0.0f, t_lh = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                float p_lh = alo[k] * bhi[k];
                float p_hl = ahi[k] * blo[k];
                float p_hh = ahi[k] * bhi[k];
                acc = acc + p_lh;
                acc = acc + p_hl;
                acc = acc + p_hh;
                t_hh = t_hh + p_hh; t_hl = t_hl + p_hl; t_lh = t_lh + p_lh;
            }
            if (terms_out) {
                terms_out[0 * nrows * N + r * N + n] = t_hh;
                terms_out[1 * nrows * N + r * N + n] = t_hl;
                terms_out[2 * nrows * N + r * N + n] = t_lh;
            }
            C[r * N + n] = epilogue_f32(acc, alpha, beta, Cold + m * ldc + n,
                                        bias ? bias + n : NULL);
        }
    }
    free(pa); free(pb); free(ha); free(hb);
    return 0;
}

/* One-pass TF32 ([Blog] "TF32x3 on Ampere GPUs": the faster, less accurate
 * comparator): a b ~= hi(a) hi(b) with hi the nearest TF32 number, one FP32
 * round-to-nearest sum over k.  Each product of two 11-bit significands is
 * exact in FP32. */
ORACLE_API int oracle_gemm_tf32x1(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                  float alpha, const float *A, int64_t lda,
                                  const float *B, int64_t ldb,
                                  float beta, const float *Cold, int64_t ldc,
                                  const float *bias, const int64_t *rows, int64_t nrows, float *C)
{
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    if (!pa || !pb) { free(pa); free(pb); return -1; }
    for (int64_t i = 0; i < M * K; ++i) pa[i] = tf32_rn(pa[i]);
    for (int64_t i = 0; i < N * K; ++i) pb[i] = tf32_rn(pb[i]);
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            const float *ar = pa + m * K, *br = pb + n * K;
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) acc = acc + ar[k] * br[k];
            C[r * N + n] = epilogue_f32(acc, alpha, beta, Cold + m * ldc + n, bias ? bias + n : NULL);
        }
    }
    free(pa); free(pb);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The emulated result with exact accumulation                               */
/* ------------------------------------------------------------------------ */

/* A fixed-point accumulator wide enough to hold any sum of up to 2^31
 * products of two FP32 numbers without rounding: 32-bit digits (kept in
 * int64 so that additions need no carry until the end) at weights
 * 2^(SA_EMIN + 32 i).  The smallest product of two nonzero FP32 numbers is
 * 2^-298 (53-bit significand in binary64: last bit 2^-350 at worst); the
 * largest is below 2^256, and 2^31 of them below 2^287. */
#define SA_EMIN (-384)
#define SA_DIGITS 24
typedef struct { int64_t d[SA_DIGITS]; } superacc;

/* Add a finite binary64 value exactly (every value added here is a normal
 * binary64 number: a product of two FP32 numbers, times a power of two). */
static inline void sa_add(superacc *s, double x)
{
    uint64_t u;
    memcpy(&u, &x, 8);
    const int be = (int)((u >> 52) & 0x7FF);
    if (be == 0) return;                           /* zero */
    const uint64_t m = (u & ((UINT64_C(1) << 52) - 1)) | (UINT64_C(1) << 52);
    const int pos = be - 1075 - SA_EMIN;           /* |x| = m 2^(SA_EMIN + pos) */
    const int i = pos >> 5;
    const unsigned __int128 v = (unsigned __int128)m << (pos & 31);
    const int64_t sg = (u >> 63) ? -1 : 1;
    s->d[i] += sg * (int64_t)(uint32_t)v;
    s->d[i + 1] += sg * (int64_t)(uint32_t)(v >> 32);
    s->d[i + 2] += sg * (int64_t)(uint32_t)(v >> 64);
}

/* Propagate carries: every digit but the last in [0, 2^32). */
static void sa_carry(superacc *s)
{
    for (int i = 0; i < SA_DIGITS - 1; ++i) {
        const int64_t c = (s->d[i] - (s->d[i] & 0xFFFFFFFF)) / ((int64_t)1 << 32);  /* floor division */
        s->d[i] -= c * ((int64_t)1 << 32);
        s->d[i + 1] += c;
    }
}

/* The accumulator's exact value rounded once to FP32, to nearest with ties
 * to even (overflow to infinity, gradual underflow), as an IEEE conversion
 * of the exact value would.  It is first rounded to 53 bits "to odd" (the
 * last bit records whether anything below it was nonzero); a rounding to
 * odd at 53 bits followed by a rounding to nearest at 24 bits or fewer is
 * the correctly rounded result. */
static float sa_round_f32(superacc *s)
{
    sa_carry(s);
    const int neg = s->d[SA_DIGITS - 1] < 0;
    if (neg) {
        for (int i = 0; i < SA_DIGITS; ++i) s->d[i] = -s->d[i];
        sa_carry(s);
    }
    int top = SA_DIGITS - 1;
    while (top >= 0 && s->d[top] == 0) --top;
    if (top < 0) return 0.0f;
    unsigned __int128 w = 0;
    int sticky = 0;
    for (int i = top; i >= top - 2; --i) w = (w << 32) | (uint32_t)(i >= 0 ? s->d[i] : 0);
    for (int i = top - 3; i >= 0; --i) sticky |= s->d[i] != 0;
    int e = SA_EMIN + 32 * (top - 2);              /* weight of bit 0 of w */
    int nbits = 0;
    for (unsigned __int128 t = w; t; t >>= 1) ++nbits;
    if (nbits > 53) {
        const int sh = nbits - 53;
        sticky |= (w & ((((unsigned __int128)1) << sh) - 1)) != 0;
        w >>= sh;
        e += sh;
    }
    uint64_t t53 = (uint64_t)w;
    if (sticky) t53 |= 1u;
    const float f = (float)ldexp((double)t53, e);  /* the double is exact; one rounding to FP32 */
    return neg ? -f : f;
}

/* The emulated GEMM with its accumulation made exact: the method's selected
 * component products -- BF16x9 ([Blog] Fig. 1): the nine products
 * 2^-8(i+j) c_i(a) c_j(b) of the scaled components; BF16x6: those of bands
 * 0-2; TF32x3 ([Blog] Eq. 1): a_hi b_hi + a_hi b_lo + a_lo b_hi; one-pass
 * TF32: a_hi b_hi -- each exact, summed over k with no rounding at all, the
 * sum then rounded once to FP32 (nearest, ties to even), then the FP32
 * epilogue.  It is the limit that "accumulated in FP32" approaches as the
 * accumulation error vanishes, whatever its order: the reference against
 * which the error of any FP32 accumulation of the same products is
 * measured.  kind: 0 BF16x9, 1 BF16x6, 2 TF32x3, 3 one-pass TF32. */
ORACLE_API int oracle_gemm_exact_sum(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                     float alpha, const float *A, int64_t lda,
                                     const float *B, int64_t ldb,
                                     float beta, const float *Cold, int64_t ldc,
                                     const float *bias, int kind,
                                     const int64_t *rows, int64_t nrows, float *C)
{
    if (kind < 0 || kind > 3) return -2;
    if (K > INT32_MAX / 9) return -2;
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    float *sa = pa ? (float *)malloc(sizeof(float) * 3 * (size_t)(M * K > 0 ? M * K : 1)) : NULL;
    float *sb = pb ? (float *)malloc(sizeof(float) * 3 * (size_t)(N * K > 0 ? N * K : 1)) : NULL;
    if (!sa || !sb) { free(pa); free(pb); free(sa); free(sb); return -1; }
    const int64_t MK = M * K, NK = N * K;
    for (int side = 0; side < 2; ++side) {
        const float *x = side ? pb : pa;
        float *out = side ? sb : sa;
        const int64_t n = side ? NK : MK;
        for (int64_t i = 0; i < n; ++i) {
            if (kind <= 1) {
                split3(x[i], &out[i], &out[n + i], &out[2 * n + i]);
            } else {
                split2(x[i], TF32X3_HI_RN, &out[i], &out[n + i]);
                out[2 * n + i] = 0.0f;
            }
        }
    }
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = row_at(rows, r);
        for (int64_t n = 0; n < N; ++n) {
            superacc s;
            memset(&s, 0, sizeof s);
            for (int64_t k = 0; k < K; ++k) {
                const double a0 = sa[m * K + k], a1 = sa[MK + m * K + k], a2 = sa[2 * MK + m * K + k];
                const double b0 = sb[n * K + k], b1 = sb[NK + n * K + k], b2 = sb[2 * NK + n * K + k];
                if (kind <= 1) {
                    /* band i + j carries the scale 2^-8(i+j); every product and
                     * scaling below is exact in binary64 */
                    sa_add(&s, a0 * b0);
                    sa_add(&s, a0 * b1 * 0x1p-8);
                    sa_add(&s, a1 * b0 * 0x1p-8);
                    sa_add(&s, a0 * b2 * 0x1p-16);
                    sa_add(&s, a1 * b1 * 0x1p-16);
                    sa_add(&s, a2 * b0 * 0x1p-16);
                    if (kind == 0) {
                        sa_add(&s, a1 * b2 * 0x1p-24);
                        sa_add(&s, a2 * b1 * 0x1p-24);
                        sa_add(&s, a2 * b2 * 0x1p-32);
                    }
                } else {
                    /* a0, b0 = hi; a1, b1 = lo */
                    sa_add(&s, a0 * b0);
                    if (kind == 2) {
                        sa_add(&s, a0 * b1);
                        sa_add(&s, a1 * b0);
                    }
                }
            }
            const float acc = sa_round_f32(&s);
            C[r * N + n] = epilogue_f32(acc, alpha, beta, Cold + m * ldc + n, bias ? bias + n : NULL);
        }
    }
    free(pa); free(pb); free(sa); free(sb);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Tensor-core accumulation model                                            */
/* ------------------------------------------------------------------------ */

/* One block FMA of a tensor core, after [TC models] "Methodology" and
 * "Results" (Hopper/Blackwell-class parts with BF16 inputs: blocks of
 * N_FMA = 16 products, n_eab = 2 extra alignment bits, truncation).
 * d = c + sum_i a_i b_i for up to n pairs of BF16 numbers a_i, b_i and an
 * FP32 accumulator input c:
 *   - every term has an alignment exponent: e(a_i) + e(b_i) for a product
 *     (the exponent of the product before normalisation; the product itself
 *     is exact), e(c) for the accumulator, e() the unbiased exponent;
 *   - with e_max the largest alignment exponent among the nonzero terms, each
 *     term keeps its bits down to 2^(e_max - 23 - neab) and loses the ones
 *     below, toward zero;
 *   - the kept parts are added exactly and the sum is rounded once to FP32,
 *     toward zero (round_mode 0) or to nearest even (round_mode 1).
 * The pages give N_FMA, n_eab and truncation but not the alignment reference
 * or the final rounding; this repository's GPU tests fix both against its
 * kernel (products aligned on e(a)+e(b), the accumulator on e(c), rounding
 * toward zero: identical bits on every tested element). */
ORACLE_API float oracle_tc_block_fma(float c, const float *a, const float *b, int n, int neab, int round_mode)
{
    if (neab < 0 || neab > 24 || n < 0 || n > 64) return NAN;   /* the exact integer sum below needs it */
    int emax = INT_MIN;
    if (c != 0.0f) emax = ilogb((double)c);
    for (int i = 0; i < n; ++i)
        if (a[i] != 0.0f && b[i] != 0.0f) {
            const int e = ilogb((double)a[i]) + ilogb((double)b[i]);
            if (e > emax) emax = e;
        }
    if (emax == INT_MIN) return 0.0f;
    const int q = emax - 23 - neab;   /* weight of the last kept bit */
    int64_t S = (int64_t)trunc(ldexp((double)c, -q));
    for (int i = 0; i < n; ++i)
        if (a[i] != 0.0f && b[i] != 0.0f) S += (int64_t)trunc(ldexp((double)a[i] * (double)b[i], -q));
    const double v = ldexp((double)S, q);   /* exact: |S| < 65 * 2^(25 + neab) <= 2^53 */
    float f = (float)v;                     /* nearest, ties to even */
    if (round_mode == 0 && fabs((double)f) > fabs(v)) f = nextafterf(f, 0.0f);
    return f;
}

/* The emulated GEMM through the tensor-core model, in the order this
 * repository's kernel issues its work.  kind: 0 BF16x9, 1 BF16x6, 2 TF32x3,
 * 3 one-pass TF32.
 *   Components: BF16 -- the BF16x9 split in natural magnitude (component i
 *   times 2^-8i, so every product carries its band scale); TF32 -- hi and lo
 *   of the TF32x3 split (hi alone for one-pass TF32).
 *   Products per stage, smallest first: BF16x9 (i,j) = (2,2) (1,2) (2,1)
 *   (0,2) (1,1) (2,0) (0,1) (1,0) (0,0); BF16x6 (0,2) (1,1) (2,0) (0,1) (1,0)
 *   (0,0); TF32x3 (lo,hi) (hi,lo) (hi,hi); one-pass TF32 (hi,hi).
 *   k runs in stages of stage_k; per stage a fresh accumulator takes, product
 *   by product, one block FMA (oracle_tc_block_fma) per `block` consecutive k
 *   (16 for BF16 inputs, 8 for TF32: one tensor-core instruction each); the
 *   stage's result is added into an FP32 sum (round to nearest).  k beyond K
 *   contributes zeros.
 *   pieces > 1: the k-stages are cut into `pieces` ranges (piece q takes
 *   stages [q KS / pieces, (q + 1) KS / pieces), KS = ceil(K / stage_k)),
 *   each summed from zero as above; the pieces' sums of an output element are
 *   then added -- the owning piece's first, the others in increasing order --
 *   where element (m, n) of a 256 x 256 tile belongs to piece
 *   (4 e + c) mod pieces, e = 4 ((n mod 256) / 128) + (m mod 128) / 32 and
 *   c = (n mod 128) / 32 (integer division).
 *   Then the epilogue. */
ORACLE_API int oracle_gemm_tc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                              float alpha, const float *A, int64_t lda,
                              const float *B, int64_t ldb,
                              float beta, const float *Cold, int64_t ldc,
                              const float *bias, const int64_t *rows, int64_t nrows, float *C,
                              int kind, int stage_k, int block, int neab, int round_mode, int pieces)
{
    static const int pi9[9] = {2, 1, 2, 0, 1, 2, 0, 1, 0}, pj9[9] = {2, 2, 1, 2, 1, 0, 1, 0, 0};
    static const int pi6[6] = {0, 1, 2, 0, 1, 0}, pj6[6] = {2, 1, 0, 1, 0, 0};
    static const int pi3[3] = {1, 0, 0}, pj3[3] = {0, 1, 0};
    static const int pi1[1] = {0}, pj1[1] = {0};
    if (kind < 0 || kind > 3) return -2;
    if (block < 1 || block > 64 || stage_k < block || stage_k % block || pieces < 1 || pieces > 64) return -2;
    const int nprod = kind == 0 ? 9 : kind == 1 ? 6 : kind == 2 ? 3 : 1;
    const int *pi = kind == 0 ? pi9 : kind == 1 ? pi6 : kind == 2 ? pi3 : pi1;
    const int *pj = kind == 0 ? pj9 : kind == 1 ? pj6 : kind == 2 ? pj3 : pj1;
    const int ncomp = kind <= 1 ? 3 : kind == 2 ? 2 : 1;
    if (!rows) nrows = M;
    float *pa = pack_opA(transA, M, K, A, lda);
    float *pb = pack_opBt(transB, N, K, B, ldb);
    float *sa = pa ? (float *)malloc(sizeof(float) * 3 * (size_t)(M * K > 0 ? M * K : 1)) : NULL;
    float *sb = pb ? (float *)malloc(sizeof(float) * 3 * (size_t)(N * K > 0 ? N * K : 1)) : NULL;
    if (!sa || !sb) { free(pa); free(pb); free(sa); free(sb); return -1; }
    for (int side = 0; side < 2; ++side) {
        const float *x = side ? pb : pa;
        float *out = side ? sb : sa;
        const int64_t n = side ? N * K : M * K;
        for (int64_t i = 0; i < n; ++i) {
            if (kind <= 1) {
                float c0, c1, c2;
                split3(x[i], &c0, &c1, &c2);
                out[i] = c0; out[n + i] = c1 * 0x1p-8f; out[2 * n + i] = c2 * 0x1p-16f;
            } else {
                float hi, lo;
                split2(x[i], TF32X3_HI_RN, &hi, &lo);
                out[i] = hi; out[n + i] = lo;
            }
        }
    }
    (void)ncomp;
    const int64_t stages = (K + stage_k - 1) / stage_k;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t m = row_at(rows, r);
        float ab[64], bb[64];
        float part[64];
        for (int64_t n = 0; n < N; ++n) {
            for (int q = 0; q < pieces; ++q) {
                const int64_t s0 = (int64_t)q * stages / pieces, s1 = (int64_t)(q + 1) * stages / pieces;
                float acc = 0.0f;
                for (int64_t s = s0; s < s1; ++s) {
                    float t = 0.0f;
                    for (int p = 0; p < nprod; ++p) {
                        const float *ai = sa + (int64_t)pi[p] * M * K + m * K;
                        const float *bj = sb + (int64_t)pj[p] * N * K + n * K;
                        for (int64_t k0 = s * stage_k; k0 < (s + 1) * stage_k; k0 += block) {
                            for (int j = 0; j < block; ++j) {
                                const int64_t k = k0 + j;
                                ab[j] = k < K ? ai[k] : 0.0f;
                                bb[j] = k < K ? bj[k] : 0.0f;
                            }
                            t = oracle_tc_block_fma(t, ab, bb, block, neab, round_mode);
                        }
                    }
                    acc = acc + t;
                }
                part[q] = acc;
            }
            float acc = part[0];
            if (pieces > 1) {
                const int64_t tm = m % 256, tn = n % 256;
                const int e = 4 * (int)(tn / 128) + (int)((tm % 128) / 32), c = (int)((tn % 128) / 32);
                const int owner = (4 * e + c) % pieces;
                acc = part[owner];
                for (int q = 0; q < pieces; ++q)
                    if (q != owner) acc = acc + part[q];
            }
            C[r * N + n] = epilogue_f32(acc, alpha, beta, Cold ? &Cold[m * ldc + n] : NULL,
                                        bias ? &bias[n] : NULL);
        }
    }
    free(pa); free(pb); free(sa); free(sb);
    return 0;
}

ORACLE_API int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
