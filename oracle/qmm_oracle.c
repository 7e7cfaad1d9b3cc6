/*
 * CPU oracle for the split-K W4A16-g128 projection matmul and the dense BF16
 * split-K GEMM.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * bench's CPU baseline call it; the library never does.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Plain, slow and meant to be read against the sources:
 *   [TL] tiny-llm book, "Week 2 Day 7: Split-K Prefill"
 *        (Why Split the Reduction Dimension?; Task 2: Reuse the Day 6 Kernel
 *        for Each Partition; Task 3: Choose Partitions From Occupancy;
 *        Task 4: Reduce and Verify)
 *   [SK] gpu-kernels-explained, "Split-K, streams and overlap"
 *        (first Concept section: copy-in / compute / copy-out engines and
 *        buffers; second Concept section; Maths, "Overlap" and "Split-K";
 *        the A100 model table)
 *   [PD] "Optimize Prefill vs Decode Kernels" (Required reasoning process,
 *        steps 4 and 5: split-K for decode matmuls, at least ~512 reduction
 *        elements per split, split-KV decode attention; Correctness
 *        requirements: the FP32 log-sum-exp merge)
 * The weight format (w = scale*q + bias, q in 0..15, eight nibbles per
 * uint32 low nibble first, BF16 scale and bias per 128-group along the
 * reduction axis) is the MLX-style affine "w4a16_g128" format [TL] checks
 * against.
 *
 * Conventions: M activation rows, Kred reduction length, Nout output width
 * ([TL] writes K for the output width and N for the reduction length).
 * A is BF16 [M, Kred]; Wq uint32 [Nout, Kred/8]; scales, biases BF16
 * [Nout, Kred/128]; C = A . W^T is [M, Nout].  BF16 values travel as uint16
 * bit patterns.  Floating point is fp64 unless a step rounds on purpose.
 * Every function returns 0 on success and a negative code on bad arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QO_GROUP 128

/* ---- number formats ---------------------------------------------------- */

/* BF16 bit pattern -> double (exact: BF16 is the top half of an fp32). */
static double bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a finite double to the nearest BF16 value, ties to even.
 * BF16 keeps 8 significant bits: write |x| = m * 2^e with m in [0.5, 1),
 * round m * 2^8 to an integer (nearbyint rounds half to even in the default
 * rounding mode) and scale back.  Values below the BF16 normal range or
 * above its maximum are refused; the workloads never produce them. */
static int bf16_round(double x, uint16_t *out) {
    if (!isfinite(x)) return -1;
    if (x == 0.0) { *out = signbit(x) ? 0x8000u : 0u; return 0; }
    int e;
    double m = frexp(fabs(x), &e);
    if (e < -125) return -2;                  /* |x| < 2^-126: subnormal */
    double y = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    if (y > 3.3895313892515355e38) return -3; /* above BF16 max */
    float f = (float)y;                       /* exact: 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    *out = (uint16_t)((u >> 16) | (signbit(x) ? 0x8000u : 0u));
    return 0;
}

int oracle_bf16_round(const double *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i)
        if (bf16_round(x[i], &out[i])) return -1;
    return 0;
}

int oracle_bf16_value(const uint16_t *b, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(b[i]);
    return 0;
}

/* ---- W4A16-g128: unpack and dequant ------------------------------------ */

/* q[n, k] = (Wq[n, k/8] >> 4*(k%8)) & 0xF : eight nibbles per word, the
 * lowest nibble holds the smallest k. */
static int nibble(const uint32_t *Wq, int64_t Kred, int64_t n, int64_t k) {
    uint32_t word = Wq[n * (Kred / 8) + k / 8];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

int oracle_unpack(const uint32_t *Wq, int64_t Nout, int64_t Kred, uint8_t *q) {
    if (Nout < 1 || Kred < 8 || Kred % 8) return -1;
    for (int64_t n = 0; n < Nout; ++n)
        for (int64_t k = 0; k < Kred; ++k)
            q[n * Kred + k] = (uint8_t)nibble(Wq, Kred, n, k);
    return 0;
}

/* w[n, k] = BF16(scale[n, g] * q[n, k] + bias[n, g]) with g = k / 128.
 * The product of a BF16 scale and a 4-bit integer has at most 12 significant
 * bits, so scale*q + bias is exact in fp64 and the single rounding to BF16
 * is the correctly rounded dequantized weight.  Rows are dequantized one at
 * a time into a caller buffer of Kred doubles (the BF16 values, exactly). */
static int dequant_row(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                       int64_t Kred, int64_t n, double *w) {
    int64_t G = Kred / QO_GROUP;
    for (int64_t k = 0; k < Kred; ++k) {
        int64_t g = k / QO_GROUP;
        double s = bf16_value(scales[n * G + g]);
        double b = bf16_value(biases[n * G + g]);
        uint16_t wb;
        if (bf16_round(s * (double)nibble(Wq, Kred, n, k) + b, &wb)) return -1;
        w[k] = bf16_value(wb);
    }
    return 0;
}

int oracle_dequant(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                   int64_t Nout, int64_t Kred, uint16_t *w_bf16) {
    if (Nout < 1 || Kred < QO_GROUP || Kred % QO_GROUP) return -1;
    double *row = (double *)malloc(sizeof(double) * (size_t)Kred);
    if (!row) return -4;
    int rc = 0;
    for (int64_t n = 0; n < Nout && !rc; ++n) {
        rc = dequant_row(Wq, scales, biases, Kred, n, row);
        for (int64_t k = 0; k < Kred && !rc; ++k) rc = bf16_round(row[k], &w_bf16[n * Kred + k]);
    }
    free(row);
    return rc ? -1 : 0;
}

/* Dequantize the whole weight into doubles (row-major [Nout, Kred]). */
static double *dequant_all(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                           int64_t Nout, int64_t Kred, int nthreads) {
    double *w = (double *)malloc(sizeof(double) * (size_t)(Nout * Kred));
    if (!w) return NULL;
    int bad = 0;
#pragma omp parallel for num_threads(nthreads) schedule(static) reduction(| : bad)
    for (int64_t n = 0; n < Nout; ++n)
        bad |= dequant_row(Wq, scales, biases, Kred, n, w + n * Kred) != 0;
    if (bad) { free(w); return NULL; }
    return w;
}

static double *bf16_matrix(const uint16_t *x, int64_t rows, int64_t cols, int nthreads) {
    double *d = (double *)malloc(sizeof(double) * (size_t)(rows * cols));
    if (!d) return NULL;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t i = 0; i < rows * cols; ++i) d[i] = bf16_value(x[i]);
    return d;
}

/* sum over k in [k0, k1) of a[k] * w[k], fp64, ascending k */
static double dot(const double *a, const double *w, int64_t k0, int64_t k1) {
    double acc = 0.0;
    for (int64_t k = k0; k < k1; ++k) acc += a[k] * w[k];
    return acc;
}

/* ---- W4A16-g128: the matmul -------------------------------------------- */

/* C64[m, n] = sum_k A[m, k] * w[n, k]: the plain definition of C = A @ W^T
 * [TL, Why Split the Reduction Dimension?], in fp64. */
int oracle_qmm(const uint16_t *A, const uint32_t *Wq, const uint16_t *scales,
               const uint16_t *biases, int64_t M, int64_t Kred, int64_t Nout,
               double *C64, int nthreads) {
    if (M < 1 || Nout < 1 || Kred < QO_GROUP || Kred % QO_GROUP || nthreads < 1) return -1;
    double *w = dequant_all(Wq, scales, biases, Nout, Kred, nthreads);
    double *a = bf16_matrix(A, M, Kred, nthreads);
    if (!w || !a) { free(w); free(a); return -4; }
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nout; ++n)
            C64[m * Nout + n] = dot(a + m * Kred, w + n * Kred, 0, Kred);
    free(w);
    free(a);
    return 0;
}

/* The same definition on a sample: out[i, j] = C64[rows[i], cols[j]].
 * Only the sampled weight rows are dequantized. */
int oracle_qmm_sampled(const uint16_t *A, const uint32_t *Wq, const uint16_t *scales,
                       const uint16_t *biases, int64_t M, int64_t Kred, int64_t Nout,
                       const int64_t *rows, int64_t nr, const int64_t *cols, int64_t nc,
                       double *out, int nthreads) {
    if (M < 1 || Nout < 1 || Kred < QO_GROUP || Kred % QO_GROUP || nthreads < 1) return -1;
    for (int64_t i = 0; i < nr; ++i) if (rows[i] < 0 || rows[i] >= M) return -1;
    for (int64_t j = 0; j < nc; ++j) if (cols[j] < 0 || cols[j] >= Nout) return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)(nc * Kred));
    double *a = (double *)malloc(sizeof(double) * (size_t)(nr * Kred));
    if (!w || !a) { free(w); free(a); return -4; }
    int bad = 0;
#pragma omp parallel for num_threads(nthreads) schedule(static) reduction(| : bad)
    for (int64_t j = 0; j < nc; ++j)
        bad |= dequant_row(Wq, scales, biases, Kred, cols[j], w + j * Kred) != 0;
    for (int64_t i = 0; i < nr; ++i)
        for (int64_t k = 0; k < Kred; ++k) a[i * Kred + k] = bf16_value(A[rows[i] * Kred + k]);
    if (!bad) {
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2)
        for (int64_t i = 0; i < nr; ++i)
            for (int64_t j = 0; j < nc; ++j)
                out[i * nc + j] = dot(a + i * Kred, w + j * Kred, 0, Kred);
    }
    free(w);
    free(a);
    return bad ? -1 : 0;
}

/* One output element of the partition emulation below: the fp64 sum of each
 * partition rounded to the plane type, the planes added in FP32 in
 * ascending p, the sum rounded once to BF16.  planes (nullable) receives
 * the split plane values. */
static int emulate_element(const double *am, const double *wn, int64_t Kred, int split,
                           int partial_mode, uint16_t *c, double *planes) {
    if (split == 1) {
        double exact = dot(am, wn, 0, Kred);
        if (planes) planes[0] = exact;
        return bf16_round(exact, c);
    }
    int64_t G = Kred / QO_GROUP, g0 = 0;
    float acc = 0.0f; /* the reduce adds the planes in FP32 */
    for (int p = 0; p < split; ++p) {
        int64_t ng = G / split + (p < G % split ? 1 : 0); /* groups in partition p */
        double exact = dot(am, wn, g0 * QO_GROUP, (g0 + ng) * QO_GROUP);
        g0 += ng;
        double plane;
        if (partial_mode == 0) {
            uint16_t pb;
            if (bf16_round(exact, &pb)) return -1;
            plane = bf16_value(pb);
        } else {
            plane = (double)(float)exact;
        }
        if (planes) planes[p] = plane;
        acc = acc + (float)plane;
    }
    return bf16_round((double)acc, c);
}

/* Partition emulation [TL, Task 2 and Task 4].  With split s dividing
 * G = Kred/128, partition p covers groups [p*G/s, (p+1)*G/s): equal length,
 * starting and ending on group boundaries.  A split that does not divide G
 * (1 < s <= G) cuts the groups into s slices as equal as whole groups allow,
 * in order, the first G mod s slices one group longer [SK, Concept: split-K
 * slices the reduction axis; the same rule as the dense GEMM below].
 * With s dividing G that is the equal cut.  Each partition's fp64 sum is
 * rounded to the partial-plane type (partial_mode 0: BF16, 1: FP32) and
 * stored in its own plane partial[p, m, n]; the planes are then added in
 * FP32 in ascending p and the sum is rounded once to BF16.  With s = 1 there
 * is no partial plane: C = BF16(C64).  Outputs: C_bf16 [M, Nout] and, if
 * partials is not NULL, the planes as doubles [s, M, Nout]. */
int oracle_qmm_partitioned(const uint16_t *A, const uint32_t *Wq, const uint16_t *scales,
                           const uint16_t *biases, int64_t M, int64_t Kred, int64_t Nout,
                           int split, int partial_mode, uint16_t *C_bf16, double *partials,
                           int nthreads) {
    if (M < 1 || Nout < 1 || Kred < QO_GROUP || Kred % QO_GROUP || nthreads < 1) return -1;
    int64_t G = Kred / QO_GROUP;
    if (split < 1 || split > 4096 || split > G || (partial_mode != 0 && partial_mode != 1))
        return -1;
    double *w = dequant_all(Wq, scales, biases, Nout, Kred, nthreads);
    double *a = bf16_matrix(A, M, Kred, nthreads);
    if (!w || !a) { free(w); free(a); return -4; }
    int bad = 0;
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2) reduction(| : bad)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < Nout; ++n) {
            double planes_mn[4096];
            uint16_t c;
            bad |= emulate_element(a + m * Kred, w + n * Kred, Kred, split, partial_mode, &c,
                                   partials ? planes_mn : NULL) != 0;
            C_bf16[m * Nout + n] = c;
            if (partials)
                for (int p = 0; p < split; ++p) partials[((int64_t)p * M + m) * Nout + n] = planes_mn[p];
        }
    free(w);
    free(a);
    return bad ? -1 : 0;
}

/* The partition emulation on a sample: out[i, j] = C_bf16[rows[i], cols[j]]
 * of oracle_qmm_partitioned, computed element by element; planes (nullable)
 * receives the split plane values, [nr, nc, split]. */
int oracle_qmm_partitioned_sampled(const uint16_t *A, const uint32_t *Wq, const uint16_t *scales,
                                   const uint16_t *biases, int64_t M, int64_t Kred, int64_t Nout,
                                   const int64_t *rows, int64_t nr, const int64_t *cols,
                                   int64_t nc, int split, int partial_mode, uint16_t *out,
                                   double *planes, int nthreads) {
    if (M < 1 || Nout < 1 || Kred < QO_GROUP || Kred % QO_GROUP || nthreads < 1) return -1;
    int64_t G = Kred / QO_GROUP;
    if (split < 1 || split > G || (partial_mode != 0 && partial_mode != 1)) return -1;
    for (int64_t i = 0; i < nr; ++i) if (rows[i] < 0 || rows[i] >= M) return -1;
    for (int64_t j = 0; j < nc; ++j) if (cols[j] < 0 || cols[j] >= Nout) return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)(nc * Kred));
    double *a = (double *)malloc(sizeof(double) * (size_t)(nr * Kred));
    if (!w || !a) { free(w); free(a); return -4; }
    int bad = 0;
#pragma omp parallel for num_threads(nthreads) schedule(static) reduction(| : bad)
    for (int64_t j = 0; j < nc; ++j)
        bad |= dequant_row(Wq, scales, biases, Kred, cols[j], w + j * Kred) != 0;
    for (int64_t i = 0; i < nr; ++i)
        for (int64_t k = 0; k < Kred; ++k) a[i * Kred + k] = bf16_value(A[rows[i] * Kred + k]);
    if (!bad) {
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2) reduction(| : bad)
        for (int64_t i = 0; i < nr; ++i)
            for (int64_t j = 0; j < nc; ++j)
                bad |= emulate_element(a + i * Kred, w + j * Kred, Kred, split, partial_mode,
                                       &out[i * nc + j],
                                       planes ? planes + (i * nc + j) * split : NULL) != 0;
    }
    free(w);
    free(a);
    return bad ? -1 : 0;
}

/* ---- occupancy policy and wave count ----------------------------------- */

/* [TL, Task 3]: base = ceil(M/BM)*ceil(Nout/BN);
 * s = min(cap, floor(target/base), Kred/128), then decreased by one until
 * Kred is divisible by s*128; s <= 1 means the unsplit kernel.  The
 * Kred/128 bound becomes floor(Kred/min_k) when a minimum number of
 * reduction elements per split is asked for [PD, step 5]; min_k = 128
 * is the rule as [TL] states it. */
int oracle_splitk_plan(int64_t M, int64_t Kred, int64_t Nout, int64_t bm, int64_t bn,
                       int64_t target, int64_t cap, int64_t min_k, int *split) {
    if (M < 1 || Nout < 1 || Kred < QO_GROUP || Kred % QO_GROUP) return -1;
    if (bm < 1 || bn < 1 || target < 0 || cap < 1 || min_k < QO_GROUP || min_k % QO_GROUP) return -1;
    int64_t base = ((M + bm - 1) / bm) * ((Nout + bn - 1) / bn);
    int64_t s = cap;
    if (target / base < s) s = target / base;
    if (Kred / min_k < s) s = Kred / min_k;
    while (s > 1 && Kred % (s * QO_GROUP) != 0) s -= 1;
    if (s <= 1) s = 1;
    *split = (int)s;
    return 0;
}

/* The plan for near-equal slices (no divisibility step).  B = min(cap,
 * floor(target/base), floor(Kred/min_k)) bounds the split as in [TL, Task 3];
 * B <= 1 means the unsplit kernel.  The longest slice holds ceil(G/s) groups,
 * and no split within the bound makes it shorter than L = ceil(G/B); the plan
 * takes the fewest slices that reach L, s = ceil(G/L).  That is the model of
 * [SK, Maths, Split-K]: the time falls with the work of the longest slice
 * while the blocks fit one wave, and more slices than needed only add partial
 * planes to reduce.  There the slices need not divide k: its A100 example
 * takes s = 6 of 256 k-tiles.  When B divides G the plan is B, the divisor
 * rule's split. */
int oracle_splitk_plan_near_equal(int64_t M, int64_t Kred, int64_t Nout, int64_t bm, int64_t bn,
                                  int64_t target, int64_t cap, int64_t min_k, int *split) {
    if (M < 1 || Nout < 1 || Kred < QO_GROUP || Kred % QO_GROUP) return -1;
    if (bm < 1 || bn < 1 || target < 0 || cap < 1 || min_k < QO_GROUP || min_k % QO_GROUP) return -1;
    int64_t G = Kred / QO_GROUP;
    int64_t base = ((M + bm - 1) / bm) * ((Nout + bn - 1) / bn);
    int64_t B = cap;
    if (target / base < B) B = target / base;
    if (Kred / min_k < B) B = Kred / min_k;
    if (B <= 1) {
        *split = 1;
        return 0;
    }
    int64_t L = (G + B - 1) / B; /* shortest reachable longest slice */
    *split = (int)((G + L - 1) / L);
    return 0;
}

/* [SK, Maths, Split-K]: tiles*s blocks run in ceil(tiles*s / SMs) waves. */
int64_t oracle_waves(int64_t tiles, int64_t split, int64_t sms) {
    if (tiles < 1 || split < 1 || sms < 1) return -1;
    return (tiles * split + sms - 1) / sms;
}

/* ---- dense BF16 split-K GEMM ------------------------------------------- */

/* C64[m, n] = sum_k A[m, k] * W[n, k] for BF16 A [M, K] and W [N, K]. */
int oracle_gemm(const uint16_t *A, const uint16_t *W, int64_t M, int64_t N, int64_t K,
                double *C64, int nthreads) {
    if (M < 1 || N < 1 || K < 1 || nthreads < 1) return -1;
    double *a = bf16_matrix(A, M, K, nthreads);
    double *w = bf16_matrix(W, N, K, nthreads);
    if (!a || !w) { free(a); free(w); return -4; }
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) C64[m * N + n] = dot(a + m * K, w + n * K, 0, K);
    free(a);
    free(w);
    return 0;
}

/* Split-K with k cut into T = K/ktile tiles, grouped into s slices [SK,
 * Concept: split-K].  When s does not divide T the slices are as
 * equal as whole tiles allow: the first T mod s slices get one extra tile.
 * Partial sums are FP32 planes [s, M, N] [SK, Maths: 4-byte partials];
 * the second pass adds them in FP32, ascending slice, and rounds to BF16. */
int oracle_gemm_partitioned(const uint16_t *A, const uint16_t *W, int64_t M, int64_t N,
                            int64_t K, int64_t ktile, int split, uint16_t *C_bf16,
                            int nthreads) {
    if (M < 1 || N < 1 || ktile < 1 || K < ktile || K % ktile || nthreads < 1) return -1;
    int64_t T = K / ktile;
    if (split < 1 || split > T) return -1;
    double *a = bf16_matrix(A, M, K, nthreads);
    double *w = bf16_matrix(W, N, K, nthreads);
    if (!a || !w) { free(a); free(w); return -4; }
    int bad = 0;
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2) reduction(| : bad)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            float acc = 0.0f;
            int64_t t0 = 0;
            for (int p = 0; p < split; ++p) {
                int64_t nt = T / split + (p < T % split ? 1 : 0);
                double exact = dot(a + m * K, w + n * K, t0 * ktile, (t0 + nt) * ktile);
                acc = acc + (float)exact;
                t0 += nt;
            }
            uint16_t c;
            bad |= bf16_round((double)acc, &c) != 0;
            C_bf16[m * N + n] = c;
        }
    free(a);
    free(w);
    return bad ? -1 : 0;
}

/* ---- copy / compute overlap schedule ----------------------------------- */

/* [SK, first Concept section and Maths, Overlap]: n tiles pass three engines
 * in tile order -- copy in (load), compute, copy out (store) -- each engine
 * working on one tile at a time.  With b buffers, tile i's load needs a free
 * buffer: it starts when tile i-1's load has ended and tile i-b's compute has
 * ended.  Tile i's compute starts when its load and tile i-1's compute have
 * ended; its store when its compute and tile i-1's store have ended.  The
 * schedule is built tile by tile from these rules (event by event, as the
 * page's model does) and T is the end of the last store.
 * out_reuse = 1 adds a rule the page's model leaves out: the outputs also sit
 * in b buffers, so tile i's compute also waits for tile i-b's store.
 * Per-tile times t_load[i], t_comp[i], t_store[i] >= 0.  events (nullable)
 * receives [n][6]: load start/end, compute start/end, store start/end. */
int oracle_overlap_schedule(int64_t n, int64_t b, const double *t_load, const double *t_comp,
                            const double *t_store, int out_reuse, double *T, double *events) {
    if (n < 1 || b < 1 || !t_load || !t_comp || !t_store || !T) return -1;
    if (out_reuse != 0 && out_reuse != 1) return -1;
    double *ev = (double *)malloc(sizeof(double) * (size_t)(6 * n));
    if (!ev) return -4;
    for (int64_t i = 0; i < n; ++i) {
        if (t_load[i] < 0 || t_comp[i] < 0 || t_store[i] < 0) { free(ev); return -1; }
        double *e = ev + 6 * i;
        double ls = i > 0 ? ev[6 * (i - 1) + 1] : 0.0;        /* previous load ended */
        if (i >= b && ev[6 * (i - b) + 3] > ls) ls = ev[6 * (i - b) + 3]; /* buffer free */
        e[0] = ls;
        e[1] = ls + t_load[i];
        double cs = e[1];                                      /* own load ended */
        if (i > 0 && ev[6 * (i - 1) + 3] > cs) cs = ev[6 * (i - 1) + 3];
        if (out_reuse && i >= b && ev[6 * (i - b) + 5] > cs) cs = ev[6 * (i - b) + 5];
        e[2] = cs;
        e[3] = cs + t_comp[i];
        double ss = e[3];                                      /* own compute ended */
        if (i > 0 && ev[6 * (i - 1) + 5] > ss) ss = ev[6 * (i - 1) + 5];
        e[4] = ss;
        e[5] = ss + t_store[i];
    }
    *T = ev[6 * (n - 1) + 5];
    if (events) memcpy(events, ev, sizeof(double) * (size_t)(6 * n));
    free(ev);
    return 0;
}

/* ---- split-KV decode attention ----------------------------------------- */

/* [PD, step 4 (decode attention), step 5 and Correctness requirements]:
 * one query token per sequence attends to its whole KV history.  q is BF16
 * [B, Hq, D]; K and V are BF16 [B, Hkv, Lmax, D] (head-major, contiguous
 * along the sequence); sequence b has lens[b] valid positions (1 <= lens[b]
 * <= Lmax).  Query head h reads KV head h / (Hq / Hkv) (grouped-query
 * attention; Hq a multiple of Hkv).
 *   O[b, h, :] = sum_{l < lens[b]} softmax_l(scale * q[b, h] . K[b, g, l]) V[b, g, l]
 * computed in fp64: the scores, their maximum, exp(s - max), their sum and
 * the weighted sum of V rows, then one division.  O is fp64 [B, Hq, D]. */
static int attn_check(int64_t B, int64_t Hq, int64_t Hkv, int64_t Lmax, int64_t D,
                      const int32_t *lens) {
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Lmax < 1 || D < 1 || !lens) return -1;
    for (int64_t b = 0; b < B; ++b)
        if (lens[b] < 1 || lens[b] > Lmax) return -1;
    return 0;
}

/* scores of one (b, h) over positions [l0, l1): s[l - l0] (fp64) */
static void attn_scores(const uint16_t *q, const uint16_t *K, int64_t b, int64_t h, int64_t Hq,
                        int64_t Hkv, int64_t Lmax, int64_t D, double scale, int64_t l0,
                        int64_t l1, double *s) {
    int64_t g = h / (Hq / Hkv);
    const uint16_t *qv = q + (b * Hq + h) * D;
    for (int64_t l = l0; l < l1; ++l) {
        const uint16_t *kv = K + ((b * Hkv + g) * Lmax + l) * D;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += bf16_value(qv[d]) * bf16_value(kv[d]);
        s[l - l0] = scale * acc;
    }
}

int oracle_decode_attention(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                            const int32_t *lens, int64_t B, int64_t Hq, int64_t Hkv, int64_t Lmax,
                            int64_t D, double scale, double *O, int nthreads) {
    if (!q || !K || !V || !O || nthreads < 1 || attn_check(B, Hq, Hkv, Lmax, D, lens)) return -1;
    int bad = 0;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic) collapse(2) reduction(| : bad)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < Hq; ++h) {
            int64_t L = lens[b], g = h / (Hq / Hkv);
            double *s = (double *)malloc(sizeof(double) * (size_t)L);
            if (!s) { bad = 1; continue; }
            attn_scores(q, K, b, h, Hq, Hkv, Lmax, D, scale, 0, L, s);
            double mx = s[0];
            for (int64_t l = 1; l < L; ++l) if (s[l] > mx) mx = s[l];
            double sum = 0.0;
            for (int64_t l = 0; l < L; ++l) { s[l] = exp(s[l] - mx); sum += s[l]; }
            double *o = O + (b * Hq + h) * D;
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t l = 0; l < L; ++l) {
                const uint16_t *vv = V + ((b * Hkv + g) * Lmax + l) * D;
                for (int64_t d = 0; d < D; ++d) o[d] += s[l] * bf16_value(vv[d]);
            }
            for (int64_t d = 0; d < D; ++d) o[d] /= sum;
            free(s);
        }
    return bad ? -4 : 0;
}

/* The split-KV algorithm [PD, step 4, step 5 and Correctness requirements],
 * in fp64: the positions of sequence b are cut into chunks of `chunk`
 * positions; chunk c gives a partial softmax state -- its maximum m_c, its
 * sum l_c of exp(s - m_c) and its unnormalized output o_c = sum exp(s - m_c)
 * V -- and the states are merged with the log-sum-exp correction:
 * M = max_c m_c, O = sum_c exp(m_c - M) o_c / sum_c exp(m_c - M) l_c
 * (merge 0).  merge 1 is the naive combine the page warns about: the mean
 * of the chunks' normalized outputs o_c / l_c, with no correction.  O is fp64
 * [B, Hq, D]. */
int oracle_decode_attention_split(const uint16_t *q, const uint16_t *K, const uint16_t *V,
                                  const int32_t *lens, int64_t B, int64_t Hq, int64_t Hkv,
                                  int64_t Lmax, int64_t D, double scale, int64_t chunk, int merge,
                                  double *O, int nthreads) {
    if (!q || !K || !V || !O || nthreads < 1 || chunk < 1 || (merge != 0 && merge != 1) ||
        attn_check(B, Hq, Hkv, Lmax, D, lens))
        return -1;
    int bad = 0;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic) collapse(2) reduction(| : bad)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < Hq; ++h) {
            int64_t L = lens[b], g = h / (Hq / Hkv), nc = (L + chunk - 1) / chunk;
            double *s = (double *)malloc(sizeof(double) * (size_t)chunk);
            double *m = (double *)malloc(sizeof(double) * (size_t)nc);
            double *l = (double *)malloc(sizeof(double) * (size_t)nc);
            double *oc = (double *)malloc(sizeof(double) * (size_t)(nc * D));
            if (!s || !m || !l || !oc) { bad = 1; free(s); free(m); free(l); free(oc); continue; }
            for (int64_t c = 0; c < nc; ++c) {
                int64_t l0 = c * chunk, l1 = l0 + chunk < L ? l0 + chunk : L;
                attn_scores(q, K, b, h, Hq, Hkv, Lmax, D, scale, l0, l1, s);
                double mx = s[0];
                for (int64_t t = 1; t < l1 - l0; ++t) if (s[t] > mx) mx = s[t];
                m[c] = mx;
                l[c] = 0.0;
                for (int64_t d = 0; d < D; ++d) oc[c * D + d] = 0.0;
                for (int64_t t = 0; t < l1 - l0; ++t) {
                    double p = exp(s[t] - mx);
                    l[c] += p;
                    const uint16_t *vv = V + ((b * Hkv + g) * Lmax + l0 + t) * D;
                    for (int64_t d = 0; d < D; ++d) oc[c * D + d] += p * bf16_value(vv[d]);
                }
            }
            double *o = O + (b * Hq + h) * D;
            if (merge == 0) {
                double M = m[0];
                for (int64_t c = 1; c < nc; ++c) if (m[c] > M) M = m[c];
                double den = 0.0;
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int64_t c = 0; c < nc; ++c) {
                    double w = exp(m[c] - M);
                    den += w * l[c];
                    for (int64_t d = 0; d < D; ++d) o[d] += w * oc[c * D + d];
                }
                for (int64_t d = 0; d < D; ++d) o[d] /= den;
            } else {
                for (int64_t d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int64_t c = 0; c < nc; ++c) acc += oc[c * D + d] / l[c];
                    o[d] = acc / (double)nc;
                }
            }
            free(s); free(m); free(l); free(oc);
        }
    return bad ? -4 : 0;
}

/* [PD, step 5]: the split-KV factor.  S = ceil(SMs * blocks_per_sm /
 * (B * Hkv)) blocks of work per (sequence, KV head), at least 1, clamped so
 * every split keeps at least min_chunk positions of the longest sequence:
 * S <= max(1, floor(Lmax / min_chunk)). */
int oracle_attention_splits(int64_t B, int64_t Hkv, int64_t Lmax, int64_t sms,
                            int64_t blocks_per_sm, int64_t min_chunk, int *splits) {
    if (B < 1 || Hkv < 1 || Lmax < 1 || sms < 1 || blocks_per_sm < 1 || min_chunk < 1 || !splits)
        return -1;
    int64_t work = B * Hkv;
    int64_t S = (sms * blocks_per_sm + work - 1) / work;
    int64_t cap = Lmax / min_chunk;
    if (cap < 1) cap = 1;
    if (S > cap) S = cap;
    if (S < 1) S = 1;
    *splits = (int)S;
    return 0;
}
