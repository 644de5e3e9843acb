/*
 * kda_oracle.c -- fp64 CPU oracle for the KDA prefill chunk solver.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (LightLLM PR #1703, "perf(kda): parallelize diagonal solves
 * in Prefill", PR description): for every 64-token chunk of every head, the
 * inverse of the unit lower-triangular matrix (I + A), where A is the chunk's
 * strictly lower-triangular 64x64 block.  The PR's method (four diagonal
 * 16x16 inverses merged into the 64x64 inverse) reaches exactly this inverse
 * up to rounding order, so the oracle is the plain definition: row-by-row
 * forward substitution in fp64 on the already-rounded input values,
 *
 *     X[i][i] = 1,   X[i][j] = - sum_{k=j}^{i-1} M[i][k] * X[k][j]   (j < i),
 *
 * with M[i][k] = A[row0 + i, h, k] for k < i < n and n = the chunk's number of
 * valid rows.  Elements on or above the diagonal of A, and rows past n, are
 * never read.  Output row i (< n) is X[i][0..n) followed by 64 - n zeros.
 *
 * Chunk boundaries (readings of the packed and dense batches the same PR
 * description supports): dense [B, T, H, 64] restarts chunks at t = 0 of every
 * batch row; packed [1, T, H, 64] with cu_seqlens restarts at every request
 * start cu_seqlens[s]; the last chunk of a row/request may be partial.
 *
 * The same page presents this as the shared solver's branch for 64-token
 * chunks, so the chunk length is a parameter here (the _bt entry points; 16, 32 and 64 are
 * used): the definition above is unchanged with 64 replaced by the chunk
 * length bt.
 *
 * The chunk matrix itself (the _kgb entry point): KDA prefill builds A from the
 * keys k, the per-token betas and the per-channel cumulative log decays g of
 * the chunk's tokens, and on the same page KDA prefill is a user of the shared
 * solver.  The construction, written out as its definition with one exp per
 * term (no factorisation of the decay), is
 *
 *     A[i][j] = beta[i] * sum_d k[i][d] * k[j][d] * exp(g[i][d] - g[j][d])
 *
 * for j < i < n and zero elsewhere; only differences of g inside one chunk
 * enter, so g may restart at chunk starts or run on.
 *
 * Build: plain C99, -O2 -ffp-contract=off (no fused multiply-add, so the x86
 * and Arm builds give identical bits), optional -fopenmp.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_BT 64

/* Planted mistakes for the negative-control tests (compiled only into
 * throw-away copies built by the test suite). */
#ifndef KDA_ORACLE_PLANT
#define KDA_ORACLE_PLANT 0
#endif

/* Invert one chunk of length bt.  M: row-major with leading dimension ldm;
 * only M[i*ldm+k] with k < i < n is read.  X: bt x bt row-major output (rows
 * >= n are left as identity rows, columns >= n are zero). */
void kda_oracle_invert_chunk_bt(const double *M, int64_t ldm, int n, int bt, double *X)
{
    memset(X, 0, sizeof(double) * bt * bt);
    for (int i = 0; i < bt; ++i) X[i * bt + i] = 1.0;
    for (int i = 1; i < n; ++i) {
        for (int j = 0; j < i; ++j) {
            double s = 0.0;
            int kend = i;
#if KDA_ORACLE_PLANT == 1
            kend = i - 1;                /* planted: drops the k = i-1 term */
#endif
            for (int k = j; k < kend; ++k) s += M[i * ldm + k] * X[k * bt + j];
#if KDA_ORACLE_PLANT == 2
            X[i * bt + j] = s;           /* planted: wrong sign */
#else
            X[i * bt + j] = -s;
#endif
        }
    }
}

/* The 64-token chunk (X is 64 x 64). */
void kda_oracle_invert_chunk(const double *M, int64_t ldm, int n, double *X)
{
    kda_oracle_invert_chunk_bt(M, ldm, n, KDA_ORACLE_BT, X);
}

typedef struct {
    int64_t row0;   /* first row on the flattened B*T axis */
    int n;          /* valid rows */
} kda_oracle_chunk_t;

/* Enumerate chunks of length bt; returns the count (writes up to cap entries). */
static int64_t kda_oracle_chunks(const int32_t *cu, int32_t nseq, int64_t B, int64_t T, int bt,
                                 kda_oracle_chunk_t *out, int64_t cap)
{
    int64_t c = 0;
    if (cu == NULL) {
        for (int64_t b = 0; b < B; ++b)
            for (int64_t t0 = 0; t0 < T; t0 += bt) {
                if (c < cap) {
                    out[c].row0 = b * T + t0;
                    out[c].n = (int)((T - t0) < bt ? (T - t0) : bt);
                }
                ++c;
            }
    } else {
        for (int32_t s = 0; s < nseq; ++s) {
            int64_t start = cu[s], end = cu[s + 1];
#if KDA_ORACLE_PLANT == 3
            if (s > 0) start += 1;       /* planted: chunk boundary shifted by a token */
#endif
            for (int64_t t0 = start; t0 < end; t0 += bt) {
                if (c < cap) {
                    out[c].row0 = t0;
                    out[c].n = (int)((end - t0) < bt ? (end - t0) : bt);
                }
                ++c;
            }
        }
    }
    return c;
}

/* Solve every chunk-head, chunk length bt.  A, Ai: fp64 [rows, H, bt] with
 * rows = B*T, row-major, contiguous.  cu_seqlens (int32 [nseq+1]) selects the
 * packed layout (then B must be 1); NULL selects the dense layout.  Rows of Ai
 * that belong to no chunk are left untouched.  Returns 0, or -1 on a bad
 * argument. */
int kda_oracle_solve_tril_bt(const double *A, double *Ai, const int32_t *cu_seqlens,
                             int32_t nseq, int64_t B, int64_t T, int32_t H, int32_t bt)
{
    if (H <= 0 || T < 0 || B < 0 || bt < 1 || bt > 64) return -1;
    if (cu_seqlens != NULL && (B != 1 || nseq < 0)) return -1;
    int64_t nc = kda_oracle_chunks(cu_seqlens, nseq, B, T, bt, NULL, 0);
    kda_oracle_chunk_t *ch = (kda_oracle_chunk_t *)malloc(sizeof(*ch) * (size_t)(nc > 0 ? nc : 1));
    if (!ch) return -1;
    kda_oracle_chunks(cu_seqlens, nseq, B, T, bt, ch, nc);
    const int64_t ld = (int64_t)H * bt;          /* row stride of A / Ai in elements */
    const int64_t ntask = nc * H;
#pragma omp parallel
    {
        double *X = (double *)malloc(sizeof(double) * bt * bt);
#pragma omp for schedule(dynamic, 8)
        for (int64_t q = 0; q < ntask; ++q) {
            const kda_oracle_chunk_t c = ch[q / H];
            const int64_t h = q % H;
            const double *M = A + c.row0 * ld + h * bt;
            kda_oracle_invert_chunk_bt(M, ld, c.n, bt, X);
            for (int i = 0; i < c.n; ++i)
                memcpy(Ai + (c.row0 + i) * ld + h * bt, X + i * bt, sizeof(double) * bt);
        }
        free(X);
    }
    free(ch);
    return 0;
}

/* Chunk matrix of one chunk-head (64 x 64 row-major into M) from the chunk's
 * rows of k and g (K channels, row stride ldk elements) and beta (row stride
 * ldb); rows i, j < n are used, everything else of M is zero. */
static void kda_oracle_kgb_chunk(const double *k, const double *g, const double *beta, int64_t ldk,
                                 int64_t ldb, int n, int K, double *M)
{
    memset(M, 0, sizeof(double) * KDA_ORACLE_BT * KDA_ORACLE_BT);
    for (int i = 1; i < n; ++i) {
        for (int j = 0; j < i; ++j) {
            double s = 0.0;
            for (int d = 0; d < K; ++d) {
#if KDA_ORACLE_PLANT == 4
                const double e = exp(g[j * ldk + d] - g[i * ldk + d]);   /* planted: decay reversed */
#else
                const double e = exp(g[i * ldk + d] - g[j * ldk + d]);
#endif
                s += k[i * ldk + d] * k[j * ldk + d] * e;
            }
#if KDA_ORACLE_PLANT == 5
            M[i * KDA_ORACLE_BT + j] = beta[j * ldb] * s;                 /* planted: beta of the column */
#else
            M[i * KDA_ORACLE_BT + j] = beta[i * ldb] * s;
#endif
        }
    }
}

/* Build every 64-token chunk's A from k, g, beta and solve it.  k, g: fp64
 * [rows, H, K]; beta: fp64 [rows, H]; Ai (and A_out if not NULL): fp64
 * [rows, H, 64], rows = B*T, written on the rows of every chunk only.  Layouts
 * as for kda_oracle_solve_tril.  Returns 0, or -1 on a bad argument. */
int kda_oracle_solve_kgb(const double *k, const double *g, const double *beta, double *Ai, double *A_out,
                         const int32_t *cu_seqlens, int32_t nseq, int64_t B, int64_t T, int32_t H, int32_t K)
{
    if (H <= 0 || T < 0 || B < 0 || K < 1) return -1;
    if (cu_seqlens != NULL && (B != 1 || nseq < 0)) return -1;
    const int bt = KDA_ORACLE_BT;
    int64_t nc = kda_oracle_chunks(cu_seqlens, nseq, B, T, bt, NULL, 0);
    kda_oracle_chunk_t *ch = (kda_oracle_chunk_t *)malloc(sizeof(*ch) * (size_t)(nc > 0 ? nc : 1));
    if (!ch) return -1;
    kda_oracle_chunks(cu_seqlens, nseq, B, T, bt, ch, nc);
    const int64_t ldk = (int64_t)H * K, ldo = (int64_t)H * bt;
    const int64_t ntask = nc * H;
#pragma omp parallel
    {
        double *M = (double *)malloc(sizeof(double) * bt * bt);
        double *X = (double *)malloc(sizeof(double) * bt * bt);
#pragma omp for schedule(dynamic, 4)
        for (int64_t q = 0; q < ntask; ++q) {
            const kda_oracle_chunk_t c = ch[q / H];
            const int64_t h = q % H;
            kda_oracle_kgb_chunk(k + c.row0 * ldk + h * K, g + c.row0 * ldk + h * K, beta + c.row0 * H + h,
                                 ldk, H, c.n, K, M);
            kda_oracle_invert_chunk_bt(M, bt, c.n, bt, X);
            for (int i = 0; i < c.n; ++i) {
                memcpy(Ai + (c.row0 + i) * ldo + h * bt, X + i * bt, sizeof(double) * bt);
                if (A_out) memcpy(A_out + (c.row0 + i) * ldo + h * bt, M + i * bt, sizeof(double) * bt);
            }
        }
        free(M);
        free(X);
    }
    free(ch);
    return 0;
}

/* The 64-token branch. */
int kda_oracle_solve_tril(const double *A, double *Ai, const int32_t *cu_seqlens,
                          int32_t nseq, int64_t B, int64_t T, int32_t H)
{
    return kda_oracle_solve_tril_bt(A, Ai, cu_seqlens, nseq, B, T, H, KDA_ORACLE_BT);
}

/* Number of 64-token chunks a layout holds (the chunk enumeration above). */
int64_t kda_oracle_num_chunks(const int32_t *cu_seqlens, int32_t nseq, int64_t B, int64_t T)
{
    return kda_oracle_chunks(cu_seqlens, nseq, B, T, KDA_ORACLE_BT, NULL, 0);
}

/* Threads an OpenMP parallel region of this library uses (1 without OpenMP). */
int kda_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Which mistake this copy was compiled with (0 = the real oracle). */
int kda_oracle_planted(void) { return KDA_ORACLE_PLANT; }
