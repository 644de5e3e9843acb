/*
 * kda_solve_tril.h -- C ABI of the KDA prefill chunk solver for sm_103a.
 *
 * Operation (LightLLM PR #1703, "perf(kda): parallelize diagonal solves in
 * Prefill", PR description): KDA prefill splits every sequence into chunks of
 * 64 tokens.  For every chunk and every head the solver inverts the unit
 * lower-triangular matrix (I + A), where A is the chunk's strictly
 * lower-triangular 64x64 block.  The four independent 16x16 diagonal blocks
 * are inverted in parallel and then merged into the 64x64 inverse with the
 * off-diagonal inverse tiles kept in FP32,
 *
 *     Linv_ii = (I + A_ii)^-1,
 *     Linv_ij = -Linv_ii * sum_{k=j}^{i-1} A_ik * Linv_kj      (i > j).
 *
 * The same page says the shared solver's branch for 64-token chunks handles
 * packed and dense batches, and that it decides whether to split from the FP32
 * workspace budget and a minimum input length, the workspace being capped at
 * the size of the input in FP32.  The split path runs the diagonal inverses as their own kernel and
 * keeps the four FP32 16x16 inverse tiles of every chunk-head in a caller
 * workspace; the single-pass path does everything on chip.  Both paths give
 * bit-identical results.
 *
 * Layouts (all tensors contiguous, row-major, last dimension = 64):
 *   dense : A, Ai are [B, T, H, 64]; chunks restart at t = 0 of each batch row.
 *   packed: A, Ai are [1, T, H, 64] with T = cu_seqlens[num_seqs]; request s
 *           covers rows [cu_seqlens[s], cu_seqlens[s+1]) and its chunks start at
 *           cu_seqlens[s] + 64 c.  The last chunk of a row or request may hold
 *           n < 64 rows.
 * Element (row i, column j) of chunk-head (c, h) is A[t0 + i, h, j] with t0 the
 * chunk's first row.  Only the strictly lower part of the valid n x n block is
 * read (j < i < n); the diagonal, the upper triangle and anything at or past
 * column n may hold any bits, NaN included.  Output rows t0 .. t0+n-1 of Ai
 * are written in full: the n x n inverse, an exact 1.0 diagonal, exact zeros
 * above it and exact zeros in columns n .. 63.  No other element of Ai is
 * touched.
 *
 * Ownership: the caller owns every buffer (A, Ai, cu_seqlens, workspace); the
 * library allocates no device memory and keeps no per-call state.  All device
 * calls are asynchronous on the given stream (a cudaStream_t passed as void*;
 * NULL = the legacy default stream) and do not synchronise the host.  The
 * single-pass, short-chunk and fused kernels are launched with programmatic
 * stream serialization (the split path's two kernels are not): one may be scheduled
 * onto the SMs while the previous kernel of its stream finishes, but it waits
 * for that kernel to complete, with its writes visible, before it reads or
 * writes any global memory, so stream order holds as for ordinary launches.
 *
 * Stream capture: the first call of each entry point on a device sets up
 * per-device state (device attributes, the error word's address, kernel
 * attributes and occupancy), so make it outside a CUDA-graph capture; later
 * calls only encode tensor maps on the host (the last 16 distinct (A, Ai,
 * dtypes, H, rows) encodings are kept and reused) and launch kernels, and can
 * be captured.  kda_solve_tril_host also creates its copy streams on first use.
 * That per-device state lives until the process exits and does not survive a
 * cudaDeviceReset (or anything else that destroys the device's primary
 * context): after one, do not call the library on that device again.
 *
 * Errors: every function returns a kda_status_t.  Argument errors are found on
 * the host before any CUDA call and leave all buffers untouched.  KDA_ERR_CUDA
 * reports a launch failure (cudaGetLastError); faults during asynchronous
 * execution surface at the caller's next synchronisation, as for any CUDA
 * kernel.  A kernel whose bounded wait for its own TMA copies runs out (it
 * never should) stops, and records a code that kda_device_error() returns.
 */
#ifndef KDA_SOLVE_TRIL_H
#define KDA_SOLVE_TRIL_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_BT 64                 /* chunk length of every entry point but kda_solve_tril_bt */
#define KDA_WS_TILE_BYTES 4096    /* FP32 workspace per chunk-head: 4 tiles of 16x16 */

typedef enum {
    KDA_F32 = 0,
    KDA_BF16 = 1,
    KDA_F16 = 2
} kda_dtype_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* bad pointer, size, alignment, overlap or layout */
    KDA_ERR_UNSUPPORTED = 2,      /* dtype or size the library does not handle */
    KDA_ERR_WORKSPACE = 3,        /* split path forced with a missing or too small workspace */
    KDA_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    KDA_ERR_DEVICE = 5            /* kda_device_error() found a recorded device-side error */
} kda_status_t;

typedef enum {
    KDA_PATH_AUTO = 0,            /* let the selector decide (kda_solve_tril_select) */
    KDA_PATH_SPLIT = 1,           /* diagonal-inverse kernel + merge kernel, FP32 workspace */
    KDA_PATH_SINGLE = 2           /* one kernel, no workspace */
} kda_path_t;

/* Precision mode of the merge products (the PR description lists precision
 * modes among the solver's regression axes; see kda_solve_tril_prec). */
typedef enum {
    KDA_PREC_IEEE = 0,            /* FP32-accurate: split-TF32 products (the default of every entry) */
    KDA_PREC_TF32 = 1             /* plain TF32 products: faster, about 2^-9 relative per product */
} kda_precision_t;

/* Smallest B*T (total rows) for which the selector takes the split path (the
 * minimum input length of the same PR description).  Set from GB300
 * measurements: the single-pass kernel already inverts the four diagonal
 * blocks in parallel inside one CTA, so splitting only adds the workspace round
 * trip and a launch, and it was slower at every size measured (64 to 131072
 * rows); the threshold therefore lies above any size the library supports. */
#define KDA_SPLIT_MIN_TOKENS (INT64_C(1) << 32)

/*
 * Workspace bytes the split path needs for this shape: KDA_WS_TILE_BYTES per
 * chunk-head, for an upper bound on the number of chunks that needs no look at
 * cu_seqlens: B * ceil(T/64) (dense, num_seqs == 0) or min(T, floor((T +
 * 63 * num_seqs) / 64)) (packed, num_seqs >= 1).  Returns 0 for an empty or
 * invalid shape.
 */
KDA_API size_t kda_solve_tril_workspace_size(int64_t B, int64_t T, int32_t H, int32_t num_seqs);

/*
 * The path KDA_PATH_AUTO takes for this shape with a workspace of
 * workspace_bytes (0 = none): KDA_PATH_SPLIT iff the workspace is at least
 * kda_solve_tril_workspace_size(), that size is at most the FP32 input size
 * B*T*H*64*4 bytes (equivalently, chunks are on average at least 16 rows full:
 * the choice rests on chunk occupancy) and B*T >= KDA_SPLIT_MIN_TOKENS;
 * KDA_PATH_SINGLE otherwise.  Pure host arithmetic.
 */
KDA_API kda_path_t kda_solve_tril_select(int64_t B, int64_t T, int32_t H, int32_t num_seqs,
                                 size_t workspace_bytes);

/*
 * Solve every chunk-head: Ai = (I + strict_lower(A))^-1 per chunk and head.
 *
 *   A           device, [B, T, H, 64] of in_dtype, 16-byte aligned, read only.
 *   Ai          device, same shape, out_dtype, 16-byte aligned; must not overlap A.
 *   cu_seqlens  device int32 [num_seqs + 1], or NULL for the dense layout.
 *               Packed requires B == 1, num_seqs >= 1, cu_seqlens[0] == 0,
 *               non-decreasing entries and cu_seqlens[num_seqs] == T; the values
 *               are not read on the host.  Malformed values give unspecified
 *               results but every access stays inside rows [0, T).
 *   num_seqs    number of requests (packed) or 0 (dense).
 *   B, T, H     shape; T == 0 or B == 0 is a no-op returning KDA_OK.  H >= 1,
 *               H * 64 * 64 < 2^31 (H < 524288), B*T < 2^31 and
 *               (chunks * H) < 2^30; larger sizes give KDA_ERR_UNSUPPORTED.
 *   in_dtype    KDA_F32 / KDA_BF16 / KDA_F16; values are widened to FP32.
 *   out_dtype   KDA_F32 / KDA_BF16 / KDA_F16; FP32 results rounded to nearest even.
 *   workspace   device, 16-byte aligned, or NULL; used only by the split path.
 *   workspace_bytes  its size.
 *   stream      cudaStream_t to launch on.
 *
 * Computes in FP32: FP32 FMA for the diagonal inverses, split-TF32 tensor-core
 * products (three TF32 products per FP32 product, FP32 accumulation) for the
 * merge; result within 2e-5*(1+|ref|) of the exact inverse of the
 * FP32-widened input on the specified workloads.
 */
KDA_API kda_status_t kda_solve_tril(const void *A, void *Ai, const int32_t *cu_seqlens,
                            int32_t num_seqs, int64_t B, int64_t T, int32_t H,
                            int32_t in_dtype, int32_t out_dtype, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * kda_solve_tril with the path forced.  path = KDA_PATH_AUTO behaves exactly
 * like kda_solve_tril; KDA_PATH_SPLIT returns KDA_ERR_WORKSPACE when the
 * workspace is NULL or smaller than kda_solve_tril_workspace_size();
 * KDA_PATH_SINGLE ignores the workspace.  *path_taken (if not NULL) receives
 * the path that ran (KDA_PATH_SPLIT or KDA_PATH_SINGLE).
 */
KDA_API kda_status_t kda_solve_tril_ex(const void *A, void *Ai, const int32_t *cu_seqlens,
                               int32_t num_seqs, int64_t B, int64_t T, int32_t H,
                               int32_t in_dtype, int32_t out_dtype, void *workspace,
                               size_t workspace_bytes, void *stream, int32_t path,
                               int32_t *path_taken);

/*
 * End-to-end call for callers whose data lives in host memory: copies A (and
 * cu_seqlens) from host to the caller's device buffers, solves, and copies Ai
 * back.  The caller synchronises `stream` before reading Ai_host; the stream
 * waits for the whole call.  Host buffers should be pinned (page-locked) for
 * the copies to be asynchronous.  A_dev / Ai_dev / cu_dev / workspace follow
 * the rules of kda_solve_tril; cu_seqlens_host and cu_dev are both NULL for
 * the dense layout (cu_seqlens_host is read on the host).
 *
 * Calls moving more than 32 MiB are cut into up to 8 pieces at chunk
 * boundaries (whole batch rows, 64-row multiples of a batch row, or whole
 * requests); the piece copies run on two non-blocking streams that the library
 * creates once per device and keeps until the process exits, so host-to-device
 * copies, solves and device-to-host copies of different pieces overlap.  No
 * device memory is allocated.
 */
KDA_API kda_status_t kda_solve_tril_host(const void *A_host, void *Ai_host, const int32_t *cu_seqlens_host,
                                 int32_t num_seqs, int64_t B, int64_t T, int32_t H,
                                 int32_t in_dtype, int32_t out_dtype, void *A_dev, void *Ai_dev,
                                 int32_t *cu_dev, void *workspace, size_t workspace_bytes,
                                 void *stream);

/* Size of the workspace built into the library for kda_solve_tril_split_static. */
#define KDA_STATIC_WS_BYTES (64u << 20)

/*
 * Split-path solve that allocates nothing and takes no workspace.  The PR has
 * no counterpart to this entry point.
 *
 * It is for callers that cannot allocate device memory where they call the
 * solver: a plugin inside a host framework that owns all device memory and
 * gives its plugins no allocation hook, or a serving loop that fixed its memory
 * at start-up and must not call cudaMalloc / cudaFree later (those calls can
 * synchronise the device).  The caller still passes A, Ai and cu_seqlens, with
 * the meaning, layout and rules of kda_solve_tril; the split path's FP32
 * workspace is a static device array of KDA_STATIC_WS_BYTES (64 MiB) inside the
 * library, held by every GPU that loads the library until the process exits.
 *
 *   - Argument errors (those of kda_solve_tril) are reported before any CUDA
 *     call.  Shapes whose workspace (kda_solve_tril_workspace_size) exceeds
 *     KDA_STATIC_WS_BYTES are rejected with KDA_ERR_WORKSPACE, also before any
 *     CUDA call; 64 MiB holds 16384 chunk-heads, e.g. the 16 x 512-token,
 *     64-head packed solve (35.75 MiB).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls whose kernels
 *     overlap on the GPU -- on different streams or from different host
 *     threads -- race on it and give wrong results: issue them in order on one
 *     stream.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
KDA_API kda_status_t kda_solve_tril_split_static(const void *A, void *Ai, const int32_t *cu_seqlens,
                                                 int32_t num_seqs, int64_t B, int64_t T, int32_t H,
                                                 int32_t in_dtype, int32_t out_dtype, void *stream);

/*
 * The same solve for chunks of bt = 16, 32 or 64 tokens.  The PR description
 * presents the path it optimises as the shared solver's branch for 64-token
 * chunks; the solver's other branches invert (I + A) for shorter chunks, with A
 * the chunk's strictly lower-triangular bt x bt block:
 *
 *   bt = 16  one forward substitution per chunk-head (the 16x16 diagonal
 *            inverse on its own);
 *   bt = 32  two 16x16 diagonal inverses and one merge step,
 *            Linv_10 = -Linv_11 * A_10 * Linv_00, in split TF32 on the tensor
 *            cores;
 *   bt = 64  kda_solve_tril_ex with KDA_PATH_SINGLE (no workspace).
 *
 * Every argument has the meaning, layout and rules of kda_solve_tril with 64
 * replaced by bt: A and Ai are [B, T, H, bt] (dense, chunks restart at t = 0 of
 * each batch row) or [1, T, H, bt] with cu_seqlens (packed, chunks restart at
 * every request start); the last chunk may hold n < bt rows; only j < i < n of
 * a chunk's block is read; output rows of a chunk are written in full (the
 * n x n inverse, exact ones on the diagonal, exact zeros elsewhere) and no
 * other element of Ai is touched.  H * bt * bt < 2^31, B*T < 2^31 and
 * (chunks * H) < 2^30, counted with chunks of bt rows.  Returns
 * KDA_ERR_UNSUPPORTED for any other bt.
 * Accuracy: within 2e-5*(1+|ref|) of the exact inverse of the FP32-widened
 * input on the specified workloads, as for kda_solve_tril.
 */
KDA_API kda_status_t kda_solve_tril_bt(const void *A, void *Ai, const int32_t *cu_seqlens,
                                       int32_t num_seqs, int64_t B, int64_t T, int32_t H, int32_t bt,
                                       int32_t in_dtype, int32_t out_dtype, void *stream);

/*
 * The 64-token solve with the chunk matrix built on chip from the quantities
 * KDA prefill builds it from (on the same page, KDA prefill is a user of the
 * shared solver):
 *
 *     A[i][j] = beta[i] * sum_d k[i][d] * k[j][d] * exp(g[i][d] - g[j][d])   (j < i),
 *
 * per chunk and head, for the chunk's token rows i, j; Ai = (I + A)^-1 is
 * written as by kda_solve_tril.  A itself is never stored.
 *
 *   k           device, [B, T, H, K] of in_dtype (keys), 16-byte aligned.
 *   g           device, [B, T, H, K] float32: per-channel cumulative log decay;
 *               only differences inside a chunk are used, so g may restart at
 *               chunk starts or run on.  16-byte aligned.  g must not increase
 *               along a chunk (each token's decay is at most 1); how far it
 *               falls is not limited.  A channel whose g, over the chunk's
 *               live rows, lies more than 48 from its value at the chunk's
 *               middle live row (row (n - 1) / 2 of a chunk of n rows) takes
 *               a slower path for that chunk-head (KDA's decays, about one
 *               per token, do not).
 *   beta        device, [B, T, H] of in_dtype, aligned to its element size.
 *   Ai          device, [B, T, H, 64] of out_dtype, 16-byte aligned; must not
 *               overlap k, g or beta.
 *   cu_seqlens, num_seqs, B, T, H, stream: as for kda_solve_tril (layouts,
 *               partial last chunks, size limits).
 *   K           channels: 32, 64, 96 or 128 (KDA_ERR_UNSUPPORTED otherwise).
 *   in_dtype    KDA_F32 / KDA_BF16 / KDA_F16 for k and beta (widened to FP32).
 *   out_dtype   KDA_F32 / KDA_BF16 / KDA_F16.
 *
 * Computes in FP32 (exp, split-TF32 tensor-core products with FP32
 * accumulation, the solve of kda_solve_tril); within 2e-5*(1+|ref|) of the
 * exact inverse of the matrix built from the given (rounded) inputs on the
 * specified workloads.
 */
KDA_API kda_status_t kda_solve_tril_kgb(const void *k, const float *g, const void *beta, void *Ai,
                                        const int32_t *cu_seqlens, int32_t num_seqs, int64_t B, int64_t T,
                                        int32_t H, int32_t K, int32_t in_dtype, int32_t out_dtype,
                                        void *stream);

/*
 * The single-pass 64-token solve in a chosen precision mode (no workspace; the
 * split path has the FP32-accurate mode only).
 *
 *   precision   KDA_PREC_IEEE: exactly kda_solve_tril_ex with KDA_PATH_SINGLE.
 *               KDA_PREC_TF32: the four diagonal 16x16 inverses as in the IEEE
 *               mode (FP32 forward substitution), but each 16x16 merge product
 *               as one TF32 tensor-core product: both operands truncated to
 *               TF32 (10 explicit mantissa bits; 16-bit input is exact), FP32
 *               accumulation.  Each product then carries a relative error of
 *               about 2^-9 of |P| |Q| instead of about 2^-21, so the result is
 *               not within the IEEE mode's 2e-5*(1+|ref|); its error is bounded
 *               elementwise by 2^-6 * (|X| |L| |X| + |X| |L| |X| |L| |X|), with X
 *               the exact inverse and L the strictly lower A.
 *               Anything else: KDA_ERR_INVALID_ARGUMENT.
 *   All other arguments, layouts, rules and errors: as for kda_solve_tril.
 */
KDA_API kda_status_t kda_solve_tril_prec(const void *A, void *Ai, const int32_t *cu_seqlens, int32_t num_seqs,
                                         int64_t B, int64_t T, int32_t H, int32_t in_dtype, int32_t out_dtype,
                                         int32_t precision, void *stream);

/*
 * Self-test of the device-side failure detection.  Launches one thread on
 * `stream` that waits, with the kernels' bounded wait and a limit of limit_us
 * microseconds, on an mbarrier that completes only if `complete` is non-zero.
 * With complete = 0 the wait runs out, the kernel records bit 1 in the device
 * error word and returns (about limit_us plus up to 6.4 ms later); the context
 * stays usable.  Read the word with kda_device_error.
 *   limit_us    1 .. 1000000, else KDA_ERR_INVALID_ARGUMENT (before any CUDA call).
 */
KDA_API kda_status_t kda_selftest_wait(int32_t complete, uint32_t limit_us, void *stream);

/* Static description of a status code (never NULL). */
KDA_API const char *kda_status_string(int32_t status);

/*
 * Read and clear the device-side error word of `device` (synchronises that
 * device).  *code receives 0 when no kernel of this library recorded an
 * error since the last call, else a bit set (1 = a bounded TMA wait ran out).
 * Returns KDA_OK, or KDA_ERR_CUDA when the device cannot be queried.
 */
KDA_API kda_status_t kda_device_error(int32_t device, uint32_t *code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
KDA_API int32_t kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_SOLVE_TRIL_H */
