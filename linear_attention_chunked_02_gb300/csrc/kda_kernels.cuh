// kda_kernels.cuh -- sm_103a kernels of the KDA prefill chunk solver.
//
// Operation (LightLLM PR #1703, "perf(kda): parallelize diagonal solves in
// Prefill", PR description): per 64-token chunk and head, (I + A)^-1 for the
// strictly lower-triangular 64x64 chunk matrix A.  The four 16x16 diagonal
// blocks are inverted independently and in parallel; the inverse tiles stay in
// FP32 through the merge into the 64x64 inverse.
//
// GB300 design
//   * One persistent CTA of 64 threads (four 16-lane "units") per resident
//     slot; a CTA walks its chunk-heads q = blockIdx.x, blockIdx.x + grid, ...
//     (q = chunk * H + head, so neighbouring CTAs share the chunk's token rows).
//   * A thread issues TMA tile loads (cp.async.bulk.tensor, mbarrier
//     completion) for the next chunk-head while the CTA computes the current
//     one (2-stage ring).  Only the ten lower 16x16 blocks of each chunk are
//     fetched: block-row r as one box of 16 rows x 16(r+1) columns.
//   * Diagonal blocks: one unit per block, one lane per column, forward
//     substitution in registers (fp32 FMA).
//   * Merge, as two 32x32 levels (the 64x64 matrix is lower block-triangular
//     with 32x32 blocks TL, BR and off-diagonal BL):
//        level A: X10 = -(X11 A10) X00,  X32 = -(X33 A32) X22
//        level B: U = X_BR A_BL,  X_BL = -U X_TL
//     which is Linv_ij = -Linv_ii sum_k A_ik Linv_kj regrouped.  Every product
//     is a 16x16x16 FP32 FMA product computed by one unit with a 4x4 register
//     tile per lane; products with a triangular factor skip the k-quads whose
//     factor entries are structurally zero.
//   * The output tile (n rows x 64 columns incl. exact zeros and the unit
//     diagonal) is written with 16-byte coalesced stores.
//   * Split path: MODE_DIAG runs only the diagonal inverses and stores their
//     FP32 tiles to the workspace; MODE_MERGE loads them back and runs the
//     merge.  Both call the same device functions as MODE_FUSED, so every
//     element is computed with the same operations in the same order.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kda {

constexpr int BT = 64;          // chunk length
constexpr int BS = 16;          // diagonal block size
constexpr int NTHREADS = 64;    // four 16-lane units
constexpr int STAGES = 2;

constexpr int MODE_FUSED = 0;
constexpr int MODE_DIAG = 1;
constexpr int MODE_MERGE = 2;

// FP32 on-chip tiles.  A blocks: pitch 16, block stride 272 floats (1088 B) so
// that blocks with odd slot distance sit in different bank quads.  X / U
// blocks: pitch 20 floats (rows 4 apart land in distinct bank quads), block
// stride 336 floats (1344 B).
constexpr int AP = 16;
constexpr int ABS = 272;
constexpr int XP = 20;
constexpr int XBS = 336;

__host__ __device__ constexpr int blk(int i, int j) { return i * (i + 1) / 2 + j; }

// transposed-copy slots and U slots
constexpr int T_X00 = 0, T_X22 = 1, T_X11 = 2, T_X10 = 3;
constexpr int U_00 = 0, U_10 = 1, U_01 = 2, U_11 = 3;

// device-side error word (bit 0: a bounded TMA wait ran out)
constexpr unsigned ERR_WAIT_TIMEOUT = 1u;
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;   // 1 s

struct Params {
    void *out;                 // Ai (MODE_FUSED / MODE_MERGE)
    float *ws;                 // workspace tiles (MODE_DIAG writes, MODE_MERGE reads)
    const int32_t *cu;         // packed: cu_seqlens (device); dense: nullptr
    int32_t nseq;
    int32_t H;
    int64_t T;                 // dense: rows per batch row; packed: total rows
    int64_t rows;              // B * T
    int32_t cpr;               // dense: chunks per batch row
    int32_t n_tasks;           // loop bound on chunk-head indices
    unsigned *err;             // device error word
};

struct Meta {
    int32_t row0;              // first row of the chunk on the flattened B*T axis
    int32_t n;                 // valid rows (0 = nothing to store)
    int32_t h;
    int32_t valid;             // 0 = past the last chunk-head: stop
};

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase `parity` of `bar`; gives up after WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u && globaltimer() - t0 > WAIT_LIMIT_NS) return false;
    }
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
          "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// --------------------------------------------------------- dtype helpers
template <typename T> struct Elt;
template <> struct Elt<float> {
    static constexpr int VEC = 4;            // elements per 16-byte vector
    __device__ static __forceinline__ void widen(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};
template <> struct Elt<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ static __forceinline__ void widen(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {                      // bf16 -> fp32 is exact
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <> struct Elt<__half> {
    static constexpr int VEC = 8;
    __device__ static __forceinline__ void widen(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h2 = *reinterpret_cast<const __half2 *>(&w[i]);
            const float2 t = __half22float2(h2);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
};

// 8 fp32 -> 16 bytes of bf16 / fp16 (round to nearest even)
__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16 *) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half *) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------------------------ smem layout
template <int MODE, typename TIn>
struct Layout {
    static constexpr int ELT = sizeof(TIn);
    // stage: raw TMA landing area
    static constexpr int A_ELEMS = MODE == MODE_FUSED ? 10 * 256 : MODE == MODE_DIAG ? 4 * 256 : 6 * 256;
    static constexpr int A_BYTES = A_ELEMS * ELT;
    static constexpr int WS_OFF = (A_BYTES + 127) / 128 * 128;
    static constexpr int STAGE_BYTES = MODE == MODE_MERGE ? WS_OFF + 4096 : WS_OFF;
    static constexpr uint32_t TX_BYTES = MODE == MODE_MERGE ? A_BYTES + 4096 : A_BYTES;
    static constexpr int NAF = MODE == MODE_DIAG ? 4 : 10;     // A-block slots
    static constexpr int NXN = MODE == MODE_DIAG ? 0 : 10;     // X-block slots
    static constexpr int NXT = MODE == MODE_DIAG ? 0 : 4;
    static constexpr int NU = MODE == MODE_DIAG ? 0 : 4;
    static constexpr int OFF_BAR = 0;
    static constexpr int OFF_META = 64;
    static constexpr int OFF_STAGE = 128;
    static constexpr int OFF_AF = OFF_STAGE + STAGES * STAGE_BYTES;
    static constexpr int OFF_XN = OFF_AF + NAF * ABS * 4;
    static constexpr int OFF_XT = OFF_XN + NXN * XBS * 4;
    static constexpr int OFF_U = OFF_XT + NXT * XBS * 4;
    static constexpr int BYTES = OFF_U + NU * XBS * 4;
    // stage offset (bytes) of block-row r's box
    __host__ __device__ static constexpr int row_off(int r) {
        return MODE == MODE_FUSED ? 256 * ELT * (r * (r + 1) / 2)
             : MODE == MODE_DIAG  ? 256 * ELT * r
                                  : 256 * ELT * ((r - 1) * r / 2);
    }
};

// A-block slot of block (i, j) in the Af area
template <int MODE>
__device__ __forceinline__ int af_slot(int i, int j) { return MODE == MODE_DIAG ? i : blk(i, j); }

// ------------------------------------------------------------ task decode
// Per-CTA state of the walk over cu_seqlens (packed layout).
struct Walk {
    int32_t s;        // current request
    int32_t cbase;    // chunks before request s
};

__device__ __forceinline__ int32_t nchunks(int32_t a, int32_t b) {
    const int32_t L = b - a;
    return L > 0 ? (L + BT - 1) / BT : 0;
}

__device__ __forceinline__ Meta decode(const Params &p, int32_t q, Walk &w) {
    Meta m{0, 0, 0, 0};
    if (q >= p.n_tasks) return m;
    const int32_t c = q / p.H;
    m.h = q - c * p.H;
    if (p.cu == nullptr) {
        const int32_t b = c / p.cpr;
        const int32_t cc = c - b * p.cpr;
        const int64_t t0 = int64_t(cc) * BT;
        m.row0 = static_cast<int32_t>(int64_t(b) * p.T + t0);
        const int64_t left = p.T - t0;
        m.n = static_cast<int32_t>(left < BT ? left : BT);
        m.valid = 1;
        return m;
    }
    // advance to the request that holds chunk c (tasks of a CTA increase)
    while (w.s < p.nseq) {
        const int32_t a = __ldg(p.cu + w.s), b = __ldg(p.cu + w.s + 1);
        const int32_t nc = nchunks(a, b);
        if (c < w.cbase + nc) {
            int64_t r0 = int64_t(a) + int64_t(c - w.cbase) * BT;
            int64_t end = b < p.T ? b : p.T;                  // clamp malformed cu_seqlens
            if (r0 < 0) r0 = 0;
            int64_t n = end - r0;
            if (n > BT) n = BT;
            if (n < 0 || r0 >= p.T) n = 0;
            m.row0 = static_cast<int32_t>(r0 < p.T ? r0 : 0);
            m.n = static_cast<int32_t>(n);
            m.valid = 1;
            return m;
        }
        w.cbase += nc;
        ++w.s;
    }
    return m;
}

// Issue the loads of task q into stage `st` (one thread).
template <int MODE, typename TIn>
__device__ __forceinline__ void issue(const Params &p, const CUtensorMap *maps, int32_t q, Walk &w,
                                      unsigned char *smem, int st) {
    using L = Layout<MODE, TIn>;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR) + st;
    Meta *meta = reinterpret_cast<Meta *>(smem + L::OFF_META) + st;
    const Meta m = decode(p, q, w);
    *meta = m;
    if (!m.valid) {
        mbar_arrive(bar);
        return;
    }
    unsigned char *stage = smem + L::OFF_STAGE + st * L::STAGE_BYTES;
    mbar_arrive_expect_tx(bar, L::TX_BYTES);
    if (MODE == MODE_FUSED) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
            tma_load_3d(stage + L::row_off(r), &maps[r], 0, m.h, m.row0 + 16 * r, bar);
    } else if (MODE == MODE_DIAG) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
            tma_load_3d(stage + L::row_off(r), &maps[0], 16 * r, m.h, m.row0 + 16 * r, bar);
    } else {
#pragma unroll
        for (int r = 1; r < 4; ++r)
            tma_load_3d(stage + L::row_off(r), &maps[r - 1], 0, m.h, m.row0 + 16 * r, bar);
        bulk_load(stage + L::WS_OFF, p.ws + size_t(q) * 1024, 4096, bar);
    }
}

// --------------------------------------------------------- stage -> FP32
// Box of block-row r: 16 rows x (16 * nb) elements starting at block column c0.
// Rows at or past n become exact zeros (they may hold the next request's data).
template <int MODE, typename TIn, int R, int C0, int NB>
__device__ __forceinline__ void widen_box(const unsigned char *src, float *Af, int n, int tid) {
    constexpr int VEC = Elt<TIn>::VEC;
    constexpr int W = 16 * NB;
    constexpr int VPR = W / VEC;              // vectors per row
    constexpr int NV = 16 * VPR;
    const bool full = n >= 16 * R + 16;
#pragma unroll
    for (int e0 = 0; e0 < NV; e0 += NTHREADS) {
        const int e = e0 + tid;
        if (NV % NTHREADS == 0 || e < NV) {
            const int i = e / VPR;
            const int k = (e - i * VPR) * VEC;
            const uint4 v = *reinterpret_cast<const uint4 *>(src + (i * W + k) * int(sizeof(TIn)));
            float f[VEC];
            Elt<TIn>::widen(v, f);
            const bool keep = full || (16 * R + i < n);
            float *dst = Af + af_slot<MODE>(R, C0 + k / 16) * ABS + i * AP + (k & 15);
#pragma unroll
            for (int t = 0; t < VEC; t += 4) {
                float4 o;
                o.x = keep ? f[t] : 0.f;
                o.y = keep ? f[t + 1] : 0.f;
                o.z = keep ? f[t + 2] : 0.f;
                o.w = keep ? f[t + 3] : 0.f;
                *reinterpret_cast<float4 *>(dst + t) = o;
            }
        }
    }
}

// ------------------------------------------------------ diagonal inverse
// Unit-lower-triangular 16x16 inverse by forward substitution, one lane per
// column j: x[i] = -sum_{k<i} a[i][k] x[k] for i > j, x[j] = 1, x[i<j] = 0.
// `a` holds the block (pitch AP); only entries with k < i are used.
__device__ __forceinline__ void diag_invert(const float *a, int j, float (&x)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
        float s = 0.f;
#pragma unroll
        for (int kq = 0; kq < (i + 3) / 4; ++kq) {
            const float4 v = *reinterpret_cast<const float4 *>(a + i * AP + 4 * kq);
            if (4 * kq + 0 < i) s = fmaf(v.x, x[4 * kq + 0], s);
            if (4 * kq + 1 < i) s = fmaf(v.y, x[4 * kq + 1], s);
            if (4 * kq + 2 < i) s = fmaf(v.z, x[4 * kq + 2], s);
            if (4 * kq + 3 < i) s = fmaf(v.w, x[4 * kq + 3], s);
        }
        x[i] = (i > j) ? -s : x[i];
    }
}

// ----------------------------------------------------------- 16x16 products
// A unit computes a 16x16 tile; lane l (0..15): rg = l >> 2, cg = l & 3.
// acc[m][n] is row rg + 4m.  prod_left: column 4cg + n.  prod_right: column cg + 4n.

__device__ __forceinline__ float comp(const float4 &v, int kk) {
    return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
}

// acc += P Q; P row-major (pitch pp), Q row-major (pitch qp).  LTRI: P is lower
// triangular, so k-quad q only meets rows m >= q.
template <bool LTRI>
__device__ __forceinline__ void prod_left(float (&acc)[4][4], const float *__restrict__ P, int pp,
                                          const float *__restrict__ Q, int qp, int rg, int cg) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float4 pr[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (!LTRI || m >= q) pr[m] = *reinterpret_cast<const float4 *>(P + (rg + 4 * m) * pp + 4 * q);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float4 qv = *reinterpret_cast<const float4 *>(Q + (4 * q + kk) * qp + 4 * cg);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (LTRI && m < q) continue;
                const float a = comp(pr[m], kk);
                acc[m][0] = fmaf(a, qv.x, acc[m][0]);
                acc[m][1] = fmaf(a, qv.y, acc[m][1]);
                acc[m][2] = fmaf(a, qv.z, acc[m][2]);
                acc[m][3] = fmaf(a, qv.w, acc[m][3]);
            }
        }
    }
}

// acc += P R with R given transposed (Rt[c * XP + k] = R[k][c]).  RTRI: R is
// lower triangular, so column cg + 4n only meets k-quads q >= n.
template <bool RTRI>
__device__ __forceinline__ void prod_right(float (&acc)[4][4], const float *__restrict__ P, int pp,
                                           const float *__restrict__ Rt, int rg, int cg) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float4 pr[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) pr[m] = *reinterpret_cast<const float4 *>(P + (rg + 4 * m) * pp + 4 * q);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            if (RTRI && n > q) continue;
            const float4 rt = *reinterpret_cast<const float4 *>(Rt + (cg + 4 * n) * XP + 4 * q);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                acc[m][n] = fmaf(pr[m].x, rt.x, acc[m][n]);
                acc[m][n] = fmaf(pr[m].y, rt.y, acc[m][n]);
                acc[m][n] = fmaf(pr[m].z, rt.z, acc[m][n]);
                acc[m][n] = fmaf(pr[m].w, rt.w, acc[m][n]);
            }
        }
    }
}

__device__ __forceinline__ void zero(float (&acc)[4][4]) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[m][n] = 0.f;
}

// tile from prod_left (columns 4cg + n) -> row-major block
__device__ __forceinline__ void put_left(float *dst, const float (&acc)[4][4], int rg, int cg) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
        *reinterpret_cast<float4 *>(dst + (rg + 4 * m) * XP + 4 * cg) =
            make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
}
// -tile from prod_right (columns cg + 4n) -> row-major block (+ transposed copy)
__device__ __forceinline__ void put_right_neg(float *dst, float *dstT, const float (&acc)[4][4], int rg,
                                              int cg) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) dst[(rg + 4 * m) * XP + cg + 4 * n] = -acc[m][n];
    if (dstT != nullptr) {
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int m = 0; m < 4; ++m) dstT[(cg + 4 * n) * XP + rg + 4 * m] = -acc[m][n];
    }
}

// ------------------------------------------------------------------ merge
// Inputs: Xn diagonal blocks (row-major), Xt transposed X00/X11/X22, Af
// off-diagonal A blocks.  Outputs: the six off-diagonal X blocks in Xn.
__device__ __forceinline__ void merge(const float *Af, float *Xn, float *Xt, float *U, int tid) {
    const int unit = tid >> 4, warp = tid >> 5, half = unit & 1;
    const int l = tid & 15, rg = l >> 2, cg = l & 3;
    float acc[4][4];
    // level A (warp 0): X10 = -(X11 A10) X00 ; X32 = -(X33 A32) X22
    if (warp == 0) {
        zero(acc);
        prod_left<true>(acc, Xn + (half ? blk(3, 3) : blk(1, 1)) * XBS, XP,
                        Af + (half ? blk(3, 2) : blk(1, 0)) * ABS, AP, rg, cg);
        put_left(U + half * XBS, acc, rg, cg);
        __syncwarp();
        zero(acc);
        prod_right<true>(acc, U + half * XBS, XP, Xt + (half ? T_X22 : T_X00) * XBS, rg, cg);
        put_right_neg(Xn + (half ? blk(3, 2) : blk(1, 0)) * XBS, half ? nullptr : Xt + T_X10 * XBS, acc,
                      rg, cg);
    }
    __syncthreads();
    // level B, step 1: U = X_BR A_BL
    zero(acc);
    if (warp == 0) {     // U00 = X22 A20 ; U01 = X22 A21
        prod_left<true>(acc, Xn + blk(2, 2) * XBS, XP, Af + blk(2, half) * ABS, AP, rg, cg);
        put_left(U + (half ? U_01 : U_00) * XBS, acc, rg, cg);
    } else {             // U10 = X32 A20 + X33 A30 ; U11 = X32 A21 + X33 A31
        prod_left<false>(acc, Xn + blk(3, 2) * XBS, XP, Af + blk(2, half) * ABS, AP, rg, cg);
        prod_left<true>(acc, Xn + blk(3, 3) * XBS, XP, Af + blk(3, half) * ABS, AP, rg, cg);
        put_left(U + (half ? U_11 : U_10) * XBS, acc, rg, cg);
    }
    __syncthreads();
    // level B, step 2: X_BL = -U X_TL
    zero(acc);
    if (warp == 0) {     // X21 = -U01 X11 ; X31 = -U11 X11
        prod_right<true>(acc, U + (half ? U_11 : U_01) * XBS, XP, Xt + T_X11 * XBS, rg, cg);
        put_right_neg(Xn + (half ? blk(3, 1) : blk(2, 1)) * XBS, nullptr, acc, rg, cg);
    } else {             // X20 = -(U00 X00 + U01 X10) ; X30 = -(U10 X00 + U11 X10)
        prod_right<true>(acc, U + (half ? U_10 : U_00) * XBS, XP, Xt + T_X00 * XBS, rg, cg);
        prod_right<false>(acc, U + (half ? U_11 : U_01) * XBS, XP, Xt + T_X10 * XBS, rg, cg);
        put_right_neg(Xn + (half ? blk(3, 0) : blk(2, 0)) * XBS, nullptr, acc, rg, cg);
    }
    __syncthreads();
}

// ----------------------------------------------------------- output store
template <typename TOut>
__device__ __forceinline__ void store_tile(TOut *out, const Meta &m, int H, const float *Xn, int tid);

template <>
__device__ __forceinline__ void store_tile<float>(float *out, const Meta &m, int H, const float *Xn, int tid) {
    // 64 rows x 16 float4; thread covers rows (tid >> 4) + 4v, float4 column tid & 15
    const int c4 = tid & 15, bc = c4 >> 2;
#pragma unroll
    for (int v = 0; v < 16; ++v) {
        const int r = (tid >> 4) + 4 * v;
        if (r < m.n) {
            const int br = r >> 4;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (bc <= br) val = *reinterpret_cast<const float4 *>(Xn + blk(br, bc) * XBS + (r & 15) * XP + 4 * (c4 & 3));
            float *dst = out + (int64_t(m.row0 + r) * H + m.h) * BT + 4 * c4;
            *reinterpret_cast<float4 *>(dst) = val;
        }
    }
}

template <typename TOut>
__device__ __forceinline__ void store_tile_16(TOut *out, const Meta &m, int H, const float *Xn, int tid) {
    // 64 rows x 8 groups of 8; thread covers rows (tid >> 3) + 8v, group tid & 7
    const int c8 = tid & 7, bc = c8 >> 1;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const int r = (tid >> 3) + 8 * v;
        if (r < m.n) {
            const int br = r >> 4;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (bc <= br) {
                const float *src = Xn + blk(br, bc) * XBS + (r & 15) * XP + 8 * (c8 & 1);
                a = *reinterpret_cast<const float4 *>(src);
                b = *reinterpret_cast<const float4 *>(src + 4);
            }
            uint4 o;
            o.x = pack2(a.x, a.y, (TOut *)nullptr);
            o.y = pack2(a.z, a.w, (TOut *)nullptr);
            o.z = pack2(b.x, b.y, (TOut *)nullptr);
            o.w = pack2(b.z, b.w, (TOut *)nullptr);
            TOut *dst = out + (int64_t(m.row0 + r) * H + m.h) * BT + 8 * c8;
            *reinterpret_cast<uint4 *>(dst) = o;
        }
    }
}
template <>
__device__ __forceinline__ void store_tile<__nv_bfloat16>(__nv_bfloat16 *out, const Meta &m, int H,
                                                          const float *Xn, int tid) {
    store_tile_16(out, m, H, Xn, tid);
}
template <>
__device__ __forceinline__ void store_tile<__half>(__half *out, const Meta &m, int H, const float *Xn, int tid) {
    store_tile_16(out, m, H, Xn, tid);
}

// ----------------------------------------------------------------- kernel
struct Maps {
    CUtensorMap m[4];          // box widths 16, 32, 48, 64 columns; 16 rows; 1 head
};

template <int MODE, typename TIn, typename TOut>
__global__ void __launch_bounds__(NTHREADS)
kda_tril_kernel(const __grid_constant__ Maps maps, const Params p) {
    using L = Layout<MODE, TIn>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    const Meta *metas = reinterpret_cast<const Meta *>(smem + L::OFF_META);
    float *Af = reinterpret_cast<float *>(smem + L::OFF_AF);
    float *Xn = reinterpret_cast<float *>(smem + L::OFF_XN);
    float *Xt = reinterpret_cast<float *>(smem + L::OFF_XT);
    float *U = reinterpret_cast<float *>(smem + L::OFF_U);
    const int tid = threadIdx.x;
    const int32_t G = gridDim.x;
    Walk walk{0, 0};

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        fence_proxy_async();
        for (int s = 0; s < STAGES; ++s)
            issue<MODE, TIn>(p, maps.m, int32_t(blockIdx.x) + s * G, walk, smem, s);
    }
    __syncthreads();

    for (int it = 0;; ++it) {
        const int st = it % STAGES;
        const uint32_t parity = (it / STAGES) & 1;
        const bool ok = mbar_wait_bounded(&bars[st], parity);
        if (__syncthreads_or(!ok)) {
            // A copy never completed.  Record it, give the other stage's copy a
            // bounded chance to land, and stop; nothing else is in flight.
            if (tid == 0) {
                atomicOr(p.err, ERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bars[(st + 1) % STAGES], ((it + 1) / STAGES) & 1);
            }
            return;
        }
        const Meta m = metas[st];
        if (!m.valid) break;
        const unsigned char *stage = smem + L::OFF_STAGE + st * L::STAGE_BYTES;
        const int32_t q = int32_t(blockIdx.x) + it * G;

        // stage -> FP32 tiles (masked)
        if (MODE == MODE_FUSED) {
            widen_box<MODE, TIn, 0, 0, 1>(stage + L::row_off(0), Af, m.n, tid);
            widen_box<MODE, TIn, 1, 0, 2>(stage + L::row_off(1), Af, m.n, tid);
            widen_box<MODE, TIn, 2, 0, 3>(stage + L::row_off(2), Af, m.n, tid);
            widen_box<MODE, TIn, 3, 0, 4>(stage + L::row_off(3), Af, m.n, tid);
        } else if (MODE == MODE_DIAG) {
            widen_box<MODE, TIn, 0, 0, 1>(stage + L::row_off(0), Af, m.n, tid);
            widen_box<MODE, TIn, 1, 1, 1>(stage + L::row_off(1), Af, m.n, tid);
            widen_box<MODE, TIn, 2, 2, 1>(stage + L::row_off(2), Af, m.n, tid);
            widen_box<MODE, TIn, 3, 3, 1>(stage + L::row_off(3), Af, m.n, tid);
        } else {
            widen_box<MODE, TIn, 1, 0, 1>(stage + L::row_off(1), Af, m.n, tid);
            widen_box<MODE, TIn, 2, 0, 2>(stage + L::row_off(2), Af, m.n, tid);
            widen_box<MODE, TIn, 3, 0, 3>(stage + L::row_off(3), Af, m.n, tid);
            // workspace tile: 4 row-major 16x16 FP32 diagonal inverses
            const float *wt = reinterpret_cast<const float *>(stage + L::WS_OFF);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int e = tid + NTHREADS * v;          // float4 index 0..255
                const int u = e >> 6, i = (e >> 2) & 15, k4 = e & 3;
                const float4 x = *reinterpret_cast<const float4 *>(wt + u * 256 + i * 16 + 4 * k4);
                *reinterpret_cast<float4 *>(Xn + blk(u, u) * XBS + i * XP + 4 * k4) = x;
                if (u < 3) {
                    float *t = Xt + (u == 0 ? T_X00 : u == 1 ? T_X11 : T_X22) * XBS;
                    t[(4 * k4 + 0) * XP + i] = x.x;
                    t[(4 * k4 + 1) * XP + i] = x.y;
                    t[(4 * k4 + 2) * XP + i] = x.z;
                    t[(4 * k4 + 3) * XP + i] = x.w;
                }
            }
        }
        __syncthreads();
        if (tid == 0) {                      // refill the stage just drained
            fence_proxy_async();
            issue<MODE, TIn>(p, maps.m, q + STAGES * G, walk, smem, st);
        }

        if (MODE != MODE_MERGE) {
            const int unit = tid >> 4, j = tid & 15;
            float x[16];
            diag_invert(Af + af_slot<MODE>(unit, unit) * ABS, j, x);
            if (MODE == MODE_DIAG) {
                float *w = p.ws + size_t(q) * 1024 + unit * 256 + j;
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i * 16] = x[i];
                continue;
            }
            float *xn = Xn + blk(unit, unit) * XBS;
#pragma unroll
            for (int i = 0; i < 16; ++i) xn[i * XP + j] = x[i];
            if (unit < 3) {
                float *t = Xt + (unit == 0 ? T_X00 : unit == 1 ? T_X11 : T_X22) * XBS + j * XP;
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4 *>(t + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
            }
            __syncthreads();
        }
        if (MODE != MODE_DIAG) {
            merge(Af, Xn, Xt, U, tid);
            store_tile<TOut>(reinterpret_cast<TOut *>(p.out), m, p.H, Xn, tid);
        }
    }
}

}  // namespace kda
