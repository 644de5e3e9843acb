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
//   * Thread 0 issues TMA tile loads (cp.async.bulk.tensor, mbarrier
//     completion) into a 2-stage ring, so the next chunk-head is in flight
//     while the current one is computed.  Only the ten lower 16x16 blocks are
//     fetched: block-row r as one box of 16 rows x 16(r+1) columns.  FP32 input
//     is used in place from the landing buffer; 16-bit input is widened once.
//   * Diagonal blocks: one unit per block, one lane per column, forward
//     substitution in registers (FP32 FMA).
//   * Merge, as two 32x32 levels (the 64x64 matrix is lower block-triangular
//     with 32x32 blocks TL, BR and off-diagonal BL):
//        level A: X10 = -(X11 A10) X00,  X32 = -(X33 A32) X22
//        level B: U = X_BR A_BL,  X_BL = -U X_TL
//     which is Linv_ij = -Linv_ii sum_k A_ik Linv_kj regrouped.  Each 16x16x16
//     FP32 product is computed by one unit with a 4x4 register tile per lane.
//     The U blocks are kept negated (U' = -U), so only two product kinds
//     exist: "lower-triangular left factor, negated" (which skips the k-quads
//     where the diagonal inverse is structurally zero) and "dense".  The
//     products run as a 4-step loop over a fixed schedule in which all four
//     units are busy in every step; one call site per product kind keeps the
//     code small enough for the instruction cache.
//   * Every output block is stored straight from the registers that computed
//     it (16-byte row segments), the zero blocks above the diagonal directly.
//   * Split path: MODE_DIAG inverts the diagonal blocks, writes them (and the
//     zero blocks) to the output and their FP32 tiles to the workspace;
//     MODE_MERGE loads the tiles back and produces the off-diagonal blocks.
//     Both call the same device functions as MODE_FUSED, so every element is
//     computed with the same operations in the same order.
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

// On-chip FP32 tiles.  X / U blocks: pitch 20 floats (rows 4 apart land in
// distinct bank quads), block stride 336 floats.  Widened 16-bit A blocks:
// pitch 16, block stride 272 floats.
constexpr int XP = 20;
constexpr int XBS = 336;
constexpr int AP16 = 16;
constexpr int ABS = 272;

__host__ __device__ constexpr int blk(int i, int j) { return i * (i + 1) / 2 + j; }

// X slots 0..3 hold the diagonal inverses X00..X33; slot 4 X10, slot 5 -X32.
constexpr int XS_10 = 4, XS_32N = 5;
// Diagonal block inverted by each unit: warp 0 takes X11 and X33, warp 1 X00
// and X22, so that the first merge step only needs the unit's own warp.
__host__ __device__ constexpr int diag_of_unit(int u) { return u == 0 ? 1 : u == 1 ? 3 : u == 2 ? 0 : 2; }

// device-side error word (bit 0: a bounded TMA wait ran out)
constexpr unsigned ERR_WAIT_TIMEOUT = 1u;
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;   // 1 s

struct Params {
    void *out;                 // Ai
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

// output element conversion (round to nearest even)
__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16 *) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half *) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void put1(float *p, float v) { *p = v; }
__device__ __forceinline__ void put1(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void put1(__half *p, float v) { *p = __float2half_rn(v); }
// four consecutive output elements
__device__ __forceinline__ void put4(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}
template <typename TOut>
__device__ __forceinline__ void put4(TOut *p, float a, float b, float c, float d) {
    uint2 o;
    o.x = pack2(a, b, (TOut *)nullptr);
    o.y = pack2(c, d, (TOut *)nullptr);
    *reinterpret_cast<uint2 *>(p) = o;
}

// ------------------------------------------------------------ smem layout
template <int MODE, typename TIn>
struct Layout {
    static constexpr int ELT = sizeof(TIn);
    static constexpr bool WIDEN = ELT == 2;
    // stage: raw TMA landing area
    static constexpr int A_ELEMS = MODE == MODE_FUSED ? 10 * 256 : MODE == MODE_DIAG ? 4 * 256 : 6 * 256;
    static constexpr int A_BYTES = A_ELEMS * ELT;
    static constexpr int WS_OFF = (A_BYTES + 127) / 128 * 128;
    static constexpr int STAGE_BYTES = MODE == MODE_MERGE ? WS_OFF + 4096 : WS_OFF;
    static constexpr uint32_t TX_BYTES = MODE == MODE_MERGE ? A_BYTES + 4096 : A_BYTES;
    static constexpr int NAF = WIDEN ? (MODE == MODE_DIAG ? 4 : 10) : 0;   // widened A-block slots
    static constexpr int NX = MODE == MODE_DIAG ? 0 : 6;
    static constexpr int NU = MODE == MODE_DIAG ? 0 : 4;
    static constexpr int OFF_BAR = 0;
    static constexpr int OFF_META = 64;
    static constexpr int OFF_STAGE = 128;
    static constexpr int OFF_AF = OFF_STAGE + STAGES * STAGE_BYTES;
    static constexpr int OFF_X = OFF_AF + NAF * ABS * 4;
    static constexpr int OFF_U = OFF_X + NX * XBS * 4;
    static constexpr int BYTES = OFF_U + NU * XBS * 4;
    // stage offset (bytes) of block-row r's box, and the box width in elements
    __host__ __device__ static constexpr int row_off(int r) {
        return MODE == MODE_FUSED ? 256 * ELT * (r * (r + 1) / 2)
             : MODE == MODE_DIAG  ? 256 * ELT * r
                                  : 256 * ELT * ((r - 1) * r / 2);
    }
    __host__ __device__ static constexpr int width(int r) {
        return MODE == MODE_FUSED ? 16 * (r + 1) : MODE == MODE_DIAG ? 16 : 16 * r;
    }
    static constexpr int R0 = MODE == MODE_MERGE ? 1 : 0;   // first block-row fetched
};

// A-block slot of block (i, j) in the widened area
template <int MODE>
__device__ __forceinline__ int af_slot(int i, int j) { return MODE == MODE_DIAG ? i : blk(i, j); }

// An FP32 view of A block (i, j): pointer and row pitch (floats).
struct AView {
    const float *p;
    int pitch;
};
template <int MODE, typename TIn>
__device__ __forceinline__ AView aview(const unsigned char *stage, const float *Af, int i, int j) {
    using L = Layout<MODE, TIn>;
    if (L::WIDEN) return {Af + af_slot<MODE>(i, j) * ABS, AP16};
    const float *base = reinterpret_cast<const float *>(stage + L::row_off(i));
    if (MODE == MODE_DIAG) return {base, 16};
    return {base + 16 * j, L::width(i)};
}

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

// ------------------------------------------------------ operand preparation
// 16-bit input: block-row R's box (16 rows x 16*NB elements from block column
// C0) widened to FP32 tiles; rows at or past n become exact zeros (they may
// hold the next request's rows).
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
            float *dst = Af + af_slot<MODE>(R, C0 + k / 16) * ABS + i * AP16 + (k & 15);
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

template <int MODE, typename TIn>
__device__ __forceinline__ void widen_all(const unsigned char *stage, float *Af, int n, int tid) {
    using L = Layout<MODE, TIn>;
    if (MODE == MODE_FUSED) {
        widen_box<MODE, TIn, 0, 0, 1>(stage + L::row_off(0), Af, n, tid);
        widen_box<MODE, TIn, 1, 0, 2>(stage + L::row_off(1), Af, n, tid);
        widen_box<MODE, TIn, 2, 0, 3>(stage + L::row_off(2), Af, n, tid);
        widen_box<MODE, TIn, 3, 0, 4>(stage + L::row_off(3), Af, n, tid);
    } else if (MODE == MODE_DIAG) {
        widen_box<MODE, TIn, 0, 0, 1>(stage + L::row_off(0), Af, n, tid);
        widen_box<MODE, TIn, 1, 1, 1>(stage + L::row_off(1), Af, n, tid);
        widen_box<MODE, TIn, 2, 2, 1>(stage + L::row_off(2), Af, n, tid);
        widen_box<MODE, TIn, 3, 3, 1>(stage + L::row_off(3), Af, n, tid);
    } else {
        widen_box<MODE, TIn, 1, 0, 1>(stage + L::row_off(1), Af, n, tid);
        widen_box<MODE, TIn, 2, 0, 2>(stage + L::row_off(2), Af, n, tid);
        widen_box<MODE, TIn, 3, 0, 3>(stage + L::row_off(3), Af, n, tid);
    }
}

// FP32 input used in place: zero the rows at or past n of a partial chunk.
template <int MODE>
__device__ __forceinline__ void zero_rows(unsigned char *stage, int n, int tid) {
    using L = Layout<MODE, float>;
#pragma unroll
    for (int r = L::R0; r < 4; ++r) {
        const int w4 = L::width(r) / 4;                       // float4 per row
        float4 *base = reinterpret_cast<float4 *>(stage + L::row_off(r));
        for (int e = tid; e < 16 * w4; e += NTHREADS) {
            const int i = e / w4;
            if (16 * r + i >= n) base[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// ------------------------------------------------------ diagonal inverse
// Unit-lower-triangular 16x16 inverse by forward substitution, one lane per
// column j: x[i] = sum_{k<i} (-a[i][k]) x[k] for i > j, x[j] = 1, x[i<j] = 0.
// Only entries of `a` (pitch ap) with k < i are used.
__device__ __forceinline__ void diag_invert(const float *a, int ap, int j, float (&x)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
        float s = 0.f;
#pragma unroll
        for (int kq = 0; kq < (i + 3) / 4; ++kq) {
            const float4 v = *reinterpret_cast<const float4 *>(a + i * ap + 4 * kq);
            if (4 * kq + 0 < i) s = fmaf(-v.x, x[4 * kq + 0], s);
            if (4 * kq + 1 < i) s = fmaf(-v.y, x[4 * kq + 1], s);
            if (4 * kq + 2 < i) s = fmaf(-v.z, x[4 * kq + 2], s);
            if (4 * kq + 3 < i) s = fmaf(-v.w, x[4 * kq + 3], s);
        }
        x[i] = (i > j) ? s : x[i];
    }
}

// ----------------------------------------------------------- 16x16 products
// A unit computes a 16x16 tile; lane l (0..15): rg = l >> 2, cg = l & 3.
// acc[m][n] is row rg + 4m, column 4cg + n.

__device__ __forceinline__ float comp(const float4 &v, int kk) {
    return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
}

// TRI_NEG = false: acc += P Q.  TRI_NEG = true: acc -= P Q with P lower
// triangular, so k-quad q only meets rows m >= q (the negation is folded into
// the FMA operand).  P row-major with pitch XP, Q row-major with pitch qp.
template <bool TRI_NEG>
__device__ __forceinline__ void prod(float (&acc)[4][4], const float *__restrict__ P,
                                     const float *__restrict__ Q, int qp, int rg, int cg) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float4 pr[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (!TRI_NEG || m >= q) pr[m] = *reinterpret_cast<const float4 *>(P + (rg + 4 * m) * XP + 4 * q);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float4 qv = *reinterpret_cast<const float4 *>(Q + (4 * q + kk) * qp + 4 * cg);
            const float2 q01 = make_float2(qv.x, qv.y), q23 = make_float2(qv.z, qv.w);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (TRI_NEG && m < q) continue;
                const float a = TRI_NEG ? -comp(pr[m], kk) : comp(pr[m], kk);
                const float2 aa = make_float2(a, a);
                // two FMAs per instruction; each component rounds exactly like fmaf
                float2 c01 = __ffma2_rn(aa, q01, make_float2(acc[m][0], acc[m][1]));
                float2 c23 = __ffma2_rn(aa, q23, make_float2(acc[m][2], acc[m][3]));
                acc[m][0] = c01.x; acc[m][1] = c01.y;
                acc[m][2] = c23.x; acc[m][3] = c23.y;
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

// (+/-) tile -> row-major X/U block
template <bool NEG>
__device__ __forceinline__ void put_smem(float *dst, const float (&acc)[4][4], int rg, int cg) {
    const float s = NEG ? -1.f : 1.f;
#pragma unroll
    for (int m = 0; m < 4; ++m)
        *reinterpret_cast<float4 *>(dst + (rg + 4 * m) * XP + 4 * cg) =
            make_float4(s * acc[m][0], s * acc[m][1], s * acc[m][2], s * acc[m][3]);
}

// tile -> output block (bi, bj) of the chunk, rows below n only.  `ob` points
// at the chunk-head's first output row, `os` is the row stride (H * 64).
template <typename TOut>
__device__ __forceinline__ void put_out(TOut *ob, int os, int n, int bi, int bj, const float (&acc)[4][4],
                                        int rg, int cg) {
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
        const int r = 16 * bi + rg + 4 * mm;
        if (r < n) put4(ob + (r * os + 16 * bj + 4 * cg), acc[mm][0], acc[mm][1], acc[mm][2], acc[mm][3]);
    }
}

// The zero blocks above the diagonal (columns 16(br+1) .. 63 of rows in block-row br).
template <typename TOut>
__device__ __forceinline__ void store_upper_zeros(TOut *ob, int os, int n, int tid) {
    constexpr int VEC = 16 / int(sizeof(TOut));     // elements per 16-byte store
    constexpr int PB = 16 / VEC;                    // 16-byte stores per 16-column block
#pragma unroll
    for (int br = 0; br < 3; ++br) {
        const int per_row = PB * (3 - br);
        const int cnt = 16 * per_row;
#pragma unroll
        for (int e0 = 0; e0 < cnt; e0 += NTHREADS) {
            const int e = e0 + tid;
            if (e < cnt) {
                const int r = 16 * br + e / per_row;
                const int c = 16 * (br + 1) + VEC * (e % per_row);
                if (r < n) *reinterpret_cast<uint4 *>(ob + (r * os + c)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
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
    float *Xs = reinterpret_cast<float *>(smem + L::OFF_X);
    float *U = reinterpret_cast<float *>(smem + L::OFF_U);
    TOut *out = reinterpret_cast<TOut *>(p.out);
    const int tid = threadIdx.x;
    const int unit = tid >> 4, warp = tid >> 5, half = unit & 1;
    const int l = tid & 15, rg = l >> 2, cg = l & 3;
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
            // A copy never completed.  Record it, give the copies still in
            // flight a bounded chance to land, and stop.
            if (tid == 0) {
                atomicOr(p.err, ERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bars[st], parity);
                for (int s = 1; s < STAGES; ++s)
                    mbar_wait_bounded(&bars[(st + s) % STAGES], ((it + s) / STAGES) & 1);
            }
            return;
        }
        const Meta m = metas[st];
        if (!m.valid) break;
        unsigned char *stage = smem + L::OFF_STAGE + st * L::STAGE_BYTES;
        const int32_t q = int32_t(blockIdx.x) + it * G;
        const int32_t q_next = q + STAGES * G;
        const int os = p.H * BT;                                  // output row stride
        TOut *ob = out + (int64_t(m.row0) * p.H + m.h) * BT;      // chunk-head's first row

        if (MODE != MODE_MERGE) store_upper_zeros(ob, os, m.n, tid);

        // A operands: widened copy (16-bit input) or the landing buffer itself
        if (L::WIDEN) {
            widen_all<MODE, TIn>(stage, Af, m.n, tid);
        } else if (m.n < BT) {
            zero_rows<MODE>(stage, m.n, tid);
        }
        if (MODE == MODE_MERGE) {
            // workspace tile (4 row-major 16x16 FP32 inverses) -> X slots 0..3
            const float *wt = reinterpret_cast<const float *>(stage + L::WS_OFF);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int e = tid + NTHREADS * v;
                const int u = e >> 6, i = (e >> 2) & 15, k4 = e & 3;
                *reinterpret_cast<float4 *>(Xs + u * XBS + i * XP + 4 * k4) =
                    *reinterpret_cast<const float4 *>(wt + u * 256 + i * 16 + 4 * k4);
            }
        }
        // TMA data is visible to every thread after its own mbarrier wait; a
        // barrier is needed only when threads rewrote shared memory above.
        if (L::WIDEN || MODE == MODE_MERGE || m.n < BT) __syncthreads();
        if (L::WIDEN && tid == 0) {          // the landing buffer is no longer read
            fence_proxy_async();
            issue<MODE, TIn>(p, maps.m, q_next, walk, smem, st);
        }

        if (MODE != MODE_MERGE) {
            float x[16];
            const int b = diag_of_unit(unit);
            const AView a = aview<MODE, TIn>(stage, Af, b, b);
            diag_invert(a.p, a.pitch, l, x);
            // diagonal block of the output, one lane per column
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = 16 * b + i;
                if (r < m.n) put1(ob + (r * os + 16 * b + l), x[i]);
            }
            if (MODE == MODE_DIAG) {
                float *w = p.ws + size_t(q) * 1024 + b * 256 + l;
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i * 16] = x[i];
                if (!L::WIDEN) {
                    __syncthreads();
                    if (tid == 0) {
                        fence_proxy_async();
                        issue<MODE, TIn>(p, maps.m, q_next, walk, smem, st);
                    }
                }
                continue;
            }
            float *xs = Xs + b * XBS;
#pragma unroll
            for (int i = 0; i < 16; ++i) xs[i * XP + l] = x[i];
            __syncwarp();                    // step 0 reads only this warp's inverses
        }

        // ---- merge: four steps; U slots hold U' = -U
        //   step 0  warp 0: U_A' = -X11 A10, U_B' = -X33 A32     warp 1: U00' = -X22 A20, U01' = -X22 A21
        //   step 1  warp 0: X10 = U_A' X00, X32 = U_B' X22       warp 1: U10p' = -X33 A30, U11p' = -X33 A31
        //   step 2  warp 0: X21 = U01' X11, X20p = U00' X00      warp 1: U10' = U10p' + (-X32) A20, U11' likewise
        //   step 3  warp 0: X31 = U11' X11, X20 = X20p + U01' X10
        //           warp 1: T = U10' X00 (unit 2), X30 = U11' X10 + T (unit 3)
        float acc[4][4];
        zero(acc);
#pragma unroll 1
        for (int step = 0; step < 4; ++step) {
            const float *P;
            const float *Q;
            int qp = XP;
            bool tri = false;
            if (step == 0) {
                tri = true;
                if (warp == 0) {
                    P = Xs + (half ? 3 : 1) * XBS;
                    const AView a = aview<MODE, TIn>(stage, Af, half ? 3 : 1, half ? 2 : 0);
                    Q = a.p; qp = a.pitch;
                } else {
                    P = Xs + 2 * XBS;
                    const AView a = aview<MODE, TIn>(stage, Af, 2, half);
                    Q = a.p; qp = a.pitch;
                }
            } else if (step == 1) {
                if (warp == 0) {
                    P = U + half * XBS;
                    Q = Xs + (half ? 2 : 0) * XBS;
                } else {
                    tri = true;
                    P = Xs + 3 * XBS;
                    const AView a = aview<MODE, TIn>(stage, Af, 3, half);
                    Q = a.p; qp = a.pitch;
                }
            } else if (step == 2) {
                if (warp == 0) {
                    P = U + (half ? 2 : 3) * XBS;                 // U00' : U01'
                    Q = Xs + (half ? 0 : 1) * XBS;                // X00  : X11
                } else {
                    P = Xs + XS_32N * XBS;
                    const AView a = aview<MODE, TIn>(stage, Af, 2, half);
                    Q = a.p; qp = a.pitch;
                }
            } else {
                if (warp == 0) {
                    P = U + (half ? 3 : 1) * XBS;                 // U01' : U11'
                    Q = Xs + (half ? XS_10 : 1) * XBS;            // X10  : X11
                } else {
                    P = U + (half ? 1 : 0) * XBS;                 // U11' : U10'
                    Q = Xs + (half ? XS_10 : 0) * XBS;            // X10  : X00
                }
            }
            if (tri) prod<true>(acc, P, Q, qp, rg, cg);
            else prod<false>(acc, P, Q, qp, rg, cg);

            if (step == 0) {
                put_smem<false>(U + (warp == 0 ? half : 2 + half) * XBS, acc, rg, cg);
                zero(acc);
                __syncthreads();
            } else if (step == 1) {
                if (warp == 0) {             // X10 (half 0) / X32 (half 1)
                    if (half) put_smem<true>(Xs + XS_32N * XBS, acc, rg, cg);
                    else put_smem<false>(Xs + XS_10 * XBS, acc, rg, cg);
                    put_out(ob, os, m.n, half ? 3 : 1, half ? 2 : 0, acc, rg, cg);
                    zero(acc);
                }
                __syncthreads();
            } else if (step == 2) {
                if (warp == 0) {
                    if (!half) {             // X21 done; half 1 keeps X20p
                        put_out(ob, os, m.n, 2, 1, acc, rg, cg);
                        zero(acc);
                    }
                } else {                     // U10' / U11'
                    put_smem<false>(U + half * XBS, acc, rg, cg);
                    zero(acc);
                }
                __syncthreads();
                if (!L::WIDEN && tid == 0) { // A is no longer read
                    fence_proxy_async();
                    issue<MODE, TIn>(p, maps.m, q_next, walk, smem, st);
                }
            } else {
                if (warp == 0) {             // X31 (half 0) / X20 (half 1)
                    put_out(ob, os, m.n, half ? 2 : 3, half ? 0 : 1, acc, rg, cg);
                } else {
                    if (!half) put_smem<false>(U + 2 * XBS, acc, rg, cg);   // T
                    __syncwarp();
                    if (half) {              // X30 = U11' X10 + T
                        const float *t = U + 2 * XBS;
#pragma unroll
                        for (int mm = 0; mm < 4; ++mm) {
                            const float4 v = *reinterpret_cast<const float4 *>(t + (rg + 4 * mm) * XP + 4 * cg);
                            acc[mm][0] += v.x; acc[mm][1] += v.y; acc[mm][2] += v.z; acc[mm][3] += v.w;
                        }
                        put_out(ob, os, m.n, 3, 0, acc, rg, cg);
                    }
                }
            }
        }
    }
}

}  // namespace kda
