// kda_kgb.cuh -- KDA's chunk matrix built from keys, betas and decays, fused
// with the 64-token solve: A never leaves shared memory.
//
// LightLLM PR #1703 (PR description) has KDA prefill use the shared solver;
// the matrix it inverts is KDA's intra-chunk matrix
//     A[i][j] = beta_i sum_d k_id k_jd exp(g_id - g_jd),   j < i,
// with g the per-channel cumulative log decay.  Per chunk-head this kernel
// builds the ten lower 16x16 blocks of A and solves (I + A)^-1 with the
// 64-token kernel's schedule.
//
// Construction.  Block I of the chunk has first row rI = 16 I and last live
// row eI = min(16 I + 15, n - 1).  For block (I, J), I >= J:
//     A_IJ = (Q_I * f_IJ) P_J^T,  Q_I[i][d] = k_id exp(g_id - g_rI,d),
//     P_J[j][d] = k_jd exp(g_eJ,d - g_jd),  f_IJ[d] = exp(g_rI,d - g_eJ,d).
// g is non-increasing along the chunk (a cumulative log decay), so every
// exponent of Q and P is <= 0, and so is f's for I > J: none of these factors
// can overflow, and one that underflows stands for a term below FP32's range.
// Only the diagonal factor f_II = exp(span) with span = g_rI - g_eI >= 0
// grows: channels whose span exceeds KGB_SAFE_SPAN get f_II = 0, and their
// terms k_id k_jd exp(g_id - g_jd) are added to the diagonal block one by one
// (a slow path that KDA's ordinary decays, about 1 nat per token, never take).
// The products run on the tensor cores in split TF32 (mma.sync m16n8k8, hi/lo
// parts, FP32 accumulation).
//
// Work split (one persistent CTA of 128 threads per resident slot, one
// chunk-head at a time):
//   * warp w streams channels 32w .. 32w+31 of the chunk's k and g rows into
//     shared memory with cp.async and turns them into Q and P in place (one
//     lane per channel; rows past a partial chunk's end become zeros);
//   * each warp computes two or three of the ten blocks over all channels
//     and writes them, times beta and masked to the strict lower part of the
//     chunk's valid rows, into an FP32 A tile;
//   * warps 0 and 1 solve the tile exactly like the 64-token kernel (diagonal
//     forward substitution, two merge levels on the tensor cores) while the
//     next chunk-head's rows are in flight and warps 2 and 3 start on them.
#pragma once

#include "kda_kernels.cuh"
#include "kda_small.cuh"

namespace kda {

// factor rows per slice: the six block pairs I > J, then the four diagonal blocks
constexpr int KGB_FROWS = 10;
// largest decay (nats) over a diagonal block that its tensor-core product takes,
// in log2 units; steeper channels go through the slow path
constexpr float KGB_SAFE_SPAN2 = 32.0f * 1.4426950408889634f;

struct KgbParams {
    const void *k;             // [rows, H, K], input dtype
    const float *g;            // [rows, H, K]
    const void *beta;          // [rows, H], input dtype
    void *out;                 // [rows, H, 64], output dtype
    const int32_t *cu;         // packed: cu_seqlens (device); dense: nullptr
    int32_t nseq;
    int32_t H;
    int64_t T;                 // dense: rows per batch row; packed: total rows
    int32_t cpr;               // dense: chunks per batch row
    int32_t n_tasks;           // loop bound on chunk-head indices
    int32_t K;                 // channels: 32, 64, 96 or 128
};

constexpr int KGB_THREADS = 128;
// slice row pitch (floats): the paired 8-byte fragment loads at 8 g + 2 t hit 32
// distinct banks per half-warp
constexpr int KGB_SP = 40;
constexpr int KGB_SLICE = 64 * KGB_SP;         // floats per slice buffer
constexpr int KGB_FLOATS = 2 * 4 * KGB_SLICE   // Q and P slices
                         + 4 * KGB_FROWS * 32  // f_IJ per slice, block pair and diagonal block
                         + 10 * 256            // A blocks, pitch 16
                         + 4 * XTS + 4 * XRS   // inverse tiles of the merge
                         + 64                  // beta of the chunk's rows
                         + 16;                 // steep-channel masks [slice][diagonal block]
constexpr int KGB_BYTES = KGB_FLOATS * 4;

__device__ __forceinline__ void named_sync64() { asm volatile("bar.sync 1, 64;" ::: "memory"); }

// Chunk-heads q = q0, q0 + step, ... of one CTA (every thread walks the same sequence).
struct KgbWalk {
    int32_t q, c, h, step, sc, sh;
    Walk w;
    __device__ __forceinline__ KgbWalk(const KgbParams &p, int32_t q0, int32_t step_)
        : q(q0), step(step_), w{0, 0} {
        c = q0 / p.H;
        h = q0 - c * p.H;
        sc = step_ / p.H;
        sh = step_ - sc * p.H;
    }
    __device__ __forceinline__ Meta next(const KgbParams &p) {
        const Meta m = q < p.n_tasks ? locate<BT>(p, c, h, w) : Meta{0, 0, 0, 0};
        q += step;
        c += sc;
        h += sh;
        if (h >= p.H) {
            h -= p.H;
            ++c;
        }
        return m;
    }
};

// Channels 32 s .. 32 s + 31 of the chunk-head's k and g rows into the slice
// buffers (row pitch KGB_SP floats; 16-bit keys land at the start of each row).
template <typename TIn>
__device__ __forceinline__ void kgb_issue(const KgbParams &p, const Meta &m, int s, float *kb, float *gb, int lane) {
    if (!m.valid) return;
    constexpr int VEC = Elt<TIn>::VEC;
    constexpr int CK = 32 / VEC;                       // 16-byte copies per key row
    const int64_t rs = int64_t(p.H) * p.K;             // row stride (elements)
    const int64_t base = int64_t(m.row0) * rs + int64_t(m.h) * p.K + 32 * s;
    const TIn *ks = reinterpret_cast<const TIn *>(p.k) + base;
    const float *gs = p.g + base;
#pragma unroll 4
    for (int e = lane; e < 64 * CK; e += 32) {
        const int i = e / CK, c = e % CK;
        const bool live = i < m.n;
        cp_async16(reinterpret_cast<unsigned char *>(kb + i * KGB_SP) + 16 * c, live ? ks + i * rs + c * VEC : p.k,
                   live ? 16u : 0u);
    }
#pragma unroll 4
    for (int e = lane; e < 64 * 8; e += 32) {
        const int i = e >> 3, c = e & 7;
        const bool live = i < m.n;
        cp_async16(gb + i * KGB_SP + 4 * c, live ? gs + i * rs + 4 * c : p.g, live ? 16u : 0u);
    }
}

// Lane d of the slice's warp: the block-pair factors of channel d, then Q and
// P of channel d in place (column d of the slice is touched by this lane only).
// 2^x on the SFU (PTX ex2.approx.ftz.f32; relative error about 2^-22)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename TIn>
__device__ __forceinline__ void kgb_transform(float *kb, float *gb, float *fac, unsigned *steep, int n, int d) {
    // exponents are differences of g taken first (exact for nearby values), then
    // scaled to base 2, so their error does not grow with |g|
    constexpr float LOG2E = 1.4426950408889634f;
    float gr[4], ge[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int e = 16 * b + 15 < n ? 16 * b + 15 : n - 1;
        gr[b] = gb[16 * b * KGB_SP + d];
        ge[b] = gb[(e > 0 ? e : 0) * KGB_SP + d];
    }
    // f_IJ = exp(g_rI - g_eJ), I > J (zero when block I starts past the chunk's end)
#pragma unroll
    for (int I = 1; I < 4; ++I)
#pragma unroll
        for (int J = 0; J < I; ++J)
            fac[(I * (I - 1) / 2 + J) * 32 + d] = 16 * I < n ? ex2((gr[I] - ge[J]) * LOG2E) : 0.f;
    // f_II = exp(g_rI - g_eI), zero for a channel that falls further than the
    // safe span over the block (its terms take the slow path)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const float span = (gr[b] - ge[b]) * LOG2E;
        const bool live = 16 * b < n, st = live && !(span <= KGB_SAFE_SPAN2);
        fac[(6 + b) * 32 + d] = live && !st ? ex2(span) : 0.f;
        const unsigned m = __ballot_sync(0xffffffffu, st);
        if (d == 0) steep[b] = m;
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float kv[16];
        if constexpr (sizeof(TIn) == 4) {
#pragma unroll
            for (int i = 0; i < 16; ++i) kv[i] = kb[(16 * b + i) * KGB_SP + d];
        } else {                                       // raw 16-bit keys at the start of each row
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                kv[i] = float(reinterpret_cast<const TIn *>(kb + (16 * b + i) * KGB_SP)[d]);
            }
            __syncwarp();                              // every lane has read the raw row before it is widened
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * b + i;
            const bool live = r < n;
            const float gv = gb[r * KGB_SP + d];
            kb[r * KGB_SP + d] = live ? kv[i] * ex2((gv - gr[b]) * LOG2E) : 0.f;    // Q
            gb[r * KGB_SP + d] = live ? kv[i] * ex2((ge[b] - gv) * LOG2E) : 0.f;    // P
        }
    }
}

// Slow path of diagonal block I: the terms of the channels in the steep masks,
// k_id k_jd exp(g_id - g_jd) one by one, read again from global memory, added to
// the lane's C fragments (rows g, g + 8; columns 8 nt + 2 t + e).
template <typename TIn>
__device__ __forceinline__ void kgb_steep_terms(const KgbParams &p, const Meta &m, const unsigned *steep, int I,
                                             int nsl, int g, int t, TileC &c) {
    constexpr float LOG2E = 1.4426950408889634f;
    const int64_t rs = int64_t(p.H) * p.K;
    const int64_t base = (int64_t(m.row0) + 16 * I) * rs + int64_t(m.h) * p.K;
    const TIn *kp = reinterpret_cast<const TIn *>(p.k) + base;
    const float *gp = p.g + base;
    const int li[2] = {g, g + 8};
    const int lj[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
    for (int s = 0; s < nsl; ++s) {
        unsigned mask = steep[s * 4 + I];
        while (mask != 0u) {
            const int d = 32 * s + __ffs(mask) - 1;
            mask &= mask - 1u;
            float ki[2], gi[2], kj[4], gj[4];
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                const bool live = 16 * I + li[a] < m.n;
                ki[a] = live ? float(kp[li[a] * rs + d]) : 0.f;
                gi[a] = live ? gp[li[a] * rs + d] : 0.f;
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const bool live = 16 * I + lj[a] < m.n;
                kj[a] = live ? float(kp[lj[a] * rs + d]) : 0.f;
                gj[a] = live ? gp[lj[a] * rs + d] : 0.f;
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int a = 2 * nt + e;
                        if (lj[a] < li[h])      // strictly lower; dead rows hold k = 0
                            c.c[nt][2 * h + e] = fmaf(ki[h] * kj[a], ex2((gi[h] - gj[a]) * LOG2E), c.c[nt][2 * h + e]);
                    }
        }
    }
}

// Block (I, J) of A over all nsl slices, times beta, masked, into Ab (pitch 16).
template <typename TIn>
__device__ __forceinline__ void kgb_block(const KgbParams &p, const Meta &m, const float *kq, const float *gp,
                                          const float *fac, const unsigned *steep, const float *bs, float *Ab,
                                          int I, int J, int nsl, int g, int t) {
    const int n = m.n;
    TileC c;
    zero(c);
    const int pr = I > J ? I * (I - 1) / 2 + J : 6 + I;
    for (int s = 0; s < nsl; ++s) {
        const float *q0 = kq + s * KGB_SLICE + (16 * I + g) * KGB_SP;
        const float *q1 = q0 + 8 * KGB_SP;
        const float *pb = gp + s * KGB_SLICE + (16 * J + g) * KGB_SP;
        const float *fs = fac + (s * KGB_FROWS + pr) * 32;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            // k-slots t and t + 4 of this k-step stand for channels 8 ks + 2t and 8 ks + 2t + 1
            const int d0 = 8 * ks + 2 * t;
            const float2 f = *reinterpret_cast<const float2 *>(fs + d0);
            const float2 x0 = *reinterpret_cast<const float2 *>(q0 + d0);
            const float2 x1 = *reinterpret_cast<const float2 *>(q1 + d0);
            uint32_t ah[4], al[4];
            split_tf32(x0.x * f.x, ah[0], al[0]);
            split_tf32(x1.x * f.x, ah[1], al[1]);
            split_tf32(x0.y * f.y, ah[2], al[2]);
            split_tf32(x1.y * f.y, ah[3], al[3]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float *pj = pb + 8 * nt * KGB_SP;
                uint32_t bh0, bl0, bh1, bl1;
                const float2 y = *reinterpret_cast<const float2 *>(pj + d0);
                split_tf32(y.x, bh0, bl0);
                split_tf32(y.y, bh1, bl1);
                mma8(c.c[nt], al, bh0, bh1);
                mma8(c.c[nt], ah, bl0, bl1);
                mma8(c.c[nt], ah, bh0, bh1);
            }
        }
    }
    if (I == J) {
        unsigned any = 0u;
        for (int s = 0; s < nsl; ++s) any |= steep[s * 4 + I];
        if (any != 0u) kgb_steep_terms<TIn>(p, m, steep, I, nsl, g, t, c);
    }
    // C fragments: c[nt][2 h + e] = block row g + 8 h, block column 8 nt + 2 t + e
    float *Ad = Ab + blk(I, J) * 256;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = g + 8 * h, r = 16 * I + i, j = 8 * nt + 2 * t;
            const float b = bs[r];
            const bool live = r < n;
            float v0 = c.c[nt][2 * h], v1 = c.c[nt][2 * h + 1];
            if (I == J) {
                v0 = j < i ? v0 : 0.f;
                v1 = j + 1 < i ? v1 : 0.f;
            }
            *reinterpret_cast<float2 *>(Ad + i * 16 + j) = live ? make_float2(b * v0, b * v1) : make_float2(0.f, 0.f);
        }
}

// Solve of the A tile by threads 0..63 (the 64-token kernel's schedule on an
// FP32 tile with blocks (i, j) at Ab + 256 blk(i, j), pitch 16).
template <typename TOut>
__device__ __forceinline__ void kgb_solve(const float *Ab, float *Xt, float *Xr, TOut *ob, int os, int n, int tid) {
    const int unit = tid >> 4, warp = tid >> 5, l = tid & 15;
    const int lane = tid & 31, g = lane >> 2, t = lane & 3;
    {
        float x[16];
        const int b = unit;
        diag_invert(Ab + blk(b, b) * 256, 16, l, x);
        TOut *op = ob + (16 * b * os + 16 * b + l);    // diagonal block, lane = column
        if (n == BT) {
#pragma unroll
            for (int i = 0; i < 16; ++i, op += os) put1(op, x[i]);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i, op += os)
                if (16 * b + i < n) put1(op, x[i]);
        }
        if (b != 3) {                                  // X_bb^T row-major (row = lane)
            float4 *d = reinterpret_cast<float4 *>(Xt + (b == 0 ? XT_00 : b == 1 ? XT_11 : XT_22) * XTS + l * XTP);
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        }
        if (b != 0) {                                  // -X_bb row-major (column = lane)
            float *d = Xr + (b == 1 ? XR_11 : b == 3 ? XR_33 : XR_22) * XRS + l;
#pragma unroll
            for (int i = 0; i < 16; ++i) d[i * XRP] = -x[i];
        }
        __syncwarp();
    }
    {   // level A (warp 0: X10, warp 1: X32), transposed
        TileA la;
        TileB rb;
        TileC c1, c2;
        left_smem(la, Xt + (warp == 0 ? XT_00 : XT_22) * XTS, XTP, g, t);
        right4<false>(rb, Ab + (warp == 0 ? blk(1, 0) : blk(3, 2)) * 256, 16, g, t);
        zero(c1);
        mma_tile<false>(c1, la, rb);
        left_regs(la, c1);
        right2(rb, Xr + (warp == 0 ? XR_11 : XR_33) * XRS, XRP, g, t);
        zero(c2);
        mma_tile<false>(c2, la, rb);
        if (warp == 0) {
            smem_tile_t(Xt + XT_10 * XTS, c2, g, t);
            out_tile_t(ob, os, n, 1, 0, c2, g, t);
        } else {
            smem_tile_neg(Xr + XR_32 * XRS, c2, g, t);
            out_tile_t(ob, os, n, 3, 2, c2, g, t);
        }
    }
    named_sync64();
    {   // level B, warp w = column block w of X_BL
        TileA la, lb;
        TileB rb;
        TileC ct2, ct3, cx;
        zero(ct2);
        zero(ct3);
        left_smem(la, Xt + (warp == 0 ? XT_00 : XT_11) * XTS, XTP, g, t);
        right4<false>(rb, Ab + blk(2, warp) * 256, 16, g, t);
        mma_tile<false>(ct2, la, rb);
        right4<false>(rb, Ab + blk(3, warp) * 256, 16, g, t);
        mma_tile<false>(ct3, la, rb);
        if (warp == 0) {                               // + X10^T A21^T, X10^T A31^T
            left_smem(la, Xt + XT_10 * XTS, XTP, g, t);
            right4<false>(rb, Ab + blk(2, 1) * 256, 16, g, t);
            mma_tile<false>(ct2, la, rb);
            right4<false>(rb, Ab + blk(3, 1) * 256, 16, g, t);
            mma_tile<false>(ct3, la, rb);
        }
        left_regs(la, ct2);
        left_regs(lb, ct3);
        right2(rb, Xr + XR_22 * XRS, XRP, g, t);
        zero(cx);
        mma_tile<false>(cx, la, rb);
        out_tile_t(ob, os, n, 2, warp, cx, g, t);
        right2(rb, Xr + XR_32 * XRS, XRP, g, t);
        zero(cx);
        mma_tile<false>(cx, la, rb);
        right2(rb, Xr + XR_33 * XRS, XRP, g, t);
        mma_tile<false>(cx, lb, rb);
        out_tile_t(ob, os, n, 3, warp, cx, g, t);
    }
    store_upper_zeros(ob, os, n, tid);
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(KGB_THREADS, 2)
kda_kgb_kernel(const KgbParams p) {
    extern __shared__ __align__(128) float sm[];
    float *kq = sm;                                    // Q slices
    float *gp = kq + 4 * KGB_SLICE;                    // P slices
    float *fac = gp + 4 * KGB_SLICE;
    float *Ab = fac + 4 * KGB_FROWS * 32;
    float *Xt = Ab + 10 * 256;
    float *Xr = Xt + 4 * XTS;
    float *bs = Xr + 4 * XRS;
    unsigned *steep = reinterpret_cast<unsigned *>(bs + 64);     // [slice][diagonal block]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nsl = p.K / 32;
    const bool has_slice = warp < nsl;
    const int os = p.H * BT;
    float *kb = kq + warp * KGB_SLICE, *gb = gp + warp * KGB_SLICE;
    KgbWalk walk(p, blockIdx.x, gridDim.x);
    Meta cur = walk.next(p);
    if (has_slice) kgb_issue<TIn>(p, cur, warp, kb, gb, lane);
    cp_async_commit();
    for (;;) {
        if (!cur.valid) {                              // the same for every thread of the CTA
            cp_async_wait<0>();
            break;
        }
        float b0 = 0.f, b1 = 0.f;                      // beta of the chunk's rows (warp 0)
        if (warp == 0) {
            const TIn *bp = reinterpret_cast<const TIn *>(p.beta) + (int64_t(cur.row0) * p.H + cur.h);
            if (lane < cur.n) b0 = float(bp[int64_t(lane) * p.H]);
            if (lane + 32 < cur.n) b1 = float(bp[int64_t(lane + 32) * p.H]);
        }
        cp_async_wait<0>();
        __syncwarp();
        if (has_slice) kgb_transform<TIn>(kb, gb, fac + warp * KGB_FROWS * 32, steep + 4 * warp, cur.n, lane);
        if (warp == 0) {
            bs[lane] = b0;
            bs[lane + 32] = b1;
        }
        __syncthreads();                               // Q, P, factors, beta ready; the last solve is done
        // blocks blk = warp, warp + 4, warp + 8: (0,0) (2,1) (3,2) | (1,0) (2,2) (3,3) | (1,1) (3,0) | (2,0) (3,1)
#pragma unroll 1
        for (int b = warp; b < 10; b += 4) {
            const int I = b >= 6 ? 3 : b >= 3 ? 2 : b >= 1 ? 1 : 0;
            const int J = b - I * (I + 1) / 2;
            kgb_block<TIn>(p, cur, kq, gp, fac, steep, bs, Ab, I, J, nsl, g, t);
        }
        __syncthreads();                               // A complete; the slice buffers are free
        const Meta nxt = walk.next(p);
        if (has_slice) kgb_issue<TIn>(p, nxt, warp, kb, gb, lane);
        cp_async_commit();
        if (warp < 2) {
            TOut *ob = reinterpret_cast<TOut *>(p.out) + (int64_t(cur.row0) * p.H + cur.h) * BT;
            kgb_solve<TOut>(Ab, Xt, Xr, ob, os, cur.n, tid);
        }
        cur = nxt;
    }
}

}  // namespace kda
