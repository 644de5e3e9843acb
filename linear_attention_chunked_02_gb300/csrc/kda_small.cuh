// kda_small.cuh -- the 32- and 16-token branches of the chunk solver.
//
// LightLLM PR #1703 (PR description) presents the path it optimises as the
// shared solver's branch for 64-token chunks; the same inversion of (I + A) for the strictly
// lower-triangular chunk matrix A is solved here for chunks of 16 and 32
// tokens, with the same building blocks as the 64-token kernel:
//   * 16 tokens: one 16-lane unit per chunk-head, forward substitution with one
//     lane per column (FP32 FMA);
//   * 32 tokens: one warp per chunk-head; its two units invert the diagonal
//     16x16 blocks, then X10 = -X11 A10 X00 runs on the tensor cores in split
//     TF32, computed transposed as in the 64-token kernel's level A.
// Persistent CTAs of 64 threads walk chunk-heads q = slot, slot + slots, ...
// with one slot per unit (16 tokens) or per warp (32 tokens).  Tiles are small
// (0.5-3 KiB), so each slot streams its own tiles through a SMALL_STAGES-deep ring in
// shared memory with cp.async: 16-byte copies, zero-fill for rows past a
// partial chunk's end (never read), nothing for chunk-heads past the last one.
// The next SMALL_STAGES - 1 chunk-heads are in flight while one is computed.  The
// ring holds the input bytes as they are; with 16-bit input the diagonal
// blocks are widened once into an FP32 tile (every lane converts its share)
// and the off-diagonal block is widened in registers by the MMA operand load.
// Waits are cp.async.wait_group on the thread's own copies: no spin loop.
#pragma once

#include "kda_kernels.cuh"

namespace kda {

struct SmallParams {
    const void *A;             // [rows, H, CBT], input dtype
    void *out;                 // [rows, H, CBT], output dtype
    const int32_t *cu;         // packed: cu_seqlens (device); dense: nullptr
    int32_t nseq;
    int32_t H;
    int64_t T;                 // dense: rows per batch row; packed: total rows
    int32_t cpr;               // dense: chunks per batch row
    int32_t n_tasks;           // loop bound on chunk-head indices
};

// cp.async ring depth per slot: one chunk-head in flight while one is computed
// (GB300: 2 and 3 stages time the same within 2 %; 2 leaves more registers)
constexpr int SMALL_STAGES = 2;

// Chunk-heads q = q0, q0 + step, ... of one slot; chunk c = q / H and head
// h = q % H are advanced incrementally (one division at the start).
template <int CBT>
struct SlotWalk {
    int32_t q, c, h, step, sc, sh;
    Walk w;
    __device__ __forceinline__ SlotWalk(const SmallParams &p, int32_t q0, int32_t step_)
        : q(q0), step(step_), w{0, 0} {
        c = q0 / p.H;
        h = q0 - c * p.H;
        sc = step_ / p.H;
        sh = step_ - sc * p.H;
    }
    // meta of the current chunk-head, then advance to the next
    __device__ __forceinline__ Meta next(const SmallParams &p) {
        const Meta m = q < p.n_tasks ? locate<CBT>(p, c, h, w) : Meta{0, 0, 0, 0};
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

// cu_seqlens entries cached in shared memory by the short-chunk kernels
// (packed batches of up to 511 requests)
constexpr int SMALL_CU_CAP = 512;

// p with cu pointing to a shared-memory copy of cu_seqlens when it fits (every
// thread of the CTA calls this; it ends with a CTA barrier in that case).
__device__ __forceinline__ SmallParams with_cached_cu(const SmallParams &p, int32_t *cu_s, int tid) {
    SmallParams ps = p;
    if (p.cu != nullptr && p.nseq < SMALL_CU_CAP) {
        for (int i = tid; i <= p.nseq; i += NTHREADS) cu_s[i] = __ldg(p.cu + i);
        ps.cu = cu_s;
        __syncthreads();
    }
    return ps;
}

// 16-byte global -> shared copy; src_bytes = 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 16-bit input: `nblk` 16x16 blocks of the ring (at src + 256 * blk_of(b))
// widened into FP32 blocks dst[b] (pitch 16) by `lanes` lanes, each widening
// 8 elements per step, so every element is converted once.
template <typename TIn>
__device__ __forceinline__ void widen_blocks(const TIn *src, int b_hi, float *dst, int nblk, int lane, int lanes) {
    for (int e = lane; e < nblk * 32; e += lanes) {
        const int b = e >> 5, o = (e & 31) * 8;
        float f[8];
        Elt<TIn>::widen(*reinterpret_cast<const uint4 *>(src + (b ? b_hi : 0) * 256 + o), f);
        float4 *d = reinterpret_cast<float4 *>(dst + b * 256 + o);
        d[0] = make_float4(f[0], f[1], f[2], f[3]);
        d[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
}

// ------------------------------------------------------------ 16 tokens
// A group of 8 lanes solves one chunk-head; lane l owns columns 2l and 2l + 1,
// so every row of A it loads serves two forward substitutions.
constexpr int BT16_LANES = 8;
constexpr int BT16_SLOTS = NTHREADS / BT16_LANES;      // chunk-heads a CTA works on at once

// Ring stage of one slot: the 16x16 tile, row-major, pitch 16 elements.  Lane
// l copies 16 bytes of rows i0, i0 + DI, ... (i0 = l / PER_ROW).
template <typename TIn>
__device__ __forceinline__ void issue16(const SmallParams &p, const Meta &m, TIn *stage, int l) {
    constexpr int VEC = Elt<TIn>::VEC;
    constexpr int PER_ROW = 16 / VEC;                  // 16-byte copies per row
    constexpr int DI = BT16_LANES / PER_ROW;           // rows between a lane's copies
    if (!m.valid) return;
    const int rs = p.H * 16;                           // row stride (elements)
    const int i0 = l / PER_ROW, k = (l % PER_ROW) * VEC;
    const TIn *src = reinterpret_cast<const TIn *>(p.A) + (int64_t(m.row0) * rs + m.h * 16) + (i0 * rs + k);
    TIn *dst = stage + i0 * 16 + k;
#pragma unroll
    for (int it = 0; it < 16 / DI; ++it) {
        const bool live = i0 + DI * it < m.n;
        cp_async16(dst + DI * 16 * it, live ? src : p.A, live ? 16u : 0u);
        src += DI * rs;
    }
}

// Forward substitution for columns j and j + 1 of the 16x16 unit-lower inverse:
// the diag_invert recurrence, each row of `a` loaded once for both columns.
__device__ __forceinline__ void diag_invert2(const float *a, int ap, int j, float (&x)[16], float (&y)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = (i == j) ? 1.f : 0.f;
        y[i] = (i == j + 1) ? 1.f : 0.f;
    }
#pragma unroll
    for (int i = 1; i < 16; ++i) {
        float s = 0.f, u = 0.f;
#pragma unroll
        for (int kq = 0; kq < (i + 3) / 4; ++kq) {
            const float4 v = *reinterpret_cast<const float4 *>(a + i * ap + 4 * kq);
            if (4 * kq + 0 < i) { s = fmaf(-v.x, x[4 * kq + 0], s); u = fmaf(-v.x, y[4 * kq + 0], u); }
            if (4 * kq + 1 < i) { s = fmaf(-v.y, x[4 * kq + 1], s); u = fmaf(-v.y, y[4 * kq + 1], u); }
            if (4 * kq + 2 < i) { s = fmaf(-v.z, x[4 * kq + 2], s); u = fmaf(-v.z, y[4 * kq + 2], u); }
            if (4 * kq + 3 < i) { s = fmaf(-v.w, x[4 * kq + 3], s); u = fmaf(-v.w, y[4 * kq + 3], u); }
        }
        x[i] = (i > j) ? s : x[i];
        y[i] = (i > j + 1) ? u : y[i];
    }
}

// two consecutive output elements
__device__ __forceinline__ void put2(float *p, float a, float b) { *reinterpret_cast<float2 *>(p) = make_float2(a, b); }
template <typename TOut>
__device__ __forceinline__ void put2(TOut *p, float a, float b) {
    *reinterpret_cast<uint32_t *>(p) = pack2(a, b, (TOut *)nullptr);
}

// 16-token chunks: slot u of CTA b solves chunk-heads 8b + u, 8b + u + 8 grid, ...
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NTHREADS, 10)
kda_bt16_kernel(const SmallParams p) {
    constexpr int S = SMALL_STAGES;
    constexpr bool WIDEN = sizeof(TIn) == 2;
    __shared__ __align__(16) TIn ring[BT16_SLOTS][S][256];
    __shared__ __align__(16) float af[WIDEN ? BT16_SLOTS : 1][WIDEN ? 256 : 4];   // widened tile (16-bit input)
    __shared__ int32_t cu_s[SMALL_CU_CAP];
    const int tid = threadIdx.x, slot = tid / BT16_LANES, l = tid % BT16_LANES;
    const unsigned mask = 0xffu << (BT16_LANES * (slot & 3));
    const int32_t slots = gridDim.x * BT16_SLOTS;
    const int32_t q0 = blockIdx.x * BT16_SLOTS + slot;
    const int rs = p.H * 16;                 // row stride (elements); H * 16 * 16 < 2^31
    pdl_launch_dependents();
    pdl_wait();                              // the previous kernel's writes are visible
    const SmallParams ps = with_cached_cu(p, cu_s, tid);
    SlotWalk<16> walk(ps, q0, slots);
    // metas of the chunk-heads in the ring: m[0] is computed next
    Meta m[S];
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        m[s] = walk.next(ps);
        issue16<TIn>(p, m[s], ring[slot][s], l);
        cp_async_commit();
    }
    for (int k = 0;; ++k) {
        m[S - 1] = walk.next(ps);
        issue16<TIn>(p, m[S - 1], ring[slot][(k + S - 1) % S], l);
        cp_async_commit();
        if (!m[0].valid) {                 // later chunk-heads are past the end too (nothing issued)
            cp_async_wait<0>();
            break;
        }
        cp_async_wait<S - 1>();
        __syncwarp(mask);
        const float *a = reinterpret_cast<const float *>(ring[slot][k % S]);
        if constexpr (WIDEN) {
            widen_blocks(ring[slot][k % S], 0, af[slot], 1, l, BT16_LANES);
            __syncwarp(mask);
            a = af[slot];
        }
        float x[16], y[16];
        diag_invert2(a, 16, 2 * l, x, y);
        TOut *op = reinterpret_cast<TOut *>(p.out) + (int64_t(m[0].row0) * rs + (m[0].h * 16 + 2 * l));
        if (m[0].n == 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i, op += rs) put2(op, x[i], y[i]);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i, op += rs)
                if (i < m[0].n) put2(op, x[i], y[i]);
        }
        __syncwarp(mask);                  // stage k % S is refilled next
#pragma unroll
        for (int s = 0; s < S - 1; ++s) m[s] = m[s + 1];
    }
}

// ------------------------------------------------------------ 32 tokens
// Ring stage of one warp: blocks (0,0), (1,0), (1,1) of the chunk, each 16x16
// row-major with pitch 16 elements, at 256-element strides.  Rows 0..15 need
// 16 columns, rows 16..31 all 32: lane l copies 16 bytes of top rows i0,
// i0 + DT, ... and of bottom rows 16 + j0, 16 + j0 + DB, ...
template <typename TIn>
__device__ __forceinline__ void issue32(const SmallParams &p, const Meta &m, TIn *stage, int lane) {
    constexpr int VEC = Elt<TIn>::VEC;
    constexpr int PT = 16 / VEC, PB = 32 / VEC;        // 16-byte copies per top / bottom row
    constexpr int DT = 32 / PT, DB = 32 / PB;          // rows between a lane's copies
    if (!m.valid) return;
    const int rs = p.H * 32;
    const TIn *base = reinterpret_cast<const TIn *>(p.A) + (int64_t(m.row0) * rs + m.h * 32);
    {
        const int i0 = lane / PT, k = (lane % PT) * VEC;
        const TIn *src = base + (i0 * rs + k);
#pragma unroll
        for (int it = 0; it < 16 / DT; ++it) {
            const bool live = i0 + DT * it < m.n;
            cp_async16(stage + (i0 + DT * it) * 16 + k, live ? src : p.A, live ? 16u : 0u);
            src += DT * rs;
        }
    }
    {
        const int j0 = lane / PB, k = (lane % PB) * VEC;
        const TIn *src = base + ((16 + j0) * rs + k);
        TIn *dst = stage + (1 + (k >> 4)) * 256 + j0 * 16 + (k & 15);
#pragma unroll
        for (int it = 0; it < 16 / DB; ++it) {
            const bool live = 16 + j0 + DB * it < m.n;
            cp_async16(dst + DB * 16 * it, live ? src : p.A, live ? 16u : 0u);
            src += DB * rs;
        }
    }
}

// 32-token chunks: warp w of CTA b solves chunk-heads 2b + w, 2b + w + 2 grid, ...
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NTHREADS, 10)
kda_bt32_kernel(const SmallParams p) {
    constexpr int S = SMALL_STAGES;
    constexpr bool AX = sizeof(TIn) == 2;    // A values exact in TF32
    __shared__ __align__(16) TIn ring[2][S][3 * 256];
    __shared__ __align__(16) float af[2][AX ? 512 : 4];   // widened diagonal blocks (16-bit input)
    __shared__ __align__(16) float xt[2][256];    // X00^T, pitch XTP
    __shared__ __align__(16) float xr[2][XRS];    // -X11, pitch XRP
    __shared__ int32_t cu_s[SMALL_CU_CAP];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = (tid >> 4) & 1, l = tid & 15;
    const int g = lane >> 2, t = lane & 3;
    const int32_t slots = gridDim.x * 2;
    const int32_t q0 = blockIdx.x * 2 + warp;
    const int os = p.H * 32;
    pdl_launch_dependents();
    pdl_wait();                              // the previous kernel's writes are visible
    const SmallParams ps = with_cached_cu(p, cu_s, tid);
    SlotWalk<32> walk(ps, q0, slots);
    Meta m[S];
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        m[s] = walk.next(ps);
        issue32<TIn>(p, m[s], ring[warp][s], lane);
        cp_async_commit();
    }
    for (int k = 0;; ++k) {
        m[S - 1] = walk.next(ps);
        issue32<TIn>(p, m[S - 1], ring[warp][(k + S - 1) % S], lane);
        cp_async_commit();
        if (!m[0].valid) {                 // later chunk-heads are past the end too (nothing issued)
            cp_async_wait<0>();
            break;
        }
        cp_async_wait<S - 1>();
        __syncwarp();
        const TIn *a = ring[warp][k % S];
        const int n = m[0].n;
        TOut *ob = reinterpret_cast<TOut *>(p.out) + (int64_t(m[0].row0) * os + m[0].h * 32);
        {
            const float *d = reinterpret_cast<const float *>(a) + (half ? 512 : 0);
            if constexpr (AX) {              // blocks (0,0) and (1,1)
                widen_blocks(a, 2, af[warp], 2, lane, 32);
                __syncwarp();
                d = af[warp] + (half ? 256 : 0);
            }
            float x[16];
            diag_invert<true>(d, 16, l, x);
            TOut *op = ob + (16 * half * os + 16 * half + l);   // diagonal block, lane = column
            if (n == 32) {
#pragma unroll
                for (int i = 0; i < 16; ++i, op += os) put1(op, x[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i, op += os)
                    if (16 * half + i < n) put1(op, x[i]);
            }
            if (!half) {                     // X00^T row-major (row = lane)
                float4 *d = reinterpret_cast<float4 *>(xt[warp] + l * XTP);
#pragma unroll
                for (int i = 0; i < 4; ++i) d[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
            } else {                         // -X11 row-major (column = lane)
#pragma unroll
                for (int i = 0; i < 16; ++i) xr[warp][i * XRP + l] = -x[i];
            }
        }
        {                                    // zero block (0,1): rows 0..15 below n, columns 16..31
            constexpr int VEC = 16 / int(sizeof(TOut));
#pragma unroll
            for (int e = lane; e < 16 * (16 / VEC); e += 32) {
                const int r = e / (16 / VEC), c = 16 + VEC * (e % (16 / VEC));
                if (r < n) *reinterpret_cast<uint4 *>(ob + (r * os + c)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncwarp();
        // X10^T = (X00^T A10^T) (-X11)^T
        TileA la;
        TileB rb;
        TileC c1, c2;
        left_smem(la, xt[warp], XTP, g, t);
        right4a(rb, a + 256, 16, g, t);
        zero(c1);
        mma_tile<AX>(c1, la, rb);
        left_regs(la, c1);
        right2(rb, xr[warp], XRP, g, t);
        zero(c2);
        mma_tile<false>(c2, la, rb);
        out_tile_t<32>(ob, os, n, 1, 0, c2, g, t);
        __syncwarp();                        // xt, xr and stage k % S are rewritten next
#pragma unroll
        for (int s = 0; s < S - 1; ++s) m[s] = m[s + 1];
    }
}

}  // namespace kda
