// kda_small.cuh -- the 32- and 16-token branches of the chunk solver.
//
// LightLLM PR #1703 (PR description) calls the path it optimises the shared
// solver's "64-token branch"; the same inversion of (I + A) for the strictly
// lower-triangular chunk matrix A is solved here for chunks of 16 and 32
// tokens, with the same building blocks as the 64-token kernel:
//   * 16 tokens: one 16-lane unit per chunk-head, forward substitution with one
//     lane per column (FP32 FMA);
//   * 32 tokens: one warp per chunk-head; its two units invert the diagonal
//     16x16 blocks, then X10 = -X11 A10 X00 runs on the tensor cores in split
//     TF32, computed transposed as in the 64-token kernel's level A.
// Persistent CTAs of 64 threads walk chunk-heads q = slot, slot + slots, ...
// Tiles are small (1-3 KiB), so loads are plain 16-byte vector loads into
// shared memory (widened to FP32, rows past a partial chunk's end zeroed);
// there is no asynchronous copy and no wait on a barrier other than the warp's
// own synchronisation.
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

// Rows [r_lo, r_hi) x columns [0, w) of the chunk-head's tile (row pitch `rs`
// elements in global memory) -> FP32 shared tile `dst` (pitch 16 per 16-column
// block: column c goes to block c / 16).  Rows at or past n become zeros and
// are not read.  `lanes` threads starting at lane 0 of `lane` cooperate.
template <typename TIn>
__device__ __forceinline__ void load_rows(const TIn *src, int64_t rs, int r_lo, int r_hi, int w, int n,
                                          float *dst, int blk_stride, int lane, int lanes) {
    constexpr int VEC = Elt<TIn>::VEC;       // elements per 16-byte vector
    const int vpr = w / VEC;
    const int nv = (r_hi - r_lo) * vpr;
    for (int e = lane; e < nv; e += lanes) {
        const int i = r_lo + e / vpr;
        const int k = (e % vpr) * VEC;
        float f[VEC];
        if (i < n) {
            const uint4 v = *reinterpret_cast<const uint4 *>(src + i * rs + k);
            Elt<TIn>::widen(v, f);
        } else {
#pragma unroll
            for (int t = 0; t < VEC; ++t) f[t] = 0.f;
        }
        float *d = dst + (k >> 4) * blk_stride + (i & 15) * 16 + (k & 15);
#pragma unroll
        for (int t = 0; t < VEC; t += 4)
            *reinterpret_cast<float4 *>(d + t) = make_float4(f[t], f[t + 1], f[t + 2], f[t + 3]);
    }
}

// 16-token chunks: unit u of the CTA solves chunk-heads slot, slot + slots, ...
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NTHREADS, 20)
kda_bt16_kernel(const SmallParams p) {
    constexpr int CBT = 16;
    __shared__ __align__(16) float tile[4][256];
    const int tid = threadIdx.x, unit = tid >> 4, l = tid & 15;
    const unsigned mask = 0xffffu << (16 * (unit & 1));
    const int32_t slots = gridDim.x * 4;
    const int64_t rs = int64_t(p.H) * CBT;   // row stride (elements)
    Walk walk{0, 0};
    for (int32_t q = blockIdx.x * 4 + unit;; q += slots) {
        const Meta m = decode<CBT>(p, q, walk);
        if (!m.valid) break;
        const int64_t base = int64_t(m.row0) * rs + int64_t(m.h) * CBT;
        load_rows(reinterpret_cast<const TIn *>(p.A) + base, rs, 0, 16, 16, m.n, tile[unit], 256, l, 16);
        __syncwarp(mask);
        float x[16];
        diag_invert(tile[unit], 16, l, x);
        TOut *ob = reinterpret_cast<TOut *>(p.out) + base;
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i < m.n) put1(ob + i * rs + l, x[i]);
        __syncwarp(mask);                    // the tile is rewritten next
    }
}

// 32-token chunks: warp w of the CTA solves chunk-heads slot, slot + slots, ...
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NTHREADS, 12)
kda_bt32_kernel(const SmallParams p) {
    constexpr int CBT = 32;
    constexpr bool AX = sizeof(TIn) == 2;    // A values exact in TF32
    // per warp: A blocks (0,0), (1,0), (1,1) at stride 256, X00^T (pitch 16), -X11 (pitch 24)
    __shared__ __align__(16) float ab[2][3 * 256];
    __shared__ __align__(16) float xt[2][256];
    __shared__ __align__(16) float xr[2][XRS];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = tid >> 4, half = unit & 1, l = tid & 15;
    const int g = lane >> 2, t = lane & 3;
    const int32_t slots = gridDim.x * 2;
    const int64_t rs = int64_t(p.H) * CBT;
    const int os = p.H * CBT;
    Walk walk{0, 0};
    float *A0 = ab[warp];                    // block (0,0); (1,0) at +256; (1,1) at +512
    for (int32_t q = blockIdx.x * 2 + warp;; q += slots) {
        const Meta m = decode<CBT>(p, q, walk);
        if (!m.valid) break;
        const int64_t base = int64_t(m.row0) * rs + int64_t(m.h) * CBT;
        const TIn *src = reinterpret_cast<const TIn *>(p.A) + base;
        load_rows(src, rs, 0, 16, 16, m.n, A0, 0, lane, 32);           // block (0,0)
        load_rows(src, rs, 16, 32, 32, m.n, A0 + 256, 256, lane, 32);  // blocks (1,0), (1,1)
        __syncwarp();
        TOut *ob = reinterpret_cast<TOut *>(p.out) + base;
        {
            float x[16];
            diag_invert(A0 + (half ? 512 : 0), 16, l, x);
#pragma unroll
            for (int i = 0; i < 16; ++i) {   // diagonal block of the output, lane = column
                const int r = 16 * half + i;
                if (r < m.n) put1(ob + (r * os + 16 * half + l), x[i]);
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
        // zero block (0,1): rows 0..15 below n, columns 16..31
        {
            constexpr int VEC = 16 / int(sizeof(TOut));
#pragma unroll
            for (int e = lane; e < 16 * (16 / VEC); e += 32) {
                const int r = e / (16 / VEC), c = 16 + VEC * (e % (16 / VEC));
                if (r < m.n) *reinterpret_cast<uint4 *>(ob + (r * os + c)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncwarp();
        // X10^T = (X00^T A10^T) (-X11)^T
        TileA la;
        TileB rb;
        TileC c1, c2;
        left_smem(la, xt[warp], XTP, g, t);
        right4<AX>(rb, A0 + 256, 16, g, t);
        zero(c1);
        mma_tile<AX>(c1, la, rb);
        left_regs(la, c1);
        right2(rb, xr[warp], XRP, g, t);
        zero(c2);
        mma_tile<false>(c2, la, rb);
        out_tile_t(ob, os, m.n, 1, 0, c2, g, t);
        __syncwarp();                        // the tiles are rewritten next
    }
}

}  // namespace kda
