// kda_kgb.cuh -- KDA's chunk matrix built from keys, betas and decays on the
// fifth-generation tensor cores (tcgen05, accumulator in tensor memory), fused
// with the 64-token solve: A never leaves the SM.
//
// LightLLM PR #1703 (PR description) has KDA prefill use the shared solver;
// the matrix it inverts is KDA's intra-chunk matrix
//     A[i][j] = beta_i sum_d k_id k_jd exp(g_id - g_jd),   j < i,
// with g the per-channel cumulative log decay (non-increasing along a chunk).
//
// Construction.  With one reference value c_d per channel (g of the chunk's
// middle live row),
//     A = beta * strict_lower(Q P^T),  Q[i][d] = k_id 2^{(g_id - c_d) log2 e},
//                                      P[j][d] = k_jd 2^{(c_d - g_jd) log2 e},
// one 64 x 64 x K product per chunk-head.  A channel whose decay over the
// chunk's live rows takes g further than KGB_TC_SAFE nats from c_d on either
// side would lose accuracy in these factors (the rounding of the exponent grows
// with its size) or overflow them: it is left out of the product (Q = P = 0)
// and its terms k_id k_jd exp(g_id - g_jd) are added one by one (a slow path
// that KDA's ordinary decays, about one nat per token, never take).
//
// FP32 accuracy on TF32 tensor cores: Q = Qh + Ql and P = Ph + Pl with Qh, Ph
// truncated to TF32 and Ql, Pl the TF32 remainders, which sum to Q P^T to about
// 2^-22 relative as Qh Ph^T + Qh Pl^T + Ql Ph^T (Ql Pl^T is dropped).  The
// operand buffer holds rows [Qh; Ql] (A side) and [Ph; Pl] (B side); each step
// of K = 8 channels issues three tcgen05.mma of M = 128, N = 64 into one FP32
// accumulator (128 TMEM lanes x 64 columns): A from Qh, Qh, Ql against B from
// Ph, Pl, Ph.  Accumulator rows 0-63 (TMEM lanes 0-63) are then Q P^T; rows
// 64-127 multiply the 64 operand rows that follow the A start and are not read.
// K = 128 channels take 48 instructions.
//
// One persistent CTA per SM, 16 warps in five roles; every role walks the
// chunk-heads q = blockIdx.x + c * gridDim.x in the same order:
//   * warp 0, lane 0 (loader): TMA loads of each chunk-head's k and g, one
//     slice of 32 channels at a time, into a ring of KGB_NST staging slots;
//   * warp 1, lane 0 (MMA issue): for every slice whose operands are ready,
//     twelve tcgen05.mma (four steps of K = 8) into TMEM buffer c % 2, with tcgen05.commit
//     releasing the operand buffer and, after a chunk-head's last slice, the
//     accumulator.  Issuing a TMA or tensor-core instruction holds the issuing
//     warp for a while, so the two streams run on warps of their own;
//   * warps 2-7 and 10-11 (transform): each slice of the staging ring into the
//     four TF32 operand parts in a 128-byte-swizzled buffer (three-slice ring);
//     every warp signals the MMA warp on its own mbarrier arrival, without a
//     group barrier;
//   * warps 8-9 (epilogue): tcgen05.ld of accumulator rows 0-31 (warp 8, TMEM
//     lanes 0-31) and 32-63 (warp 9; a warp reaches the lanes 32 (w % 4) .. + 31),
//     beta and the strict-lower and live-row masks applied, any steep
//     channels' terms added, into the ten lower 16 x 16 blocks of the A tile of
//     solve pair c % 2;
//   * warps 12-13 and 14-15 (solve pairs 0, 1): the 64-token solve of the A
//     tile (diagonal forward substitution, two merge levels on mma.sync) for
//     the chunk-heads c with c % 2 == pair.  The pairs share one copy of the
//     solve's code (barrier ids in registers).
// Hand-offs are mbarriers with bounded waits: staging slot full (TMA bytes) and
// empty (transform warps), operand buffer full (transform warps) and empty (MMA
// commit), accumulator full (MMA commit + the producer's release arrive) and
// empty (epilogue), A tile full (epilogue) and empty (solve pair).
#pragma once

#include "kda_kernels.cuh"
#include "kda_small.cuh"
#include "kda_tc.cuh"

namespace kda {

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
    unsigned *err;             // device error word
};

// Tensor maps of k and g viewed as {K channels, H heads, rows}, boxes of 32
// channels x 1 head x 64 rows.
struct KgbMaps {
    CUtensorMap k, g;
};

constexpr int KGB_THREADS = 512;
constexpr int KGB_TWARPS = 8;                      // transform warps 2 .. 7 and 10 .. 11
constexpr int KGB_EW0 = 8;                         // epilogue warps 8, 9: TMEM lane quarters 0, 1
constexpr int KGB_EWARPS = 2;
constexpr int KGB_SW0 = 12;                        // first solve warp
constexpr int KGB_PAIRS = (KGB_THREADS / 32 - KGB_SW0) / 2;   // solve pairs
constexpr int KGB_TTHREADS = 32 * KGB_TWARPS;
static_assert(KGB_EW0 % 4 == 0 && KGB_EWARPS == 2, "the epilogue warps reach TMEM lanes 0-63");
// transform warp index 0 .. KGB_TWARPS - 1 of warp w (warps 2-7, then 10-11)
__device__ __forceinline__ int kgb_twarp(int w) { return w < KGB_EW0 ? w - 2 : w - 2 - KGB_EWARPS; }
// largest distance (nats) of g from the channel's reference over the chunk that
// the tensor-core product takes; further channels go through the slow path
constexpr float KGB_TC_SAFE = 48.0f;

// staging ring of raw k and g slices (one 64-row x 32-channel box of each)
constexpr int KGB_NST = 4;
constexpr int KGB_STAGE_BYTES = 2 * 64 * 128;      // k box (<= 8 KiB), then the g box at +8 KiB
constexpr int KGB_STAGE_G = 64 * 128;
// ring of TF32 operand buffers (one slice each): the transform of slice u waits
// only for the MMAs of slice u - KGB_NOPS, so the slowest transform warp and the
// MMA latency stay off the transform's path
constexpr int KGB_NOPS = 3;

// mbarriers
constexpr int BAR_ST_FULL = 0;                     // [KGB_NST]
constexpr int BAR_ST_EMPTY = KGB_NST;              // [KGB_NST]
constexpr int BAR_OPS_FULL = 2 * KGB_NST;          // [KGB_NOPS]
constexpr int BAR_OPS_EMPTY = BAR_OPS_FULL + KGB_NOPS;   // [KGB_NOPS]
constexpr int BAR_D_FULL = BAR_OPS_EMPTY + KGB_NOPS;     // [2]
constexpr int BAR_D_EMPTY = BAR_D_FULL + 2;        // [2]
constexpr int BAR_AT_FULL = BAR_D_EMPTY + 2;       // [KGB_PAIRS]
constexpr int BAR_AT_EMPTY = BAR_AT_FULL + KGB_PAIRS;   // [KGB_PAIRS]
constexpr int KGB_NBARS = BAR_AT_EMPTY + KGB_PAIRS;

// shared memory (bytes)
constexpr int KGB_OFF_BAR = 0;
constexpr int KGB_OFF_TMEM = KGB_NBARS * 8;        // TMEM base address written by tcgen05.alloc
// steep-channel masks [8 chunk-heads][4 slices]: a ring deep enough that the
// transform cannot overwrite a chunk-head's masks before its epilogue is done
constexpr int KGB_OFF_STEEP = KGB_OFF_TMEM + 64;
constexpr int KGB_OFF_OPS = 1024;                  // [KGB_NOPS slices] {A: 128 x 128 B, B: 128 x 128 B}
constexpr int KGB_OPS_BYTES = 2 * 128 * 128;
constexpr int KGB_OFF_STAGE = KGB_OFF_OPS + KGB_NOPS * KGB_OPS_BYTES;   // [KGB_NST] staging slots
constexpr int KGB_OFF_AT = KGB_OFF_STAGE + KGB_NST * KGB_STAGE_BYTES;  // [pairs] A tile, 10 blocks of 16 x 16
constexpr int KGB_OFF_X = KGB_OFF_AT + KGB_PAIRS * 10 * 256 * 4;       // [pairs] inverse tiles of the merge
constexpr int KGB_X_FLOATS = 4 * XTS + 4 * XRS;
constexpr int KGB_OFF_SC = KGB_OFF_X + KGB_PAIRS * KGB_X_FLOATS * 4;   // slow path: one channel's k and g, 64 rows
constexpr int KGB_OFF_CU = KGB_OFF_SC + 2 * 64 * 4;              // cu_seqlens copy (packed, < CU_CAP requests)
constexpr int KGB_BYTES = KGB_OFF_CU + CU_CAP * 4 + 1024;         // + alignment slack
static_assert(KGB_OFF_STEEP + 8 * 4 * 4 <= KGB_OFF_OPS, "header fits");
static_assert(KGB_OFF_OPS % 1024 == 0 && KGB_OPS_BYTES % 1024 == 0, "swizzle atoms are 1024-byte aligned");
static_assert(KGB_OFF_STAGE % 128 == 0 && KGB_STAGE_BYTES % 128 == 0, "TMA destinations are 128-byte aligned");
static_assert(KGB_BYTES <= 227 * 1024, "fits the shared memory of one CTA");

constexpr uint32_t KGB_TMEM_COLS = 512;            // the whole TMEM of the SM (one CTA per SM)
constexpr uint32_t KGB_IDESC = tc::idesc_tf32<128, 64>();
constexpr uint32_t KGB_DCOLS = 64;                 // accumulator columns per TMEM buffer

// Chunk-heads q = q0, q0 + step, ... (every thread of a group walks the same sequence).
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

// 2^x on the SFU (PTX ex2.approx.ftz.f32; relative error about 2^-22)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int ID, int N>
__device__ __forceinline__ void named_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
}
// Named barrier that also ANDs a flag over its N threads (so that a group
// leaves its loop together, never stranding a member at a later barrier).
template <int ID, int N>
__device__ __forceinline__ bool named_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(v)), "n"(ID), "n"(N)
        : "memory");
    return r != 0;
}

// Wait for phase `parity` of an mbarrier; false (and the error word set) after
// WAIT_LIMIT_NS.
__device__ __forceinline__ bool kgb_wait(uint64_t *bars, int b, uint32_t parity, unsigned *err) {
    if (mbar_wait_bounded(&bars[b], parity)) return true;
    atomicOr(err, ERR_WAIT_TIMEOUT);
    return false;
}

// --------------------------------------------------------- transform group
// TMA loads of slice s (channels 32 s .. 32 s + 31) of chunk-head m's 64 rows
// of k and g into a staging slot (rows past the tensor's end are zero-filled;
// rows past the chunk's end are masked by the transform).
template <typename TIn>
__device__ __forceinline__ void kgb_tma_slice(const KgbMaps &maps, const Meta &m, int s, unsigned char *slot,
                                              uint64_t *full) {
    constexpr uint32_t BYTES = 64 * 32 * sizeof(TIn) + 64 * 32 * 4;
    mbar_arrive_expect_tx(full, BYTES);
    tma_load_3d(slot, &maps.k, 32 * s, m.h, m.row0, full);
    tma_load_3d(slot + KGB_STAGE_G, &maps.g, 32 * s, m.h, m.row0, full);
}

__device__ __forceinline__ void load4(const unsigned char *row, int c, const float *, float (&v)[4]) {
    const float4 x = *reinterpret_cast<const float4 *>(row + 16 * c);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
}
template <typename T16>
__device__ __forceinline__ void load4(const unsigned char *row, int c, const T16 *, float (&v)[4]) {
    const uint2 x = *reinterpret_cast<const uint2 *>(row + 8 * c);
    const T16 *h = reinterpret_cast<const T16 *>(&x);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = float(h[i]);
}

// TF32 split of two values at once: hi truncated to TF32 (explicitly, so that
// hi + lo is the value whatever the tensor core does with low mantissa bits),
// lo = v - hi exactly (FP32 subtraction of numbers that share their top bits);
// the tensor core reads lo as TF32, an error of at most 2^-11 |lo| <= 2^-22 |v|.
__device__ __forceinline__ void split2(float2 v, uint32_t &h0, uint32_t &h1, uint32_t &l0, uint32_t &l1) {
    h0 = __float_as_uint(v.x) & 0xffffe000u;
    h1 = __float_as_uint(v.y) & 0xffffe000u;
    const float2 lo = __fadd2_rn(v, make_float2(-__uint_as_float(h0), -__uint_as_float(h1)));
    l0 = __float_as_uint(lo.x);
    l1 = __float_as_uint(lo.y);
}

// Slice in the staging slot -> the four operand parts in the swizzled buffer
// `ops` (A rows 0-63 Qh, 64-127 Ql; B rows 0-63 Ph, 64-127 Pl).  Transform
// thread tt (0 .. KGB_TTHREADS - 1; KGB_TTHREADS a multiple of 8) handles
// channels 4 (tt & 7) .. + 3 of rows (tt + KGB_TTHREADS v) >> 3.  Returns this
// thread's 4-bit mask of channels left out as steep.
//
// Rows at or past the chunk's end are transformed like live rows: whatever they
// hold (zeros past the tensor's end, the next request's tokens), they only reach
// accumulator rows i >= n and columns j >= n, which the epilogue's strict-lower
// and live-row selects discard.  Pairs of values go through the paired FP32
// instructions (each half rounds exactly like its scalar form).
template <typename TIn>
__device__ __forceinline__ uint32_t kgb_tc_transform(const unsigned char *stage, unsigned char *ops, int n,
                                                     int tt) {
    constexpr float LH = 1.4426950408889634f;
    constexpr float SAFE2 = KGB_TC_SAFE * LH;
    constexpr int KP = 32 * int(sizeof(TIn));          // bytes per staged key row
    const unsigned char *kb = stage, *gb = stage + KGB_STAGE_G;
    unsigned char *A = ops, *B = ops + 128 * 128;
    const int c = tt & 7;
    // reference: g of the middle live row; steep: g leaves [c - SAFE, c + SAFE]
    float ref[4], gfirst[4], glast[4];
    load4(gb + ((n - 1) >> 1) * 128, c, (const float *)nullptr, ref);
    load4(gb, c, (const float *)nullptr, gfirst);
    load4(gb + (n - 1) * 128, c, (const float *)nullptr, glast);
    uint32_t steep = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float up = (gfirst[i] - ref[i]) * LH, dn = (ref[i] - glast[i]) * LH;
        const bool keep = up <= SAFE2 && dn <= SAFE2;   // false for NaN too
        steep |= keep ? 0u : (1u << i);
    }
    const float2 nref01 = make_float2(-ref[0], -ref[1]), nref23 = make_float2(-ref[2], -ref[3]);
    const float2 lh2 = make_float2(LH, LH);
    static_assert(KGB_TTHREADS % 8 == 0, "a thread keeps its channel group");
#pragma unroll
    for (int v = 0; v < (64 * 8 + KGB_TTHREADS - 1) / KGB_TTHREADS; ++v) {
        if (tt + KGB_TTHREADS * v >= 64 * 8) break;
        const int r = (tt + KGB_TTHREADS * v) >> 3;
        float kv[4], gv[4];
        load4(kb + r * KP, c, (const TIn *)nullptr, kv);
        load4(gb + r * 128, c, (const float *)nullptr, gv);
        // the exponent (g - ref) log2 e: the difference is taken first, so its
        // error does not grow with |g|
        float2 e01 = __fmul2_rn(__fadd2_rn(make_float2(gv[0], gv[1]), nref01), lh2);
        float2 e23 = __fmul2_rn(__fadd2_rn(make_float2(gv[2], gv[3]), nref23), lh2);
        float2 k01 = make_float2(kv[0], kv[1]), k23 = make_float2(kv[2], kv[3]);
        if (steep != 0u) {
            // a steep channel enters the product as zeros: key 0, exponent 0
            // (selected, so that no 0 * inf arises)
            if (steep & 1u) k01.x = e01.x = 0.f;
            if (steep & 2u) k01.y = e01.y = 0.f;
            if (steep & 4u) k23.x = e23.x = 0.f;
            if (steep & 8u) k23.y = e23.y = 0.f;
        }
        const float2 q01 = __fmul2_rn(k01, make_float2(ex2(e01.x), ex2(e01.y)));
        const float2 q23 = __fmul2_rn(k23, make_float2(ex2(e23.x), ex2(e23.y)));
        const float2 p01 = __fmul2_rn(k01, make_float2(ex2(-e01.x), ex2(-e01.y)));
        const float2 p23 = __fmul2_rn(k23, make_float2(ex2(-e23.x), ex2(-e23.y)));
        uint4 qh, ql, ph, pl;
        split2(q01, qh.x, qh.y, ql.x, ql.y);
        split2(q23, qh.z, qh.w, ql.z, ql.w);
        split2(p01, ph.x, ph.y, pl.x, pl.y);
        split2(p23, ph.z, ph.w, pl.z, pl.w);
        const int sw = 16 * (c ^ (r & 7));             // swizzled chunk position (rows r and 64 + r alike)
        *reinterpret_cast<uint4 *>(A + r * 128 + sw) = qh;
        *reinterpret_cast<uint4 *>(A + (64 + r) * 128 + sw) = ql;
        *reinterpret_cast<uint4 *>(B + r * 128 + sw) = ph;
        *reinterpret_cast<uint4 *>(B + (64 + r) * 128 + sw) = pl;
    }
    return steep;
}

// ------------------------------------------------------------- solve pair
// The 64-token solve of the A tile (blocks (i, j) at Ab + 256 blk(i, j), pitch
// 16) by the 64 threads of one pair (tid 0..63, named barrier `bar`).
template <typename TOut>
__device__ __forceinline__ void kgb_solve(const float *Ab, float *Xt, float *Xr, TOut *ob, int os, int n, int tid,
                                          int bar) {
    const int unit = tid >> 4, warp = tid >> 5, l = tid & 15;
    const int lane = tid & 31, g = lane >> 2, t = lane & 3;
    {
        float x[16];
        const int b = unit;
        diag_invert<true>(Ab + blk(b, b) * 256, 16, l, x);   // the select form: fewer live registers
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
            for (int i = 0; i < 4; ++i) d[i ^ xt_swz(l)] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
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
        left_smem<true>(la, Xt + (warp == 0 ? XT_00 : XT_22) * XTS, XTP, g, t);
        right4<false>(rb, Ab + (warp == 0 ? blk(1, 0) : blk(3, 2)) * 256, 16, g, t);
        zero(c1);
        mma_tile<false>(c1, la, rb);
        left_regs(la, c1);
        right2(rb, Xr + (warp == 0 ? XR_11 : XR_33) * XRS, XRP, g, t);
        zero(c2);
        mma_tile<false>(c2, la, rb);
        if (warp == 0) {
            smem_tile_t<true>(Xt + XT_10 * XTS, c2, g, t);
            out_tile_t(ob, os, n, 1, 0, c2, g, t);
        } else {
            smem_tile_neg(Xr + XR_32 * XRS, c2, g, t);
            out_tile_t(ob, os, n, 3, 2, c2, g, t);
        }
    }
    bar64(bar);
    {   // level B, warp w = column block w of X_BL
        TileA la, lb;
        TileB rb;
        TileC ct2, ct3, cx;
        zero(ct2);
        zero(ct3);
        left_smem<true>(la, Xt + (warp == 0 ? XT_00 : XT_11) * XTS, XTP, g, t);
        right4<false>(rb, Ab + blk(2, warp) * 256, 16, g, t);
        mma_tile<false>(ct2, la, rb);
        right4<false>(rb, Ab + blk(3, warp) * 256, 16, g, t);
        mma_tile<false>(ct3, la, rb);
        if (warp == 0) {                               // + X10^T A21^T, X10^T A31^T
            left_smem<true>(la, Xt + XT_10 * XTS, XTP, g, t);
            right4<false>(rb, Ab + blk(2, 1) * 256, 16, g, t);
            mma_tile<false>(ct2, la, rb);
            right4<false>(rb, Ab + blk(3, 1) * 256, 16, g, t);
            mma_tile<false>(ct3, la, rb);
        }
        left_regs(la, ct2);
        left_regs(lb, ct3);
        TileB rb3;
        TileC cy;
        right2(rb, Xr + XR_22 * XRS, XRP, g, t);
        right2(rb3, Xr + XR_32 * XRS, XRP, g, t);
        zero(cx);
        zero(cy);
        mma_tile2<false>(cx, cy, la, rb, rb3);
        out_tile_t(ob, os, n, 2, warp, cx, g, t);
        right2(rb, Xr + XR_33 * XRS, XRP, g, t);
        mma_tile<false>(cy, lb, rb);
        out_tile_t(ob, os, n, 3, warp, cy, g, t);
    }
    store_upper_zeros(ob, os, n, tid);
}

// A tile element (i, j), j <= i (blocks (i/16, j/16) of the lower triangle).
__device__ __forceinline__ float *at_elem(float *Ab, int i, int j) {
    return Ab + blk(i >> 4, j >> 4) * 256 + (i & 15) * 16 + (j & 15);
}

// Solve pair PR: chunk-heads c = PR, PR + KGB_PAIRS, ... from A tile PR.
template <typename TOut>
__device__ __forceinline__ void kgb_pair_loop(const KgbParams &p, unsigned char *sm, uint64_t *bars, int PR,
                                              int pt) {
    float *Ab = reinterpret_cast<float *>(sm + KGB_OFF_AT) + PR * 2560;
    float *X = reinterpret_cast<float *>(sm + KGB_OFF_X) + PR * KGB_X_FLOATS;
    const int os = p.H * BT;
    KgbWalk walk(p, int32_t(blockIdx.x) + PR * int32_t(gridDim.x), KGB_PAIRS * int32_t(gridDim.x));
    Meta m = walk.next(p);
    for (uint32_t k = 0; m.valid; ++k, m = walk.next(p)) {
        const bool ok = kgb_wait(bars, BAR_AT_FULL + PR, k & 1, p.err);
        if (!bar64_and(4 + PR, ok)) break;
        TOut *ob = reinterpret_cast<TOut *>(p.out) + (int64_t(m.row0) * p.H + m.h) * BT;
        kgb_solve<TOut>(Ab, X, X + 4 * XTS, ob, os, m.n, pt, 4 + PR);
        __syncwarp();
        if ((pt & 31) == 0) mbar_arrive(&bars[BAR_AT_EMPTY + PR]);
    }
}

// ----------------------------------------------------------------- kernel
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(KGB_THREADS, 1)
kda_kgb_kernel(const __grid_constant__ KgbMaps maps, const KgbParams p) {
    extern __shared__ __align__(1024) unsigned char smraw[];
    // the swizzled operand buffers need 1024-byte aligned shared addresses
    unsigned char *sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + KGB_OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + KGB_OFF_TMEM);
    uint32_t *steep_m = reinterpret_cast<uint32_t *>(sm + KGB_OFF_STEEP);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsl = p.K / 32;
    const int32_t G = gridDim.x;
    pdl_launch_dependents();

    if (tid == 0) {
        prefetch_tensormap(&maps.k);
        prefetch_tensormap(&maps.g);
        for (int b = 0; b < KGB_NST; ++b) {
            mbar_init(&bars[BAR_ST_FULL + b], 1);
            mbar_init(&bars[BAR_ST_EMPTY + b], KGB_TWARPS);
        }
        for (int b = 0; b < KGB_NOPS; ++b) {
            mbar_init(&bars[BAR_OPS_FULL + b], KGB_TWARPS);
            mbar_init(&bars[BAR_OPS_EMPTY + b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[BAR_D_FULL + b], 2);
            mbar_init(&bars[BAR_D_EMPTY + b], KGB_EWARPS);
        }
        for (int b = 0; b < KGB_PAIRS; ++b) {
            mbar_init(&bars[BAR_AT_FULL + b], KGB_EWARPS);
            mbar_init(&bars[BAR_AT_EMPTY + b], 2);
        }
        fence_mbar_init();
    }
    // the previous kernel's writes are visible, and it holds no tensor memory
    pdl_wait();
    // every role's task walk reads cu_seqlens from shared memory when it fits
    KgbParams ps = p;
    if (p.cu != nullptr && p.nseq < CU_CAP) {
        int32_t *cs = reinterpret_cast<int32_t *>(sm + KGB_OFF_CU);
        for (int i = tid; i <= p.nseq; i += KGB_THREADS) cs[i] = __ldg(p.cu + i);
        ps.cu = cs;
    }
    if (warp == KGB_EW0) {                             // an epilogue warp owns the TMEM allocation
        tc::tmem_alloc(smem_u32(tmem_slot), KGB_TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------- loader (lane 0)
        if (lane == 0) {
            KgbWalk lw(ps, blockIdx.x, G);
            uint32_t lu = 0;
            for (Meta lm = lw.next(ps); lm.valid; lm = lw.next(ps)) {
                int ls = 0;
                for (; ls < nsl; ++ls, ++lu) {         // slice ls into its staging slot once it is free
                    const int slot = lu % KGB_NST;
                    if (!kgb_wait(bars, BAR_ST_EMPTY + slot, ((lu / KGB_NST) & 1) ^ 1, p.err)) break;
                    kgb_tma_slice<TIn>(maps, lm, ls, sm + KGB_OFF_STAGE + slot * KGB_STAGE_BYTES,
                                       &bars[BAR_ST_FULL + slot]);
                }
                if (ls < nsl) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issue (lane 0)
        if (lane == 0) {
            KgbWalk mw(ps, blockIdx.x, G);
            uint32_t mu = 0;
            bool ok = true;
            for (uint32_t mc = 0; ok; ++mc) {
                if (!mw.next(ps).valid) break;
                const int db = mc & 1;
                // the accumulator buffer's previous chunk-head has been read out
                ok = kgb_wait(bars, BAR_D_EMPTY + db, ((mc >> 1) & 1) ^ 1, p.err);
                for (int ms = 0; ok && ms < nsl; ++ms, ++mu) {
                    const int ob = mu % KGB_NOPS;
                    if (!(ok = kgb_wait(bars, BAR_OPS_FULL + ob, (mu / KGB_NOPS) & 1, p.err))) break;
                    tc::fence_after_sync();
                    // Qh, Ql (A side) and Ph, Pl (B side): 64 rows of 128 bytes each
                    const uint32_t qh = smem_u32(sm + KGB_OFF_OPS + ob * KGB_OPS_BYTES), ql = qh + 64 * 128;
                    const uint32_t ph = qh + 128 * 128, pl = ph + 64 * 128;
                    const uint32_t d = tmem + db * KGB_DCOLS;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {   // K = 8 channels: 32 bytes along the row
                        tc::mma_tf32(d, tc::sw128_desc(qh + 32 * kk), tc::sw128_desc(ph + 32 * kk), KGB_IDESC,
                                     ms > 0 || kk > 0);
                        tc::mma_tf32(d, tc::sw128_desc(qh + 32 * kk), tc::sw128_desc(pl + 32 * kk), KGB_IDESC, true);
                        tc::mma_tf32(d, tc::sw128_desc(ql + 32 * kk), tc::sw128_desc(ph + 32 * kk), KGB_IDESC, true);
                    }
                    tc::commit(smem_u32(&bars[BAR_OPS_EMPTY + ob]));
                    if (ms == nsl - 1) {
                        tc::commit(smem_u32(&bars[BAR_D_FULL + db]));
                        mbar_arrive(&bars[BAR_D_FULL + db]);     // releases the steep masks
                    }
                }
            }
        }
    } else if (warp < KGB_EW0 || (warp >= KGB_EW0 + KGB_EWARPS && warp < KGB_SW0)) {
        // --------------------------------------------------------- transform
        const int tt = 32 * kgb_twarp(warp) + lane;    // 0 .. KGB_TTHREADS - 1
        KgbWalk walk(ps, blockIdx.x, G);
        Meta m = walk.next(ps);
        uint32_t u = 0;
        bool ok = true;
        for (uint32_t c = 0; m.valid && ok; ++c, m = walk.next(ps)) {
            for (int s = 0; s < nsl; ++s, ++u) {
                const int slot = u % KGB_NST, ob = u % KGB_NOPS;
                ok = kgb_wait(bars, BAR_ST_FULL + slot, (u / KGB_NST) & 1, p.err) &&
                     kgb_wait(bars, BAR_OPS_EMPTY + ob, ((u / KGB_NOPS) & 1) ^ 1, p.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const uint32_t st = kgb_tc_transform<TIn>(sm + KGB_OFF_STAGE + slot * KGB_STAGE_BYTES,
                                                          sm + KGB_OFF_OPS + ob * KGB_OPS_BYTES, m.n, tt);
                if (warp == 2) {                       // lanes 0-7 cover the slice's 8 channel groups
                    const uint32_t word = __reduce_or_sync(0xffffffffu, st << (4 * (lane & 7)));
                    if (lane == 0) steep_m[(c & 7) * 4 + s] = word;
                }
                fence_proxy_async();                   // operand writes visible to the tensor cores
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars[BAR_OPS_FULL + ob]);
                    mbar_arrive(&bars[BAR_ST_EMPTY + slot]);
                }
            }
        }
    } else if (warp < KGB_EW0 + KGB_EWARPS) {
        // ---------------------------------------------------------- epilogue
        const int i = tid - 32 * KGB_EW0;              // chunk row of this thread = its TMEM lane, 0..63
        float *sk = reinterpret_cast<float *>(sm + KGB_OFF_SC), *sg = sk + 64;
        KgbWalk walk(ps, blockIdx.x, G);
        Meta m = walk.next(ps);
        for (uint32_t c = 0; m.valid; ++c, m = walk.next(ps)) {
            const int pr = c % KGB_PAIRS, db = c & 1;
            float *Ab = reinterpret_cast<float *>(sm + KGB_OFF_AT) + pr * 2560;
            // beta of row i, loaded before the waits so that its latency hides behind them
            const float bi = i < m.n ? float(reinterpret_cast<const TIn *>(p.beta)[(int64_t(m.row0) + i) * p.H + m.h])
                                     : 0.f;
            bool ok = kgb_wait(bars, BAR_AT_EMPTY + pr, ((c / KGB_PAIRS) & 1) ^ 1, p.err);
            ok = ok && kgb_wait(bars, BAR_D_FULL + db, (c >> 1) & 1, p.err);
            if (!named_sync_and<3, 64>(ok)) break;
            tc::fence_after_sync();
            const uint32_t sbase = (c & 7) * 4;
            const uint32_t any_steep = (nsl > 0 ? steep_m[sbase] : 0u) | (nsl > 1 ? steep_m[sbase + 1] : 0u) |
                                       (nsl > 2 ? steep_m[sbase + 2] : 0u) | (nsl > 3 ? steep_m[sbase + 3] : 0u);
            const uint32_t tq = tmem + db * KGB_DCOLS + (uint32_t(32 * (warp - KGB_EW0)) << 16);
            float v[4][16];
#pragma unroll
            for (int j0 = 0; j0 < 4; ++j0) tc::ld16(tq + 16 * j0, v[j0]);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BAR_D_EMPTY + db]);
#pragma unroll
            for (int j0 = 0; j0 < 4; ++j0) {
                if (16 * j0 <= i) {                    // the row's blocks left of and on the diagonal
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        float o[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int j = 16 * j0 + e + x;
                            o[x] = (j < i && i < m.n) ? bi * v[j0][e + x] : 0.f;   // select: dropped rows may be NaN
                        }
                        *reinterpret_cast<float4 *>(at_elem(Ab, i, 16 * j0 + e)) = make_float4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            if (any_steep != 0u) {
                // slow path: the steep channels' terms, k_i k_j exp(g_i - g_j), one by one
                constexpr float L2E = 1.4426950408889634f;
                const int64_t rs = int64_t(p.H) * p.K;
                for (int jh = 0; jh < 2; ++jh) {       // columns 32 jh .. 32 jh + 31 of row i
                    float acc[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) acc[x] = 0.f;
                    for (int s = 0; s < nsl; ++s) {
                        uint32_t mask = steep_m[sbase + s];
                        while (mask != 0u) {
                            const int d = 32 * s + __ffs(mask) - 1;
                            mask &= mask - 1u;
                            named_sync<3, 64>();         // previous channel's values consumed
                            const bool live = i < m.n;
                            const int64_t off = (int64_t(m.row0) + i) * rs + int64_t(m.h) * p.K + d;
                            sk[i] = live ? float(reinterpret_cast<const TIn *>(p.k)[off]) : 0.f;
                            sg[i] = live ? p.g[off] : 0.f;
                            named_sync<3, 64>();
                            const float ki = sk[i], gi = sg[i];
#pragma unroll
                            for (int x = 0; x < 32; ++x) {
                                const int j = 32 * jh + x;
                                if (j < i) acc[x] = fmaf(ki * sk[j], ex2((gi - sg[j]) * L2E), acc[x]);
                            }
                        }
                    }
                    if (i < m.n) {
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            const int j = 32 * jh + x;
                            if (j < i) *at_elem(Ab, i, j) += bi * acc[x];
                        }
                    }
                }
                named_sync<3, 64>();                     // sk, sg free for the next chunk-head
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BAR_AT_FULL + pr]);     // releases the A tile
        }
    } else {
        // -------------------------------------------------------- solve pairs
        const int pr = (warp - KGB_SW0) >> 1, pt = tid - 32 * KGB_SW0 - 64 * pr;   // pair, thread 0..63 in it
        kgb_pair_loop<TOut>(ps, sm, bars, pr, pt);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == KGB_EW0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, KGB_TMEM_COLS);
    }
}

}  // namespace kda
