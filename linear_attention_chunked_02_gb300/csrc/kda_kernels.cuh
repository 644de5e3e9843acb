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
//   * One thread (thread 0; thread 32 in the single pass on 16-bit input)
//     issues TMA tile loads (cp.async.bulk.tensor, mbarrier completion) into a
//     2-stage ring, so the next chunk-head is in flight while the current one
//     is computed.  The single pass fetches two boxes, rows 0-31 x columns
//     0-31 and rows 32-63 x columns 0-63: exactly the 128-byte lines that hold
//     the strictly lower triangle, in two TMA instructions (issuing a TMA
//     instruction holds up the issuer's warp, so fewer, larger boxes shorten
//     the critical path).  FP32 input is used in
//     place from the landing buffer; 16-bit input is widened once.
//   * Diagonal blocks: one unit per block, one lane per column, forward
//     substitution in registers (FP32 FMA).
//   * Merge, as two 32x32 levels (the 64x64 matrix is lower block-triangular
//     with 32x32 blocks TL, BR and off-diagonal BL):
//        level A: X10 = -X11 A10 X00,  X32 = -X33 A32 X22
//        level B: T = A_BL X_TL,  X_BL = -X_BR T
//     which is Linv_ij = -Linv_ii sum_k A_ik Linv_kj regrouped.  The 16x16x16
//     products run on the tensor cores (mma.sync TF32, split into hi + lo
//     parts so the result keeps FP32 accuracy) and are computed transposed
//     (T^T = X_TL^T A_BL^T, X_BL^T = T^T (-X_BR)^T): A is then read row-major
//     straight from the landing buffer, and each intermediate T stays in
//     registers as the next product's left operand.  One barrier per chunk-head.
//   * On 16-bit input the inverse tiles and the widened diagonal blocks are kept
//     in shared memory with their 16-byte chunks swizzled by row, so that a
//     quarter-warp's stores and fragment reads hit distinct banks.
//   * Every output block is stored from the registers that computed it; the
//     zero blocks above the diagonal are 16-byte vector stores.
//   * Split path: MODE_DIAG inverts the diagonal blocks, writes them (and the
//     zero blocks) to the output and their transposed FP32 tiles to the
//     workspace; MODE_MERGE loads the tiles back and produces the
//     off-diagonal blocks.
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

// cu_seqlens entries cached in shared memory (packed batches of up to 255
// requests); larger batches walk cu_seqlens in global memory
constexpr int CU_CAP = 256;

constexpr int MODE_FUSED = 0;
constexpr int MODE_DIAG = 1;
constexpr int MODE_MERGE = 2;
// launch selector for the single pass in the TF32 precision mode (the kernel is
// MODE_FUSED with its TF32 template flag set)
constexpr int MODE_FUSED_TF32 = 3;

// On-chip FP32 tiles.  Widened 16-bit A blocks: pitch 16, block stride 272
// floats.  X tiles: "Xt" slots hold transposed inverse blocks row-major with
// pitch 16 (left operands, one 16-byte load per fragment row), "Xr" slots hold
// negated inverse blocks row-major with pitch 24 (right operands, 8-byte loads
// that fall in distinct banks).
constexpr int AP16 = 16;
constexpr int ABS = 272;
constexpr int XTP = 16, XTS = 256;     // Xt pitch / slot stride (floats)
constexpr int XRP = 24, XRS = 384;     // Xr pitch / slot stride (floats)

// Shared-memory swizzles of rows of 16 floats (four 16-byte chunks; chunk c of
// row r stored at c ^ swz(r)), so that the 16-byte accesses of a quarter-warp
// fall in distinct banks.  Xt (16-bit input, and the fused construction
// kernel's solve): a lane writing row l of a transposed inverse puts its four
// chunks at distinct banks from its neighbours', and the MMA fragment reads
// (rows g, g + 1 of a quarter-warp) stay conflict-free.  Widened A blocks: the
// two 16-byte stores of each widening lane land on distinct banks across rows.
__host__ __device__ constexpr int xt_swz(int r) { return (r >> 1) & 3; }
__host__ __device__ constexpr int af_swz(int r) { return (r >> 1) & 1; }

__host__ __device__ constexpr int blk(int i, int j) { return i * (i + 1) / 2 + j; }

// Xt slots: X00^T, X22^T, X11^T, X10^T.  Xr slots: -X11, -X33, -X22, -X32.
constexpr int XT_00 = 0, XT_22 = 1, XT_11 = 2, XT_10 = 3;
constexpr int XR_11 = 0, XR_33 = 1, XR_22 = 2, XR_32 = 3;

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
// Programmatic dependent launch (the kernels are launched with programmatic
// stream serialization).  launch_dependents lets the next kernel of the stream be
// scheduled onto SMs as this grid's CTAs leave; wait blocks until the previous
// kernel of the stream has completed and its memory writes are visible, so
// every kernel calls it before its first global memory access.  Both are no-ops
// for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// try_wait that may suspend the thread for up to `ns` nanoseconds; the thread
// resumes as soon as the phase completes, so a waiting warp issues few
// instructions (they would take issue slots from the warps doing work)
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// Wait for phase `parity` of `bar`; gives up (false) after limit_ns, checked
// every 64 suspended tries.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned long long limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_suspend(bar, parity, 100000u)) return true;
        if ((it & 63u) == 0u && globaltimer() - t0 > limit_ns) return false;
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

// Prefetch a tensor map (kernel parameter) into the TMA descriptor cache.
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
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
    // stage: raw TMA landing area (single pass: rows 0-31 x 32 columns, then
    // rows 32-63 x 64 columns; split kernels: 16-row boxes per block-row)
    static constexpr int A_ELEMS = MODE == MODE_FUSED ? 32 * 32 + 32 * 64 : MODE == MODE_DIAG ? 4 * 256 : 6 * 256;
    static constexpr int A_BYTES = A_ELEMS * ELT;
    static constexpr int WS_OFF = (A_BYTES + 127) / 128 * 128;
    static constexpr int STAGE_BYTES = MODE == MODE_MERGE ? WS_OFF + 4096 : WS_OFF;
    static constexpr uint32_t TX_BYTES = MODE == MODE_MERGE ? A_BYTES + 4096 : A_BYTES;
    static constexpr int NAF = WIDEN && MODE != MODE_MERGE ? 4 : 0;   // widened diagonal A blocks
    static constexpr int X_BYTES = MODE == MODE_DIAG ? 0 : 4 * (4 * XTS + 4 * XRS);
    static constexpr int OFF_BAR = 0;
    static constexpr int OFF_META = 64;
    static constexpr int OFF_STAGE = 128;
    static constexpr int OFF_AF = OFF_STAGE + STAGES * STAGE_BYTES;
    static constexpr int OFF_XT = OFF_AF + NAF * ABS * 4;
    static constexpr int OFF_XR = OFF_XT + (MODE == MODE_DIAG ? 0 : 4 * XTS * 4);
    // cu_seqlens of a packed batch of up to CU_CAP - 1 requests, so that the
    // per-task walk reads shared rather than global memory
    static constexpr int OFF_CU = OFF_XT + X_BYTES;
    static constexpr int BYTES = OFF_CU + CU_CAP * 4;
    static_assert(OFF_STAGE % 128 == 0 && STAGE_BYTES % 128 == 0,
                  "TMA destination buffers must be 128-byte aligned");
    // stage offset (bytes) of block-row r's first row, and its row pitch in elements
    __host__ __device__ static constexpr int row_off(int r) {
        return MODE == MODE_FUSED ? (r < 2 ? 16 * 32 * ELT * r : 32 * 32 * ELT + 16 * 64 * ELT * (r - 2))
             : MODE == MODE_DIAG  ? 256 * ELT * r
                                  : 256 * ELT * ((r - 1) * r / 2);
    }
    __host__ __device__ static constexpr int width(int r) {
        return MODE == MODE_FUSED ? (r < 2 ? 32 : 64) : MODE == MODE_DIAG ? 16 : 16 * r;
    }
    static constexpr int R0 = MODE == MODE_MERGE ? 1 : 0;   // first block-row fetched
};

// An FP32 view of diagonal A block b: pointer and row pitch (floats).  FP32
// input is read in place from the landing buffer; 16-bit input was widened.
struct AView {
    const float *p;
    int pitch;
};
template <int MODE, typename TIn>
__device__ __forceinline__ AView adiag(const unsigned char *stage, const float *Af, int b) {
    using L = Layout<MODE, TIn>;
    if (L::WIDEN) return {Af + b * ABS, AP16};
    const float *base = reinterpret_cast<const float *>(stage + L::row_off(b));
    return {MODE == MODE_DIAG ? base : base + 16 * b, L::width(b)};
}
// Off-diagonal A block (i, j), i > j, in the input dtype inside the landing buffer.
template <typename TIn>
struct AOff {
    const TIn *p;
    int pitch;                 // elements
};
template <int MODE, typename TIn>
__device__ __forceinline__ AOff<TIn> aoff(const unsigned char *stage, int i, int j) {
    using L = Layout<MODE, TIn>;
    const TIn *base = reinterpret_cast<const TIn *>(stage + L::row_off(i));
    return {base + 16 * j, L::width(i)};
}

// ------------------------------------------------------------ task decode
// Per-walker state: packed layout, the current request of cu_seqlens; dense
// layout, the current batch row.
struct Walk {
    int32_t s;        // current request (packed) or batch row (dense)
    int32_t cbase;    // chunks before it
};

template <int CBT = BT>
__device__ __forceinline__ int32_t nchunks(int32_t a, int32_t b) {
    const int32_t L = b - a;
    return L > 0 ? (L + CBT - 1) / CBT : 0;
}

// Chunk c, head h -> (first row, valid rows, head) for chunk length CBT; P has
// the layout fields cu, nseq, T, cpr.  w walks forward (cu_seqlens, or the batch
// rows), so the chunks a walker locates must not decrease.
template <int CBT = BT, typename P>
__device__ __forceinline__ Meta locate(const P &p, int32_t c, int32_t h, Walk &w) {
    Meta m{0, 0, h, 0};
    if (p.cu == nullptr) {
        // batch row w.s holds chunks w.cbase .. w.cbase + cpr - 1; the walk moves
        // forward, dividing only when it leaves the row
        if (c - w.cbase >= p.cpr) {
            const int32_t d = (c - w.cbase) / p.cpr;
            w.s += d;
            w.cbase += d * p.cpr;
        }
        const int32_t b = w.s;
        const int32_t cc = c - w.cbase;
        const int64_t t0 = int64_t(cc) * CBT;
        m.row0 = static_cast<int32_t>(int64_t(b) * p.T + t0);
        const int64_t left = p.T - t0;
        m.n = static_cast<int32_t>(left < CBT ? left : CBT);
        m.valid = 1;
        return m;
    }
    // advance to the request that holds chunk c (p.cu may point to global or
    // shared memory: generic loads)
    while (w.s < p.nseq) {
        const int32_t a = p.cu[w.s], b = p.cu[w.s + 1];
        const int32_t nc = nchunks<CBT>(a, b);
        if (c < w.cbase + nc) {
            int64_t r0 = int64_t(a) + int64_t(c - w.cbase) * CBT;
            int64_t end = b < p.T ? b : p.T;                  // clamp malformed cu_seqlens
            if (r0 < 0) r0 = 0;
            int64_t n = end - r0;
            if (n > CBT) n = CBT;
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

// Chunk-heads q = q0, q0 + step, ... of one walker: chunk c = q / H and head
// h = q % H advanced incrementally (two divisions at the start only).
struct TaskWalk {
    int32_t q, c, h, step, sc, sh;
    Walk w;
    template <typename P>
    __device__ __forceinline__ TaskWalk(const P &p, int32_t q0, int32_t step_) : q(q0), step(step_), w{0, 0} {
        c = q0 / p.H;
        h = q0 - c * p.H;
        sc = step_ / p.H;
        sh = step_ - sc * p.H;
    }
    // meta of the current chunk-head (q returned in *qout), then advance
    template <int CBT = BT, typename P>
    __device__ __forceinline__ Meta next(const P &p, int32_t *qout = nullptr) {
        const Meta m = q < p.n_tasks ? locate<CBT>(p, c, h, w) : Meta{0, 0, 0, 0};
        if (qout != nullptr) *qout = q;
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

// Issue the loads of the walker's next task into stage `st` (one thread).
template <int MODE, typename TIn>
__device__ __forceinline__ void issue(const Params &p, const CUtensorMap *maps, TaskWalk &walk,
                                      unsigned char *smem, int st) {
    using L = Layout<MODE, TIn>;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR) + st;
    Meta *meta = reinterpret_cast<Meta *>(smem + L::OFF_META) + st;
    int32_t q;
    const Meta m = walk.next(p, &q);
    *meta = m;
    if (!m.valid) {
        mbar_arrive(bar);
        return;
    }
    unsigned char *stage = smem + L::OFF_STAGE + st * L::STAGE_BYTES;
    mbar_arrive_expect_tx(bar, L::TX_BYTES);
    if (MODE == MODE_FUSED) {                // maps[4]: 32 x 32 box, maps[5]: 64 x 32 box
        tma_load_3d(stage, &maps[4], 0, m.h, m.row0, bar);
        tma_load_3d(stage + L::row_off(2), &maps[5], 0, m.h, m.row0 + 32, bar);
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
// 16-bit input: the four diagonal blocks widened to FP32 tiles (pitch 16);
// rows at or past n become exact zeros (they may hold the next request's rows).
template <int MODE, typename TIn>
__device__ __forceinline__ void widen_diag(const unsigned char *stage, float *Af, int n, int tid) {
    using L = Layout<MODE, TIn>;
    constexpr int VEC = Elt<TIn>::VEC;       // 8 elements per 16-byte vector
#pragma unroll
    for (int v = 0; v < 4 * 16 * 16 / VEC / NTHREADS; ++v) {
        const int e = tid + NTHREADS * v;    // vector index over the four blocks
        const int b = e >> 5, i = (e >> 1) & 15, k = 8 * (e & 1);
        const TIn *src = reinterpret_cast<const TIn *>(stage + L::row_off(b)) + i * L::width(b) +
                         (MODE == MODE_DIAG ? 0 : 16 * b) + k;
        const uint4 raw = *reinterpret_cast<const uint4 *>(src);
        float f[VEC];
        Elt<TIn>::widen(raw, f);
        const bool keep = 16 * b + i < n;
        float *row = Af + b * ABS + i * AP16;
        *reinterpret_cast<float4 *>(row + 4 * ((k >> 2) ^ af_swz(i))) =
            keep ? make_float4(f[0], f[1], f[2], f[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(row + 4 * (((k >> 2) + 1) ^ af_swz(i))) =
            keep ? make_float4(f[4], f[5], f[6], f[7]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// A partial chunk: zero the rows at or past n in the landing buffer (they may
// hold the next request's rows, and a zero times a non-finite value is not zero).
template <int MODE, typename TIn>
__device__ __forceinline__ void zero_rows(unsigned char *stage, int n, int tid) {
    using L = Layout<MODE, TIn>;
    constexpr int VEC = 16 / int(sizeof(TIn));
#pragma unroll
    for (int r = L::R0; r < 4; ++r) {
        const int wv = L::width(r) / VEC;    // 16-byte vectors per row
        uint4 *base = reinterpret_cast<uint4 *>(stage + L::row_off(r));
        for (int e = tid; e < 16 * wv; e += NTHREADS) {
            const int i = e / wv;
            if (16 * r + i >= n) base[e] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// ------------------------------------------------------ diagonal inverse
// Unit-lower-triangular 16x16 inverse by forward substitution, one lane per
// column j: x[i] = [i == j] + sum_{k<i} (-a[i][k]) x[k].  Rows above j need no
// select: every x[k] with k < j is +0, so they come out as exact zeros and x[j]
// as exactly 1, and the rows below j take the same FMAs in the same order.
// SELECT = true keeps the rows at or above j by a select instead: the same
// values for finite a, with fewer registers live.  The 32-token kernel uses it
// (without it, it spills within its 96 registers), and so do the fused
// construction kernel's solve warps (3 % faster with it on GB300, among 16
// warps of 128 registers).  Only entries of `a` (pitch ap) with k < i are used.
template <bool SELECT = false, bool SWZ = false>
__device__ __forceinline__ void diag_invert(const float *a, int ap, int j, float (&x)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
        float s = SELECT ? 0.f : x[i];
#pragma unroll
        for (int kq = 0; kq < (i + 3) / 4; ++kq) {
            const float4 v = *reinterpret_cast<const float4 *>(a + i * ap + 4 * (SWZ ? (kq ^ af_swz(i)) : kq));
            if (4 * kq + 0 < i) s = fmaf(-v.x, x[4 * kq + 0], s);
            if (4 * kq + 1 < i) s = fmaf(-v.y, x[4 * kq + 1], s);
            if (4 * kq + 2 < i) s = fmaf(-v.z, x[4 * kq + 2], s);
            if (4 * kq + 3 < i) s = fmaf(-v.w, x[4 * kq + 3], s);
        }
        x[i] = SELECT ? ((i > j) ? s : x[i]) : s;
    }
}

// ------------------------------------------------------ tensor-core products
// 16x16x16 products on mma.sync m16n8k8 (TF32 in, FP32 accumulate) in split
// precision: an FP32 operand x = hi + lo with hi = x truncated to TF32 and lo =
// (x - hi) truncated to TF32, and P Q ~ Pl Qh + Ph Ql + Ph Qh (the dropped Pl Ql
// is ~2^-22 relative).  Operands exact in TF32 (widened bf16 / fp16 input) skip
// their lo term.
//
// m16n8k8 fragments (lane = 4 g + t): A a0 = A[g][s], a1 = A[g+8][s], a2 =
// A[g][s'], a3 = A[g+8][s']; B b0 = B[s][n], b1 = B[s'][n] with n = g; C c0 =
// C[g][2t], c1 = C[g][2t+1], c2 = C[g+8][2t], c3 = C[g+8][2t+1]; s, s' are the
// k-slots t, t+4.  The contraction index a k-slot stands for is free as long as
// A and B agree; two assignments are used:
//   kperm4: k-step 0 slots -> k = 4t, 4t+1; k-step 1 -> 4t+2, 4t+3
//           (left operand read with one 16-byte load per fragment row)
//   kperm2: k-step 0 slots -> k = 2t, 2t+1; k-step 1 -> 8+2t, 9+2t
//           (left operand taken from a previous product's C fragments)
struct TileA { uint32_t h[2][4], l[2][4]; };      // [k-step][a0..a3]
struct TileB { uint32_t h[2][2][2], l[2][2][2]; };  // [k-step][n-tile][b0, b1]
struct TileC { float c[2][4]; };                   // [n-tile][c0..c3]

__device__ __forceinline__ void split_tf32(float v, uint32_t &h, uint32_t &l) {
    const uint32_t b = __float_as_uint(v) & 0xffffe000u;
    h = b;
    l = __float_as_uint(v - __uint_as_float(b)) & 0xffffe000u;
}

__device__ __forceinline__ void mma8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void zero(TileC &c) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) c.c[nt][i] = 0.f;
}

// Left operand (kperm4): row-major 16x16 tile at p with pitch lp.  SWZ: the
// tile's 16-byte chunks are stored swizzled, chunk c of row r at c ^ xt_swz(r)
// (rows g and g + 8 share the swizzle).
template <bool SWZ = false>
__device__ __forceinline__ void left_smem(TileA &a, const float *p, int lp, int g, int t) {
    float4 r0, r1;
    if (SWZ) {
        const int tc = 4 * (t ^ xt_swz(g));
        r0 = *reinterpret_cast<const float4 *>(p + g * lp + tc);
        r1 = *reinterpret_cast<const float4 *>(p + (g + 8) * lp + tc);
    } else {
        r0 = *reinterpret_cast<const float4 *>(p + g * lp + 4 * t);
        r1 = *reinterpret_cast<const float4 *>(p + (g + 8) * lp + 4 * t);
    }
    split_tf32(r0.x, a.h[0][0], a.l[0][0]); split_tf32(r1.x, a.h[0][1], a.l[0][1]);
    split_tf32(r0.y, a.h[0][2], a.l[0][2]); split_tf32(r1.y, a.h[0][3], a.l[0][3]);
    split_tf32(r0.z, a.h[1][0], a.l[1][0]); split_tf32(r1.z, a.h[1][1], a.l[1][1]);
    split_tf32(r0.w, a.h[1][2], a.l[1][2]); split_tf32(r1.w, a.h[1][3], a.l[1][3]);
}

// Left operand (kperm2): the C fragments of a previous 16x16 product.
__device__ __forceinline__ void left_regs(TileA &a, const TileC &c) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        split_tf32(c.c[ks][0], a.h[ks][0], a.l[ks][0]);
        split_tf32(c.c[ks][2], a.h[ks][1], a.l[ks][1]);
        split_tf32(c.c[ks][1], a.h[ks][2], a.l[ks][2]);
        split_tf32(c.c[ks][3], a.h[ks][3], a.l[ks][3]);
    }
}

// Right operand Q = R^T (kperm4) for row-major R at r with pitch rp; EXACT: R
// holds TF32-exact values (no lo part).
template <bool EXACT>
__device__ __forceinline__ void right4(TileB &b, const float *r, int rp, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const float4 v = *reinterpret_cast<const float4 *>(r + (8 * nt + g) * rp + 4 * t);
        if (EXACT) {
            b.h[0][nt][0] = __float_as_uint(v.x); b.h[0][nt][1] = __float_as_uint(v.y);
            b.h[1][nt][0] = __float_as_uint(v.z); b.h[1][nt][1] = __float_as_uint(v.w);
        } else {
            split_tf32(v.x, b.h[0][nt][0], b.l[0][nt][0]); split_tf32(v.y, b.h[0][nt][1], b.l[0][nt][1]);
            split_tf32(v.z, b.h[1][nt][0], b.l[1][nt][0]); split_tf32(v.w, b.h[1][nt][1], b.l[1][nt][1]);
        }
    }
}

// Right operand Q = R^T (kperm4) for a row-major A block in the input dtype.
__device__ __forceinline__ void right4a(TileB &b, const float *r, int rp, int g, int t) {
    right4<false>(b, r, rp, g, t);
}
__device__ __forceinline__ void right4a(TileB &b, const __nv_bfloat16 *r, int rp, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {        // bf16 -> fp32 is exact (and exact in TF32)
        const uint2 v = *reinterpret_cast<const uint2 *>(r + (8 * nt + g) * rp + 4 * t);
        b.h[0][nt][0] = v.x << 16; b.h[0][nt][1] = v.x & 0xffff0000u;
        b.h[1][nt][0] = v.y << 16; b.h[1][nt][1] = v.y & 0xffff0000u;
    }
}
__device__ __forceinline__ void right4a(TileB &b, const __half *r, int rp, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {        // fp16 -> fp32 is exact (and exact in TF32)
        const uint2 v = *reinterpret_cast<const uint2 *>(r + (8 * nt + g) * rp + 4 * t);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
        b.h[0][nt][0] = __float_as_uint(f0.x); b.h[0][nt][1] = __float_as_uint(f0.y);
        b.h[1][nt][0] = __float_as_uint(f1.x); b.h[1][nt][1] = __float_as_uint(f1.y);
    }
}

// Right operand Q = R^T (kperm2) for row-major R at r with pitch rp.
__device__ __forceinline__ void right2(TileB &b, const float *r, int rp, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const float2 v = *reinterpret_cast<const float2 *>(r + (8 * nt + g) * rp + 8 * ks + 2 * t);
            split_tf32(v.x, b.h[ks][nt][0], b.l[ks][nt][0]);
            split_tf32(v.y, b.h[ks][nt][1], b.l[ks][nt][1]);
        }
}

// c += P Q in split TF32 (B_EXACT: Q has no lo part).  TF32: the precision mode
// that takes P Q as one TF32 product (Ph Qh; the lo parts are not used).
template <bool B_EXACT, bool TF32 = false>
__device__ __forceinline__ void mma_tile(TileC &c, const TileA &a, const TileB &b) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (!TF32) mma8(c.c[nt], a.l[ks], b.h[ks][nt][0], b.h[ks][nt][1]);
            if (!B_EXACT && !TF32) mma8(c.c[nt], a.h[ks], b.l[ks][nt][0], b.l[ks][nt][1]);
            mma8(c.c[nt], a.h[ks], b.h[ks][nt][0], b.h[ks][nt][1]);
        }
}

// c += P Q and d += P R, interleaved (two independent accumulator chains; each
// accumulates in the same order as mma_tile).
template <bool B_EXACT, bool TF32 = false>
__device__ __forceinline__ void mma_tile2(TileC &c, TileC &d, const TileA &a, const TileB &q, const TileB &r) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (!TF32) {
                mma8(c.c[nt], a.l[ks], q.h[ks][nt][0], q.h[ks][nt][1]);
                mma8(d.c[nt], a.l[ks], r.h[ks][nt][0], r.h[ks][nt][1]);
            }
            if (!B_EXACT && !TF32) {
                mma8(c.c[nt], a.h[ks], q.l[ks][nt][0], q.l[ks][nt][1]);
                mma8(d.c[nt], a.h[ks], r.l[ks][nt][0], r.l[ks][nt][1]);
            }
            mma8(c.c[nt], a.h[ks], q.h[ks][nt][0], q.h[ks][nt][1]);
            mma8(d.c[nt], a.h[ks], r.h[ks][nt][0], r.h[ks][nt][1]);
        }
}

// C tile holding Y^T -> output block (bi, bj) of the chunk (rows below n only).
template <int CBT = BT, typename TOut>
__device__ __forceinline__ void out_tile_t(TOut *ob, int os, int n, int bi, int bj, const TileC &c, int g, int t) {
    if (CBT == BT && n == CBT) {             // a full 64-token chunk: no row test
        TOut *base = ob + ((16 * bi + 2 * t) * os + 16 * bj + g);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                TOut *row = base + (8 * nt + e) * os;
                put1(row, c.c[nt][e]);
                put1(row + 8, c.c[nt][2 + e]);
            }
        return;
    }
    const bool full = n == CBT;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 16 * bi + 8 * nt + 2 * t + e;
            if (full || r < n) {
                TOut *row = ob + (r * os + 16 * bj + g);
                put1(row, c.c[nt][e]);
                put1(row + 8, c.c[nt][2 + e]);
            }
        }
}

// C tile holding Y^T -> Y^T row-major (pitch XTP) in shared memory (SWZ: the
// chunks swizzled as left_smem<true> reads them).
template <bool SWZ = false>
__device__ __forceinline__ void smem_tile_t(float *dst, const TileC &c, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        if (SWZ) {
            const int col = 4 * ((2 * nt + (t >> 1)) ^ xt_swz(g)) + 2 * (t & 1);
            *reinterpret_cast<float2 *>(dst + g * XTP + col) = make_float2(c.c[nt][0], c.c[nt][1]);
            *reinterpret_cast<float2 *>(dst + (g + 8) * XTP + col) = make_float2(c.c[nt][2], c.c[nt][3]);
        } else {
            *reinterpret_cast<float2 *>(dst + g * XTP + 8 * nt + 2 * t) = make_float2(c.c[nt][0], c.c[nt][1]);
            *reinterpret_cast<float2 *>(dst + (g + 8) * XTP + 8 * nt + 2 * t) = make_float2(c.c[nt][2], c.c[nt][3]);
        }
    }
}

// C tile holding Y^T -> -Y row-major (pitch XRP) in shared memory.
__device__ __forceinline__ void smem_tile_neg(float *dst, const TileC &c, int g, int t) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 8 * nt + 2 * t + e;
            dst[r * XRP + g] = -c.c[nt][e];
            dst[r * XRP + g + 8] = -c.c[nt][2 + e];
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
    CUtensorMap m[6];          // A: box widths 16, 32, 48, 64 columns x 16 rows (split kernels),
                               // then 32 and 64 columns x 32 rows (single pass); 1 head
};

// CTAs per SM the registers must allow: the single pass on 16-bit input fits
// eight in shared memory (28 KB each), on FP32 input six (36 KB)
template <int MODE, typename TIn>
constexpr int min_ctas() {
    return MODE == MODE_DIAG ? 1 : (MODE == MODE_FUSED && sizeof(TIn) == 2) ? 8 : 6;
}

// TF32 (MODE_FUSED only): the precision mode, merge products in plain TF32.
template <int MODE, typename TIn, typename TOut, bool TF32 = false>
__global__ void __launch_bounds__(NTHREADS, min_ctas<MODE, TIn>())
kda_tril_kernel(const __grid_constant__ Maps maps, const Params p) {
    using L = Layout<MODE, TIn>;
    constexpr bool AX = L::WIDEN;            // A values exact in TF32
    // 16-bit input: the Xt tiles (and the split path's workspace tiles) are
    // swizzled; FP32 input keeps them plain (measured 1.4 % slower swizzled)
    constexpr bool XSW = AX;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    const Meta *metas = reinterpret_cast<const Meta *>(smem + L::OFF_META);
    float *Af = reinterpret_cast<float *>(smem + L::OFF_AF);
    float *Xt = reinterpret_cast<float *>(smem + L::OFF_XT);
    float *Xr = reinterpret_cast<float *>(smem + L::OFF_XR);
    TOut *out = reinterpret_cast<TOut *>(p.out);
    const int tid = threadIdx.x;
    const int unit = tid >> 4, warp = tid >> 5;
    // the thread that issues the loads (and owns the walk): warp 1's first for
    // the single pass on 16-bit input, whose level B gives warp 1 the lighter
    // share (measured 0.5-0.8 % faster there, 2 % slower on FP32 input)
    constexpr int ISSUER = MODE == MODE_FUSED && AX ? 32 : 0;
    pdl_launch_dependents();
    if (tid == ISSUER) {
        // the tensor maps this kernel uses, into the TMA unit's descriptor cache
        if (MODE == MODE_FUSED) {
            prefetch_tensormap(&maps.m[4]);
            prefetch_tensormap(&maps.m[5]);
        } else {
            for (int r = 0; r < 4; ++r) prefetch_tensormap(&maps.m[r]);
        }
        for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    pdl_wait();                              // the previous kernel's writes (A, cu_seqlens) are visible
    // the task walk reads cu_seqlens from shared memory when it fits
    Params ps = p;
    if (p.cu != nullptr && p.nseq < CU_CAP) {
        int32_t *cs = reinterpret_cast<int32_t *>(smem + L::OFF_CU);
        for (int i = tid; i <= p.nseq; i += NTHREADS) cs[i] = __ldg(p.cu + i);
        ps.cu = cs;
        __syncthreads();
    }
    const int l = tid & 15;                  // lane in the 16-lane unit (diagonal inverse)
    const int lane = tid & 31, g = lane >> 2, t = lane & 3;   // mma fragment coordinates
    const int32_t G = gridDim.x;
    const int os = p.H * BT;                 // output row stride (elements)
    TaskWalk walk(p, int32_t(blockIdx.x), G);   // the issuer's walk over the tasks it loads

    if (tid == ISSUER) {
        for (int s = 0; s < STAGES; ++s) issue<MODE, TIn>(ps, maps.m, walk, smem, s);
    }
    __syncthreads();

    for (int it = 0;; ++it) {
        const int st = it % STAGES;
        const uint32_t parity = (it / STAGES) & 1;
        const bool ok = mbar_wait_bounded(&bars[st], parity);
        if (__syncthreads_or(!ok)) {
            // A copy never completed.  Record it, give the copies still in
            // flight a bounded chance to land, and stop.
            if (tid == ISSUER) {
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
        // Every thread is past the previous chunk-head, so the stage it used,
        // (it - 1) % STAGES, is free: refill it with the chunk-head STAGES - 1
        // iterations ahead (the prologue issued iterations 0 .. STAGES - 1).
        if (it >= 1 && tid == ISSUER) {
            fence_proxy_async();
            issue<MODE, TIn>(ps, maps.m, walk, smem, (it + STAGES - 1) % STAGES);
        }
        TOut *ob = out + (int64_t(m.row0) * p.H + m.h) * BT;      // chunk-head's first row

        if (MODE != MODE_MERGE) store_upper_zeros(ob, os, m.n, tid);   // zero blocks above the diagonal

        // A operands: the landing buffer itself (rows past a partial chunk's end
        // zeroed), plus FP32 copies of the diagonal blocks for 16-bit input
        if (m.n < BT) zero_rows<MODE, TIn>(stage, m.n, tid);
        if (L::WIDEN && MODE != MODE_MERGE) widen_diag<MODE, TIn>(stage, Af, m.n, tid);
        // X00^T, X11^T, X22^T: the workspace tile (MODE_MERGE) or the Xt slots
        const float *xt00, *xt11, *xt22;
        if (MODE == MODE_MERGE) {
            // the workspace tile holds X00^T .. X33^T row-major; the negated
            // inverses -X11, -X33, -X22 are transposed out of it
            const float *wt = reinterpret_cast<const float *>(stage + L::WS_OFF);
            xt00 = wt; xt11 = wt + 256; xt22 = wt + 512;
#pragma unroll
            for (int v = 0; v < 3; ++v) {
                const int e = tid + NTHREADS * v;       // float4 index in blocks 1..3
                const int b = 1 + (e >> 6), j = (e >> 2) & 15, i4 = 4 * (e & 3);
                const float4 x = *reinterpret_cast<const float4 *>(wt + b * 256 + j * 16 + (XSW ? 4 * ((e & 3) ^ xt_swz(j)) : i4));
                float *d = Xr + (b == 1 ? XR_11 : b == 3 ? XR_33 : XR_22) * XRS + j;
                d[(i4 + 0) * XRP] = -x.x; d[(i4 + 1) * XRP] = -x.y;
                d[(i4 + 2) * XRP] = -x.z; d[(i4 + 3) * XRP] = -x.w;
            }
        } else {
            xt00 = Xt + XT_00 * XTS; xt11 = Xt + XT_11 * XTS; xt22 = Xt + XT_22 * XTS;
        }
        // TMA data is visible to every thread after its own mbarrier wait; a
        // barrier is needed only when threads rewrote shared memory above.
        if ((L::WIDEN && MODE != MODE_MERGE) || MODE == MODE_MERGE || m.n < BT) __syncthreads();

        if (MODE != MODE_MERGE) {
            // unit u inverts diagonal block u (warp 0: X00, X11; warp 1: X22, X33)
            float x[16];
            const int b = unit;
            const AView a = adiag<MODE, TIn>(stage, Af, b);
            diag_invert<!AX, AX>(a.p, a.pitch, l, x);   // FP32 input: the select form (more registers live there); 16-bit: the widened tiles are swizzled
            TOut *op = ob + (16 * b * os + 16 * b + l);   // diagonal block of the output, lane = column
            if (m.n == BT) {
#pragma unroll
                for (int i = 0; i < 16; ++i, op += os) put1(op, x[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i, op += os)
                    if (16 * b + i < m.n) put1(op, x[i]);
            }
            if (MODE == MODE_DIAG) {         // workspace: X_bb^T row-major, lane = row
                float4 *w = reinterpret_cast<float4 *>(p.ws + size_t(q) * 1024 + b * 256 + l * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i) w[XSW ? i ^ xt_swz(l) : i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
                continue;
            }
            if (b != 3) {                    // X_bb^T row-major (row = lane)
                float4 *d = reinterpret_cast<float4 *>(Xt + (b == 0 ? XT_00 : b == 1 ? XT_11 : XT_22) * XTS + l * XTP);
#pragma unroll
                for (int i = 0; i < 4; ++i) d[XSW ? i ^ xt_swz(l) : i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
            }
            if (b != 0) {                    // -X_bb row-major (column = lane)
                float *d = Xr + (b == 1 ? XR_11 : b == 3 ? XR_33 : XR_22) * XRS + l;
#pragma unroll
                for (int i = 0; i < 16; ++i) d[i * XRP] = -x[i];
            }
            __syncwarp();                    // level A reads only this warp's inverses
        }

        // ---- level A (warp 0: X10, warp 1: X32), computed transposed:
        //   T_A^T = X00^T A10^T,  X10^T = T_A^T (-X11)^T
        //   T_B^T = X22^T A32^T,  X32^T = T_B^T (-X33)^T
        {
            TileA la;
            TileB rb;
            TileC c1, c2;
            const AOff<TIn> a = warp == 0 ? aoff<MODE, TIn>(stage, 1, 0) : aoff<MODE, TIn>(stage, 3, 2);
            left_smem<XSW>(la, warp == 0 ? xt00 : xt22, XTP, g, t);
            right4a(rb, a.p, a.pitch, g, t);
            zero(c1);
            mma_tile<AX, TF32>(c1, la, rb);
            left_regs(la, c1);
            right2(rb, Xr + (warp == 0 ? XR_11 : XR_33) * XRS, XRP, g, t);
            zero(c2);
            mma_tile<false, TF32>(c2, la, rb);
            if (warp == 0) {
                smem_tile_t<XSW>(Xt + XT_10 * XTS, c2, g, t);
                out_tile_t(ob, os, m.n, 1, 0, c2, g, t);
            } else {
                smem_tile_neg(Xr + XR_32 * XRS, c2, g, t);
                out_tile_t(ob, os, m.n, 3, 2, c2, g, t);
            }
        }
        __syncthreads();

        // ---- level B, warp w = column block j of X_BL (w = 0: X20, X30; w = 1: X21, X31):
        //   T_2w^T = X_TL(:, w)^T A_BL(0, :)^T,  T_3w^T = X_TL(:, w)^T A_BL(1, :)^T
        //   X_2w^T = T_2w^T (-X22)^T,  X_3w^T = T_2w^T (-X32)^T + T_3w^T (-X33)^T
        {
            TileA la, lb;
            TileB rb;
            TileC ct2, ct3, cx;
            zero(ct2);
            zero(ct3);
            left_smem<XSW>(la, warp == 0 ? xt00 : xt11, XTP, g, t);   // X00^T | X11^T
            {
                const AOff<TIn> a2 = aoff<MODE, TIn>(stage, 2, warp), a3 = aoff<MODE, TIn>(stage, 3, warp);
                right4a(rb, a2.p, a2.pitch, g, t);
                mma_tile<AX, TF32>(ct2, la, rb);
                right4a(rb, a3.p, a3.pitch, g, t);
                mma_tile<AX, TF32>(ct3, la, rb);
            }
            if (warp == 0) {                 // + X10^T A21^T, X10^T A31^T
                left_smem<XSW>(la, Xt + XT_10 * XTS, XTP, g, t);
                const AOff<TIn> a2 = aoff<MODE, TIn>(stage, 2, 1), a3 = aoff<MODE, TIn>(stage, 3, 1);
                right4a(rb, a2.p, a2.pitch, g, t);
                mma_tile<AX, TF32>(ct2, la, rb);
                right4a(rb, a3.p, a3.pitch, g, t);
                mma_tile<AX, TF32>(ct3, la, rb);
            }
            // X_2w^T = T_2w^T (-X22)^T and the first term of X_3w^T, T_2w^T (-X32)^T,
            // as two interleaved chains; then + T_3w^T (-X33)^T
            left_regs(la, ct2);
            left_regs(lb, ct3);
            TileB rb3;
            TileC cy;
            right2(rb, Xr + XR_22 * XRS, XRP, g, t);
            right2(rb3, Xr + XR_32 * XRS, XRP, g, t);
            zero(cx);
            zero(cy);
            mma_tile2<false, TF32>(cx, cy, la, rb, rb3);
            out_tile_t(ob, os, m.n, 2, warp, cx, g, t);
            right2(rb, Xr + XR_33 * XRS, XRP, g, t);
            mma_tile<false, TF32>(cy, lb, rb);
            out_tile_t(ob, os, m.n, 3, warp, cy, g, t);
        }
    }
}

// ------------------------------------------------------- named barriers
// Named barriers of 64 threads (one pair of warps) with the barrier id in a
// register, so that every pair runs the same code (one copy of the solve in
// the instruction cache, whatever the number of pairs).
__device__ __forceinline__ bool bar64_and(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, 64, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(v)), "r"(id)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void bar64(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

}  // namespace kda
