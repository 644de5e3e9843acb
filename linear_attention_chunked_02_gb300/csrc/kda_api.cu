// kda_api.cu -- C ABI of the KDA prefill chunk solver: argument checks, the
// split / single-pass selector, TMA descriptors and kernel dispatch.
//
// The selector follows LightLLM PR #1703 (PR description and summary): the
// split path is taken only when an FP32 workspace no larger than the FP32
// input fits the caller's budget and the input is long enough, i.e. the choice
// rests on how full the chunks are -- the workspace is 4 KiB per chunk-head and the
// FP32 input is 256 B per row and head, so the budget holds exactly when
// chunks are on average at least 16 rows full.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kda_internal.h"
#include "kda_launch.cuh"
#include "kda_solve_tril.h"

namespace {

__device__ unsigned g_kda_err;   // device-side error word, one per device

// Self-test of the kernels' failure detection (one thread): an mbarrier that
// expects one arrival and gets it only when `complete` is set.  The bounded wait
// must then succeed; otherwise it gives up after limit_ns and the kernel records
// ERR_WAIT_TIMEOUT in the error word and returns, as the solver kernels do.
__global__ void kda_wait_selftest_kernel(unsigned *err, int complete, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    kda::mbar_init(&bar, 1);
    kda::fence_mbar_init();
    if (complete) kda::mbar_arrive(&bar);
    if (!kda::mbar_wait_bounded(&bar, 0, limit_ns)) atomicOr(err, kda::ERR_WAIT_TIMEOUT);
}

constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1 - 2 * kda::BT;

int elt_size(int32_t dt) { return dt == KDA_F32 ? 4 : 2; }
bool dtype_ok(int32_t dt) { return dt == KDA_F32 || dt == KDA_BF16 || dt == KDA_F16; }

// Upper bound on the number of chunks of length bt that needs no look at cu_seqlens.
int64_t max_chunks(int64_t B, int64_t T, int32_t num_seqs, int bt = kda::BT) {
    if (B <= 0 || T <= 0) return 0;
    if (num_seqs <= 0) return B * ((T + bt - 1) / bt);
    const int64_t bound = (T + int64_t(bt - 1) * num_seqs) / bt;
    return bound < T ? bound : T;
}

struct DeviceInfo {
    int num_sms = 0;
    unsigned *err = nullptr;
};

cudaError_t device_info(int device, DeviceInfo &out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device].num_sms == 0) {
        int sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e != cudaSuccess) return e;
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_kda_err);
        if (e != cudaSuccess) return e;
        cache[device].err = static_cast<unsigned *>(ptr);
        cache[device].num_sms = sms;
    }
    out = cache[device];
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A tensor [rows, H, 64] viewed as 3-D {64 columns, H heads, rows}, with boxes of
// {width[w] columns, 1 head, box_rows rows} for w = 0 .. n-1.
bool encode_maps(const void *base, int32_t dt, int32_t H, int64_t rows, CUtensorMap *maps, const int *width, int n,
                 int box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const CUtensorMapDataType ty = dt == KDA_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dt == KDA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t es = cuuint64_t(elt_size(dt));
    const cuuint64_t dims[3] = {cuuint64_t(kda::BT), cuuint64_t(H), cuuint64_t(rows)};
    const cuuint64_t strides[2] = {kda::BT * es, cuuint64_t(H) * kda::BT * es};
    const cuuint32_t estr[3] = {1, 1, 1};
    for (int w = 0; w < n; ++w) {
        const cuuint32_t box[3] = {cuuint32_t(width[w]), 1, cuuint32_t(box_rows)};
        CUresult r = fn(&maps[w], ty, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return false;
    }
    return true;
}

// Input boxes of A: 16 rows x 16, 32, 48, 64 columns (the split kernels' block
// rows), then 32 rows x 32 and 64 columns (the single pass's two boxes).
bool make_maps(const void *A, int32_t in_dt, void *, int32_t, int32_t H, int64_t rows, kda::Maps &maps) {
    static const int w16[4] = {16, 32, 48, 64}, w32[2] = {32, 64};
    return encode_maps(A, in_dt, H, rows, maps.m, w16, 4, 16) && encode_maps(A, in_dt, H, rows, maps.m + 4, w32, 2, 32);
}

// Encoded tensor maps of recent calls, keyed by everything they encode (base
// addresses, dtypes, H, rows): a map is a pure function of its key, so a hit is
// exact even if the caller's buffers were freed and reallocated meanwhile.
// Saves the seven encodings on the host for repeated solves on the same buffers.
struct MapKey {
    const void *A, *Ai;
    int32_t in_dt, out_dt, H;
    int64_t rows;
    bool operator==(const MapKey &o) const {
        return A == o.A && Ai == o.Ai && in_dt == o.in_dt && out_dt == o.out_dt && H == o.H && rows == o.rows;
    }
};
constexpr int kMapCache = 16;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
kda::Maps g_map_val[kMapCache];
int g_map_n = 0, g_map_next = 0;

bool cached_maps(const void *A, int32_t in_dt, void *Ai, int32_t out_dt, int32_t H, int64_t rows, kda::Maps &maps) {
    const MapKey key{A, Ai, in_dt, out_dt, H, rows};
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_map_n; ++i)
        if (g_map_key[i] == key) {
            maps = g_map_val[i];
            return true;
        }
    std::memset(&maps, 0, sizeof(maps));
    if (!make_maps(A, in_dt, Ai, out_dt, H, rows, maps)) return false;
    g_map_key[g_map_next] = key;
    g_map_val[g_map_next] = maps;
    g_map_next = (g_map_next + 1) % kMapCache;
    if (g_map_n < kMapCache) ++g_map_n;
    return true;
}

// k [rows, H, K] (input dtype) and g [rows, H, K] (FP32) viewed as 3-D {K
// channels, H heads, rows}, boxes of 32 channels x 1 head x 64 rows.
bool encode_kg_maps(const void *k, int32_t in_dt, const float *g, int32_t H, int32_t K, int64_t rows,
                    kda::KgbMaps &maps) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint32_t box[3] = {32, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    for (int t = 0; t < 2; ++t) {
        const int32_t dt = t == 0 ? in_dt : KDA_F32;
        const CUtensorMapDataType ty = dt == KDA_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : dt == KDA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const cuuint64_t es = cuuint64_t(elt_size(dt));
        const cuuint64_t dims[3] = {cuuint64_t(K), cuuint64_t(H), cuuint64_t(rows)};
        const cuuint64_t strides[2] = {cuuint64_t(K) * es, cuuint64_t(H) * cuuint64_t(K) * es};
        CUresult r = fn(t == 0 ? &maps.k : &maps.g, ty, 3, const_cast<void *>(t == 0 ? k : static_cast<const void *>(g)),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return false;
    }
    return true;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t dispatch(int mode, int32_t in_dt, int32_t out_dt, const kda::Maps &maps, const kda::Params &p,
                     int device, int sms, cudaStream_t s) {
    switch (in_dt) {
        case KDA_F32: return kda::launch_f32(mode, out_dt, maps, p, device, sms, s);
        case KDA_BF16: return kda::launch_bf16(mode, out_dt, maps, p, device, sms, s);
        default: return kda::launch_f16(mode, out_dt, maps, p, device, sms, s);
    }
}

// Host-side checks shared by every entry point.  Returns KDA_OK or an error.
kda_status_t check_args(const void *A, const void *Ai, const int32_t *cu, int32_t num_seqs, int64_t B,
                        int64_t T, int32_t H, int32_t in_dt, int32_t out_dt, int bt = kda::BT) {
    if (!dtype_ok(in_dt) || !dtype_ok(out_dt)) return KDA_ERR_UNSUPPORTED;
    if (H < 1 || B < 0 || T < 0 || num_seqs < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (int64_t(H) * bt * bt > INT32_MAX) return KDA_ERR_UNSUPPORTED;   // in-chunk offsets are 32-bit
    if ((cu != nullptr) != (num_seqs > 0)) return KDA_ERR_INVALID_ARGUMENT;
    if (cu != nullptr && B != 1) return KDA_ERR_INVALID_ARGUMENT;
    if (B == 0 || T == 0) return KDA_OK;
    if (A == nullptr || Ai == nullptr) return KDA_ERR_INVALID_ARGUMENT;
    if (T > kMaxRows || B > kMaxRows / T) return KDA_ERR_UNSUPPORTED;
    if (max_chunks(B, T, num_seqs, bt) * H > INT32_MAX / 2) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

// Copy streams of the end-to-end entry point, created once per device.
constexpr int kMaxPieces = 8;
constexpr size_t kPieceBytes = size_t(16) << 20;   // at least 16 MiB of copies per piece
struct CopyEngines {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[2 + 2 * kMaxPieces] = {};
    bool ready = false;
};
std::mutex g_copy_mu;
CopyEngines g_copy[64];

// With g_copy_mu held and `device` current.
cudaError_t copy_engines(int device, CopyEngines *&ce) {
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    CopyEngines &c = g_copy[device];
    if (!c.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking);
        for (int i = 0; e == cudaSuccess && i < 2 + 2 * kMaxPieces; ++i)
            e = cudaEventCreateWithFlags(&c.ev[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        c.ready = true;
    }
    ce = &c;
    return cudaSuccess;
}

}  // namespace

namespace kda {

kda_status_t validate_solve(const void *A, const void *Ai, const int32_t *cu, int32_t num_seqs, int64_t B,
                            int64_t T, int32_t H, int32_t in_dt, int32_t out_dt) {
    const kda_status_t st = check_args(A, Ai, cu, num_seqs, B, T, H, in_dt, out_dt);
    if (st != KDA_OK || B == 0 || T == 0) return st;
    const size_t elems = size_t(B) * size_t(T) * size_t(H) * BT;
    if (!aligned16(A) || !aligned16(Ai)) return KDA_ERR_INVALID_ARGUMENT;
    if (overlaps(A, elems * elt_size(in_dt), Ai, elems * elt_size(out_dt))) return KDA_ERR_INVALID_ARGUMENT;
    return KDA_OK;
}

}  // namespace kda

extern "C" {

size_t kda_solve_tril_workspace_size(int64_t B, int64_t T, int32_t H, int32_t num_seqs) {
    if (H < 1 || num_seqs < 0) return 0;
    if (num_seqs > 0 && B != 1) return 0;
    const int64_t nc = max_chunks(B, T, num_seqs);
    return size_t(nc) * size_t(H) * KDA_WS_TILE_BYTES;
}

kda_path_t kda_solve_tril_select(int64_t B, int64_t T, int32_t H, int32_t num_seqs, size_t workspace_bytes) {
    const size_t need = kda_solve_tril_workspace_size(B, T, H, num_seqs);
    if (need == 0 || workspace_bytes < need) return KDA_PATH_SINGLE;
    const size_t fp32_input = size_t(B) * size_t(T) * size_t(H) * kda::BT * 4;
    if (need > fp32_input) return KDA_PATH_SINGLE;
    if (B * T < KDA_SPLIT_MIN_TOKENS) return KDA_PATH_SINGLE;
    return KDA_PATH_SPLIT;
}

// kda_solve_tril_ex with a precision mode (the TF32 mode exists for the single pass only)
static kda_status_t solve_impl(const void *A, void *Ai, const int32_t *cu_seqlens, int32_t num_seqs, int64_t B, int64_t T,
                        int32_t H, int32_t in_dtype, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                        void *stream, int32_t path, int32_t precision, int32_t *path_taken) {
    if (path != KDA_PATH_AUTO && path != KDA_PATH_SPLIT && path != KDA_PATH_SINGLE)
        return KDA_ERR_INVALID_ARGUMENT;
    if (precision != KDA_PREC_IEEE && precision != KDA_PREC_TF32) return KDA_ERR_INVALID_ARGUMENT;
    if (precision == KDA_PREC_TF32 && path != KDA_PATH_SINGLE) return KDA_ERR_INVALID_ARGUMENT;
    kda_status_t st = check_args(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype);
    if (st != KDA_OK) return st;
    const size_t need = kda_solve_tril_workspace_size(B, T, H, num_seqs);
    const size_t have = workspace != nullptr ? workspace_bytes : 0;
    int32_t taken = KDA_PATH_SINGLE;
    if (path == KDA_PATH_SPLIT) {
        if (need > 0 && have < need) return KDA_ERR_WORKSPACE;
        taken = KDA_PATH_SPLIT;
    } else if (path == KDA_PATH_AUTO) {
        taken = kda_solve_tril_select(B, T, H, num_seqs, have);
    }
    if (path_taken != nullptr) *path_taken = taken;
    if (B == 0 || T == 0) return KDA_OK;
    const size_t elems = size_t(B) * size_t(T) * size_t(H) * kda::BT;
    if (!aligned16(A) || !aligned16(Ai)) return KDA_ERR_INVALID_ARGUMENT;
    if (overlaps(A, elems * elt_size(in_dtype), Ai, elems * elt_size(out_dtype))) return KDA_ERR_INVALID_ARGUMENT;
    if (taken == KDA_PATH_SPLIT) {
        if (!aligned16(workspace)) return KDA_ERR_INVALID_ARGUMENT;
        if (overlaps(workspace, need, A, elems * elt_size(in_dtype)) ||
            overlaps(workspace, need, Ai, elems * elt_size(out_dtype)))
            return KDA_ERR_INVALID_ARGUMENT;
    }

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    DeviceInfo info;
    if (device_info(device, info) != cudaSuccess) return KDA_ERR_CUDA;

    kda::Maps maps;
    const int64_t rows = B * T;
    if (!cached_maps(A, in_dtype, Ai, out_dtype, H, rows, maps)) return KDA_ERR_CUDA;

    kda::Params p;
    p.out = Ai;
    p.ws = static_cast<float *>(workspace);
    p.cu = cu_seqlens;
    p.nseq = num_seqs;
    p.H = H;
    p.T = T;
    p.rows = rows;
    p.cpr = static_cast<int32_t>((T + kda::BT - 1) / kda::BT);
    p.n_tasks = static_cast<int32_t>(max_chunks(B, T, num_seqs) * H);
    p.err = info.err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    cudaError_t e;
    if (taken == KDA_PATH_SPLIT) {
        e = dispatch(kda::MODE_DIAG, in_dtype, out_dtype, maps, p, device, info.num_sms, s);
        if (e == cudaSuccess) e = dispatch(kda::MODE_MERGE, in_dtype, out_dtype, maps, p, device, info.num_sms, s);
    } else {
        e = dispatch(precision == KDA_PREC_TF32 ? kda::MODE_FUSED_TF32 : kda::MODE_FUSED, in_dtype, out_dtype, maps,
                     p, device, info.num_sms, s);
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_solve_tril_ex(const void *A, void *Ai, const int32_t *cu_seqlens, int32_t num_seqs, int64_t B,
                               int64_t T, int32_t H, int32_t in_dtype, int32_t out_dtype, void *workspace,
                               size_t workspace_bytes, void *stream, int32_t path, int32_t *path_taken) {
    return solve_impl(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype, workspace, workspace_bytes, stream,
                      path, KDA_PREC_IEEE, path_taken);
}

kda_status_t kda_solve_tril_prec(const void *A, void *Ai, const int32_t *cu_seqlens, int32_t num_seqs, int64_t B,
                                 int64_t T, int32_t H, int32_t in_dtype, int32_t out_dtype, int32_t precision,
                                 void *stream) {
    return solve_impl(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype, nullptr, 0, stream,
                      KDA_PATH_SINGLE, precision, nullptr);
}

kda_status_t kda_solve_tril(const void *A, void *Ai, const int32_t *cu_seqlens, int32_t num_seqs, int64_t B,
                            int64_t T, int32_t H, int32_t in_dtype, int32_t out_dtype, void *workspace,
                            size_t workspace_bytes, void *stream) {
    return kda_solve_tril_ex(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype, workspace,
                             workspace_bytes, stream, KDA_PATH_AUTO, nullptr);
}

kda_status_t kda_solve_tril_host(const void *A_host, void *Ai_host, const int32_t *cu_seqlens_host,
                                 int32_t num_seqs, int64_t B, int64_t T, int32_t H, int32_t in_dtype,
                                 int32_t out_dtype, void *A_dev, void *Ai_dev, int32_t *cu_dev, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    if ((cu_seqlens_host == nullptr) != (cu_dev == nullptr)) return KDA_ERR_INVALID_ARGUMENT;
    kda_status_t st = check_args(A_dev, Ai_dev, cu_dev, num_seqs, B, T, H, in_dtype, out_dtype);
    if (st != KDA_OK) return st;
    if (B == 0 || T == 0) return KDA_OK;
    if (A_host == nullptr || Ai_host == nullptr) return KDA_ERR_INVALID_ARGUMENT;
    const size_t row_in = size_t(H) * kda::BT * elt_size(in_dtype);     // bytes per row of A
    const size_t row_out = size_t(H) * kda::BT * elt_size(out_dtype);   // bytes per row of Ai
    const int64_t rows = B * T;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // Pieces cut at chunk boundaries: whole batch rows, 64-row multiples of a
    // batch row, or whole requests; each solved as its own sub-problem.
    struct Piece { int64_t r0, r1, b, t0, nb, nt; int32_t s0, ns; };
    Piece pc[kMaxPieces];
    int np = 0;
    const size_t total = size_t(rows) * (row_in + row_out);
    const int want = int(std::min<size_t>(kMaxPieces, std::max<size_t>(1, total / kPieceBytes)));
    if (want > 1 && cu_dev == nullptr && B >= want) {
        for (int k = 0; k < want; ++k) {
            const int64_t b0 = B * k / want, b1 = B * (k + 1) / want;
            if (b1 > b0) pc[np++] = {b0 * T, b1 * T, b0, 0, b1 - b0, T, 0, 0};
        }
    } else if (want > 1 && cu_dev == nullptr) {
        const int per = std::max(1, want / int(B));                   // pieces per batch row, B * per <= want
        const int64_t chunks = (T + kda::BT - 1) / kda::BT;
        for (int64_t b = 0; b < B; ++b)
            for (int k = 0; k < per; ++k) {
                const int64_t t0 = std::min(T, chunks * k / per * kda::BT);
                const int64_t t1 = std::min(T, chunks * (k + 1) / per * kda::BT);
                if (t1 > t0) pc[np++] = {b * T + t0, b * T + t1, b, t0, 1, t1 - t0, 0, 0};
            }
    } else if (want > 1) {
        int32_t s0 = 0;
        for (int k = 0; k < want && s0 < num_seqs; ++k) {
            const int64_t goal = rows * (k + 1) / want;              // rows covered after this piece
            int32_t s1 = s0 + 1;
            while (s1 < num_seqs && cu_seqlens_host[s1] < goal) ++s1;
            if (k == want - 1) s1 = num_seqs;
            pc[np++] = {cu_seqlens_host[s0], cu_seqlens_host[s1], 0, 0, 1, T, s0, s1 - s0};
            s0 = s1;
        }
    }

    if (np <= 1) {                           // one piece: everything on the caller's stream
        if (cudaMemcpyAsync(A_dev, A_host, size_t(rows) * row_in, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (cu_dev != nullptr &&
            cudaMemcpyAsync(cu_dev, cu_seqlens_host, sizeof(int32_t) * size_t(num_seqs + 1),
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return KDA_ERR_CUDA;
        st = kda_solve_tril(A_dev, Ai_dev, cu_dev, num_seqs, B, T, H, in_dtype, out_dtype, workspace,
                            workspace_bytes, stream);
        if (st != KDA_OK) return st;
        if (cudaMemcpyAsync(Ai_host, Ai_dev, size_t(rows) * row_out, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return KDA_ERR_CUDA;
        return KDA_OK;
    }

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_copy_mu);
    CopyEngines *ce = nullptr;
    if (copy_engines(device, ce) != cudaSuccess) return KDA_ERR_CUDA;
    const char *ah = static_cast<const char *>(A_host);
    char *ad = static_cast<char *>(A_dev);
    char *oh = static_cast<char *>(Ai_host);
    const char *od = static_cast<const char *>(Ai_dev);
    cudaEvent_t *ev = ce->ev;                // [0] start, [1] end, then two per piece
    bool ok = cudaEventRecord(ev[0], s) == cudaSuccess && cudaStreamWaitEvent(ce->in, ev[0], 0) == cudaSuccess &&
              cudaStreamWaitEvent(ce->out, ev[0], 0) == cudaSuccess;
    if (ok && cu_dev != nullptr)
        ok = cudaMemcpyAsync(cu_dev, cu_seqlens_host, sizeof(int32_t) * size_t(num_seqs + 1),
                             cudaMemcpyHostToDevice, ce->in) == cudaSuccess;
    for (int k = 0; ok && k < np; ++k) {
        const Piece &q = pc[k];
        cudaEvent_t loaded = ev[2 + 2 * k], solved = ev[3 + 2 * k];
        ok = cudaMemcpyAsync(ad + q.r0 * row_in, ah + q.r0 * row_in, size_t(q.r1 - q.r0) * row_in,
                             cudaMemcpyHostToDevice, ce->in) == cudaSuccess &&
             cudaEventRecord(loaded, ce->in) == cudaSuccess && cudaStreamWaitEvent(s, loaded, 0) == cudaSuccess;
        if (!ok) break;
        if (cu_dev != nullptr)               // requests s0 .. s0+ns-1, rows absolute in A
            st = kda_solve_tril(A_dev, Ai_dev, cu_dev + q.s0, q.ns, 1, T, H, in_dtype, out_dtype, workspace,
                                workspace_bytes, stream);
        else
            st = kda_solve_tril(ad + (q.b * T + q.t0) * row_in, static_cast<char *>(Ai_dev) + (q.b * T + q.t0) * row_out,
                                nullptr, 0, q.nb, q.nt, H, in_dtype, out_dtype, workspace, workspace_bytes, stream);
        if (st != KDA_OK) return st;
        ok = cudaEventRecord(solved, s) == cudaSuccess && cudaStreamWaitEvent(ce->out, solved, 0) == cudaSuccess &&
             cudaMemcpyAsync(oh + q.r0 * row_out, od + q.r0 * row_out, size_t(q.r1 - q.r0) * row_out,
                             cudaMemcpyDeviceToHost, ce->out) == cudaSuccess;
    }
    // the caller's stream waits for the last copy back
    ok = ok && cudaEventRecord(ev[1], ce->out) == cudaSuccess && cudaStreamWaitEvent(s, ev[1], 0) == cudaSuccess;
    return ok ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_solve_tril_bt(const void *A, void *Ai, const int32_t *cu_seqlens, int32_t num_seqs, int64_t B,
                               int64_t T, int32_t H, int32_t bt, int32_t in_dtype, int32_t out_dtype, void *stream) {
    if (bt == kda::BT)
        return kda_solve_tril_ex(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype, nullptr, 0, stream,
                                 KDA_PATH_SINGLE, nullptr);
    if (bt != 16 && bt != 32) return KDA_ERR_UNSUPPORTED;
    kda_status_t st = check_args(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype, bt);
    if (st != KDA_OK) return st;
    if (B == 0 || T == 0) return KDA_OK;
    const size_t elems = size_t(B) * size_t(T) * size_t(H) * size_t(bt);
    if (!aligned16(A) || !aligned16(Ai)) return KDA_ERR_INVALID_ARGUMENT;
    if (overlaps(A, elems * elt_size(in_dtype), Ai, elems * elt_size(out_dtype))) return KDA_ERR_INVALID_ARGUMENT;

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    DeviceInfo info;
    if (device_info(device, info) != cudaSuccess) return KDA_ERR_CUDA;
    kda::SmallParams p;
    p.A = A;
    p.out = Ai;
    p.cu = cu_seqlens;
    p.nseq = num_seqs;
    p.H = H;
    p.T = T;
    p.cpr = static_cast<int32_t>((T + bt - 1) / bt);
    p.n_tasks = static_cast<int32_t>(max_chunks(B, T, num_seqs, bt) * H);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (in_dtype) {
        case KDA_F32: e = kda::launch_small_f32(bt, out_dtype, p, device, info.num_sms, s); break;
        case KDA_BF16: e = kda::launch_small_bf16(bt, out_dtype, p, device, info.num_sms, s); break;
        default: e = kda::launch_small_f16(bt, out_dtype, p, device, info.num_sms, s); break;
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_solve_tril_kgb(const void *k, const float *g, const void *beta, void *Ai,
                                const int32_t *cu_seqlens, int32_t num_seqs, int64_t B, int64_t T, int32_t H,
                                int32_t K, int32_t in_dtype, int32_t out_dtype, void *stream) {
    kda_status_t st = check_args(k, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype);
    if (st != KDA_OK) return st;
    if (K != 32 && K != 64 && K != 96 && K != 128) return KDA_ERR_UNSUPPORTED;
    if (B == 0 || T == 0) return KDA_OK;
    if (g == nullptr || beta == nullptr) return KDA_ERR_INVALID_ARGUMENT;
    const size_t rows = size_t(B) * size_t(T);
    const size_t kb = rows * size_t(H) * size_t(K) * elt_size(in_dtype), gbytes = rows * size_t(H) * size_t(K) * 4;
    const size_t bb = rows * size_t(H) * elt_size(in_dtype), ob = rows * size_t(H) * kda::BT * elt_size(out_dtype);
    if (!aligned16(k) || !aligned16(g) || !aligned16(Ai) ||
        (reinterpret_cast<uintptr_t>(beta) % uintptr_t(elt_size(in_dtype))) != 0)
        return KDA_ERR_INVALID_ARGUMENT;
    if (overlaps(Ai, ob, k, kb) || overlaps(Ai, ob, g, gbytes) || overlaps(Ai, ob, beta, bb))
        return KDA_ERR_INVALID_ARGUMENT;

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    DeviceInfo info;
    if (device_info(device, info) != cudaSuccess) return KDA_ERR_CUDA;
    kda::KgbParams p;
    p.k = k;
    p.g = g;
    p.beta = beta;
    p.out = Ai;
    p.cu = cu_seqlens;
    p.nseq = num_seqs;
    p.H = H;
    p.T = T;
    p.cpr = static_cast<int32_t>((T + kda::BT - 1) / kda::BT);
    p.n_tasks = static_cast<int32_t>(max_chunks(B, T, num_seqs) * H);
    p.K = K;
    p.err = info.err;
    kda::KgbMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode_kg_maps(k, in_dtype, g, H, K, int64_t(rows), maps)) return KDA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (in_dtype) {
        case KDA_F32: e = kda::launch_kgb_f32(out_dtype, maps, p, device, info.num_sms, s); break;
        case KDA_BF16: e = kda::launch_kgb_bf16(out_dtype, maps, p, device, info.num_sms, s); break;
        default: e = kda::launch_kgb_f16(out_dtype, maps, p, device, info.num_sms, s); break;
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

const char *kda_status_string(int32_t status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported dtype or size";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small for the split path";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_DEVICE: return "device-side error recorded";
        default: return "unknown status";
    }
}

kda_status_t kda_device_error(int32_t device, uint32_t *code) {
    if (code == nullptr) return KDA_ERR_INVALID_ARGUMENT;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return KDA_ERR_CUDA;
    unsigned v = 0;
    const unsigned zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_kda_err, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_kda_err, &zero, sizeof(zero));
    cudaSetDevice(prev);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    *code = v;
    return KDA_OK;
}

kda_status_t kda_selftest_wait(int32_t complete, uint32_t limit_us, void *stream) {
    if (limit_us == 0 || limit_us > 1000000u) return KDA_ERR_INVALID_ARGUMENT;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    DeviceInfo info;
    if (device_info(device, info) != cudaSuccess) return KDA_ERR_CUDA;
    kda_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(info.err, complete != 0,
                                                                             uint64_t(limit_us) * 1000u);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int32_t kda_version(void) { return 100; }

}  // extern "C"
