// kda_no_alloc.cu -- split-path solve with a built-in workspace, for callers
// that cannot allocate device memory.
//
// Some callers have no way to get scratch memory at the point where they call
// the solver: a plugin running inside a host framework that owns all device
// memory and gives its plugins no allocation hook, or a serving loop that fixed
// its memory at start-up and must not call cudaMalloc / cudaFree afterwards
// (those calls can synchronise the device and stall every stream).  This entry
// point takes only inputs and outputs; the split path's FP32 workspace lives in
// the file-scope array below, which every GPU that loads this library holds
// until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "kda_internal.h"
#include "kda_solve_tril.h"

namespace {

// The built-in workspace.  In host code this name is only a host-side stand-in
// for the device array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_kda_static_ws[KDA_STATIC_WS_BYTES];

// Device address of g_kda_static_ws per device, resolved once per device (a
// cudaDeviceReset of that device would make it stale: the library's per-device
// state does not survive one).
cudaError_t static_ws_ptr(void **out) {
    static std::mutex mu;
    static void *ptrs[64] = {nullptr};
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[device] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_kda_static_ws);   // with `device` current
        if (e != cudaSuccess) return e;
        ptrs[device] = p;
    }
    *out = ptrs[device];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status_t kda_solve_tril_split_static(const void *A, void *Ai, const int32_t *cu_seqlens,
                                                    int32_t num_seqs, int64_t B, int64_t T, int32_t H,
                                                    int32_t in_dtype, int32_t out_dtype, void *stream) {
    // every argument error is reported before any CUDA call
    const kda_status_t st = kda::validate_solve(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype);
    if (st != KDA_OK) return st;
    const size_t need = kda_solve_tril_workspace_size(B, T, H, num_seqs);
    if (need > size_t(KDA_STATIC_WS_BYTES)) return KDA_ERR_WORKSPACE;
    if (B == 0 || T == 0) return KDA_OK;
    void *ws = nullptr;
    if (static_ws_ptr(&ws) != cudaSuccess) return KDA_ERR_CUDA;
    // Nothing in the array needs to start at zero: the diagonal-inverse kernel
    // writes every tile that the merge kernel then reads.
    return kda_solve_tril_ex(A, Ai, cu_seqlens, num_seqs, B, T, H, in_dtype, out_dtype, ws,
                             size_t(KDA_STATIC_WS_BYTES), stream, KDA_PATH_SPLIT, nullptr);
}
