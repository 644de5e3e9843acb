// kda_launch.cuh -- host-side launch of one kernel instantiation.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "kda_kernels.cuh"
#include "kda_small.cuh"
#include "kda_kgb.cuh"

namespace kda {

// Launch with programmatic stream serialization (pdl = true): the kernel may be
// scheduled while the previous kernel of the stream finishes (its CTAs take the
// SMs that CTA by CTA become free), and waits in griddepcontrol.wait before it
// touches global memory, which removes the launch gap between back-to-back
// kernels.  pdl = false is an ordinary launch (griddepcontrol is then a no-op).
template <typename... Args>
cudaError_t launch_pdl(bool pdl, void (*fn)(Args...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fn, args...);
}

// Per-device cache: opt-in shared memory set and occupancy queried once.
template <int MODE, typename TIn, typename TOut, bool TF32 = false>
struct KernelInfo {
    static int blocks_per_sm(int device, cudaError_t &err) {
        static std::mutex mu;
        static int cached[64] = {0};
        std::lock_guard<std::mutex> lock(mu);
        err = cudaSuccess;
        if (device < 0 || device >= 64) {
            err = cudaErrorInvalidDevice;
            return 0;
        }
        if (cached[device] > 0) return cached[device];
        auto fn = kda_tril_kernel<MODE, TIn, TOut, TF32>;
        const int bytes = Layout<MODE, TIn>::BYTES;
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (err != cudaSuccess) return 0;
        int occ = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, NTHREADS, bytes);
        if (err != cudaSuccess) return 0;
        cached[device] = occ > 0 ? occ : 1;
        return cached[device];
    }
};

template <int MODE, typename TIn, typename TOut, bool TF32 = false>
cudaError_t launch_one(const Maps &maps, const Params &p, int device, int num_sms, cudaStream_t stream) {
    cudaError_t err;
    const int occ = KernelInfo<MODE, TIn, TOut, TF32>::blocks_per_sm(device, err);
    if (err != cudaSuccess) return err;
    long long grid = (long long)num_sms * occ;
    if (grid > p.n_tasks) grid = p.n_tasks;
    if (grid < 1) return cudaSuccess;
    // the split path's two kernels run without it: on GB300 the forced split
    // solve of 8192 tokens x 64 heads took 71.6 us back to back with it, 63.8
    // without (the single pass: 39.5 with, 41.4 without)
    return launch_pdl(MODE == MODE_FUSED, kda_tril_kernel<MODE, TIn, TOut, TF32>, (unsigned)grid, NTHREADS,
                      Layout<MODE, TIn>::BYTES, stream, maps, p);
}

// Dispatch on the output dtype (0 f32, 1 bf16, 2 f16) for one input dtype.
template <typename TIn>
cudaError_t launch_in(int mode, int out_dtype, const Maps &maps, const Params &p, int device, int num_sms,
                      cudaStream_t stream) {
    if (mode == MODE_DIAG) {        // writes the diagonal and zero blocks of the output too
        switch (out_dtype) {
            case 0: return launch_one<MODE_DIAG, TIn, float>(maps, p, device, num_sms, stream);
            case 1: return launch_one<MODE_DIAG, TIn, __nv_bfloat16>(maps, p, device, num_sms, stream);
            default: return launch_one<MODE_DIAG, TIn, __half>(maps, p, device, num_sms, stream);
        }
    }
    if (mode == MODE_FUSED) {
        switch (out_dtype) {
            case 0: return launch_one<MODE_FUSED, TIn, float>(maps, p, device, num_sms, stream);
            case 1: return launch_one<MODE_FUSED, TIn, __nv_bfloat16>(maps, p, device, num_sms, stream);
            default: return launch_one<MODE_FUSED, TIn, __half>(maps, p, device, num_sms, stream);
        }
    }
    if (mode == MODE_FUSED_TF32) {
        switch (out_dtype) {
            case 0: return launch_one<MODE_FUSED, TIn, float, true>(maps, p, device, num_sms, stream);
            case 1: return launch_one<MODE_FUSED, TIn, __nv_bfloat16, true>(maps, p, device, num_sms, stream);
            default: return launch_one<MODE_FUSED, TIn, __half, true>(maps, p, device, num_sms, stream);
        }
    }
    switch (out_dtype) {
        case 0: return launch_one<MODE_MERGE, TIn, float>(maps, p, device, num_sms, stream);
        case 1: return launch_one<MODE_MERGE, TIn, __nv_bfloat16>(maps, p, device, num_sms, stream);
        default: return launch_one<MODE_MERGE, TIn, __half>(maps, p, device, num_sms, stream);
    }
}

// ------------------------------------------------ 16- and 32-token chunks
template <int CBT, typename TIn, typename TOut>
struct SmallKernel {
    static constexpr int SLOTS = CBT == 16 ? BT16_SLOTS : 2;   // chunk-heads a CTA works on at once
    static void (*fn())(SmallParams) { return CBT == 16 ? kda_bt16_kernel<TIn, TOut> : kda_bt32_kernel<TIn, TOut>; }
    static int blocks_per_sm(int device, cudaError_t &err) {
        static std::mutex mu;
        static int cached[64] = {0};
        std::lock_guard<std::mutex> lock(mu);
        err = cudaSuccess;
        if (device < 0 || device >= 64) {
            err = cudaErrorInvalidDevice;
            return 0;
        }
        if (cached[device] > 0) return cached[device];
        int occ = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn(), NTHREADS, 0);
        if (err != cudaSuccess) return 0;
        cached[device] = occ > 0 ? occ : 1;
        return cached[device];
    }
    static cudaError_t launch(const SmallParams &p, int device, int num_sms, cudaStream_t stream) {
        cudaError_t err;
        const int occ = blocks_per_sm(device, err);
        if (err != cudaSuccess) return err;
        long long grid = (long long)num_sms * occ;
        const long long need = (p.n_tasks + SLOTS - 1) / SLOTS;
        if (grid > need) grid = need;
        if (grid < 1) return cudaSuccess;
        return launch_pdl(true, fn(), (unsigned)grid, NTHREADS, 0, stream, p);
    }
};

// Chunk length bt (16 or 32), dispatched on the output dtype.
template <typename TIn>
cudaError_t launch_small_in(int bt, int out_dtype, const SmallParams &p, int device, int num_sms,
                            cudaStream_t stream) {
    if (bt == 16) {
        switch (out_dtype) {
            case 0: return SmallKernel<16, TIn, float>::launch(p, device, num_sms, stream);
            case 1: return SmallKernel<16, TIn, __nv_bfloat16>::launch(p, device, num_sms, stream);
            default: return SmallKernel<16, TIn, __half>::launch(p, device, num_sms, stream);
        }
    }
    switch (out_dtype) {
        case 0: return SmallKernel<32, TIn, float>::launch(p, device, num_sms, stream);
        case 1: return SmallKernel<32, TIn, __nv_bfloat16>::launch(p, device, num_sms, stream);
        default: return SmallKernel<32, TIn, __half>::launch(p, device, num_sms, stream);
    }
}

// ------------------------------------ chunk matrix from keys, betas, decays
template <typename TIn, typename TOut>
struct KgbKernel {
    static int blocks_per_sm(int device, cudaError_t &err) {
        static std::mutex mu;
        static int cached[64] = {0};
        std::lock_guard<std::mutex> lock(mu);
        err = cudaSuccess;
        if (device < 0 || device >= 64) {
            err = cudaErrorInvalidDevice;
            return 0;
        }
        if (cached[device] > 0) return cached[device];
        auto fn = kda_kgb_kernel<TIn, TOut>;
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, KGB_BYTES);
        if (err != cudaSuccess) return 0;
        int occ = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, KGB_THREADS, KGB_BYTES);
        if (err != cudaSuccess) return 0;
        cached[device] = occ > 0 ? occ : 1;
        return cached[device];
    }
    static cudaError_t launch(const KgbMaps &maps, const KgbParams &p, int device, int num_sms,
                              cudaStream_t stream) {
        cudaError_t err;
        const int occ = blocks_per_sm(device, err);
        if (err != cudaSuccess) return err;
        long long grid = (long long)num_sms * occ;
        if (grid > p.n_tasks) grid = p.n_tasks;
        if (grid < 1) return cudaSuccess;
        return launch_pdl(true, kda_kgb_kernel<TIn, TOut>, (unsigned)grid, KGB_THREADS, KGB_BYTES, stream, maps,
                          p);
    }
};

template <typename TIn>
cudaError_t launch_kgb_in(int out_dtype, const KgbMaps &maps, const KgbParams &p, int device, int num_sms,
                          cudaStream_t stream) {
    switch (out_dtype) {
        case 0: return KgbKernel<TIn, float>::launch(maps, p, device, num_sms, stream);
        case 1: return KgbKernel<TIn, __nv_bfloat16>::launch(maps, p, device, num_sms, stream);
        default: return KgbKernel<TIn, __half>::launch(maps, p, device, num_sms, stream);
    }
}

// defined in kda_inst_{f32,bf16,f16}.cu
cudaError_t launch_f32(int mode, int out_dtype, const Maps &, const Params &, int, int, cudaStream_t);
cudaError_t launch_bf16(int mode, int out_dtype, const Maps &, const Params &, int, int, cudaStream_t);
cudaError_t launch_f16(int mode, int out_dtype, const Maps &, const Params &, int, int, cudaStream_t);
cudaError_t launch_small_f32(int bt, int out_dtype, const SmallParams &, int, int, cudaStream_t);
cudaError_t launch_small_bf16(int bt, int out_dtype, const SmallParams &, int, int, cudaStream_t);
cudaError_t launch_small_f16(int bt, int out_dtype, const SmallParams &, int, int, cudaStream_t);
cudaError_t launch_kgb_f32(int out_dtype, const KgbMaps &, const KgbParams &, int, int, cudaStream_t);
cudaError_t launch_kgb_bf16(int out_dtype, const KgbMaps &, const KgbParams &, int, int, cudaStream_t);
cudaError_t launch_kgb_f16(int out_dtype, const KgbMaps &, const KgbParams &, int, int, cudaStream_t);

}  // namespace kda
