// Kernel instantiations for bf16 input.
#include "kda_launch.cuh"

namespace kda {
cudaError_t launch_bf16(int mode, int out_dtype, const Maps &maps, const Params &p, int device, int num_sms,
                       cudaStream_t stream) {
    return launch_in<__nv_bfloat16>(mode, out_dtype, maps, p, device, num_sms, stream);
}
cudaError_t launch_small_bf16(int bt, int out_dtype, const SmallParams &p, int device, int num_sms,
                             cudaStream_t stream) {
    return launch_small_in<__nv_bfloat16>(bt, out_dtype, p, device, num_sms, stream);
}
cudaError_t launch_kgb_bf16(int out_dtype, const KgbMaps &maps, const KgbParams &p, int device, int num_sms,
                          cudaStream_t stream) {
    return launch_kgb_in<__nv_bfloat16>(out_dtype, maps, p, device, num_sms, stream);
}
}  // namespace kda
