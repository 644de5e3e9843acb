// Kernel instantiations for f32 input.
#include "kda_launch.cuh"

namespace kda {
cudaError_t launch_f32(int mode, int out_dtype, const Maps &maps, const Params &p, int device, int num_sms,
                       cudaStream_t stream) {
    return launch_in<float>(mode, out_dtype, maps, p, device, num_sms, stream);
}
cudaError_t launch_small_f32(int bt, int out_dtype, const SmallParams &p, int device, int num_sms,
                             cudaStream_t stream) {
    return launch_small_in<float>(bt, out_dtype, p, device, num_sms, stream);
}
cudaError_t launch_kgb_f32(int out_dtype, const KgbMaps &maps, const KgbParams &p, int device, int num_sms,
                          cudaStream_t stream) {
    return launch_kgb_in<float>(out_dtype, maps, p, device, num_sms, stream);
}
}  // namespace kda
