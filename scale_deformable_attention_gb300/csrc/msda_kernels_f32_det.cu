// Kernel instantiations for f32 I/O (see msda_device.cuh): the backward with
// the deterministic (int64 fixed-point) accumulator and its maxima and
// conversion kernels.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_backward<float, long long>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_det_max<float>(const float*, long long, const float*, long long, float, DetHeader*, int, cudaStream_t);
template void launch_det_convert<float>(const long long*, float*, long long, const DetHeader*, long long, int, int,
                                      cudaStream_t);
}  // namespace msda
