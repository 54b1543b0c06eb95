// Kernel instantiations for f16 I/O (see msda_device.cuh): the backward with
// the deterministic (int64 fixed-point) accumulator and its maxima and
// conversion kernels.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_backward<__half, long long>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_det_max<__half>(const __half*, long long, const __half*, long long, float, DetHeader*, int, cudaStream_t);
template void launch_det_convert<__half>(const long long*, __half*, long long, const DetHeader*, long long, int, int,
                                      cudaStream_t);
}  // namespace msda
