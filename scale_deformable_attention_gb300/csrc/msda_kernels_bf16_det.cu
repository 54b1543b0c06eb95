// Kernel instantiations for bf16 I/O (see msda_device.cuh): the backward with
// the deterministic (int64 fixed-point) accumulator and its maxima and
// conversion kernels.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_backward<__nv_bfloat16, long long>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_det_max<__nv_bfloat16>(const __nv_bfloat16*, long long, const __nv_bfloat16*, long long, float, DetHeader*, int, cudaStream_t);
template void launch_det_convert<__nv_bfloat16>(const long long*, __nv_bfloat16*, long long, const DetHeader*, long long, int, int,
                                      cudaStream_t);
}  // namespace msda
