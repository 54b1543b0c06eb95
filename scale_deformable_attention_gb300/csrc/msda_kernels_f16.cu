// Kernel instantiations for f16 I/O (see msda_device.cuh).
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_forward<__half>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_forward_tma<__half>(const KernelArgs&, const CUtensorMap&, int, unsigned, cudaStream_t);
template void launch_forward_pointparallel<__half>(const KernelArgs&, unsigned, cudaStream_t);
template void launch_backward<__half, __half>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_backward<__half, float>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_convert<__half>(const float*, __half*, long long, int, int, cudaStream_t);
template void launch_widen<__half>(const __half*, float*, long long, int, cudaStream_t);
template void launch_backward<__half, long long>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_det_max<__half>(const __half*, long long, const __half*, long long, float, DetHeader*, int, cudaStream_t);
template void launch_det_convert<__half>(const long long*, __half*, long long, const DetHeader*, long long, int, int,
                                      cudaStream_t);
template void launch_fused_ref_grad<__half>(const __half*, __half*, const int64_t*, long long, int, int, int, cudaStream_t);
}  // namespace msda
