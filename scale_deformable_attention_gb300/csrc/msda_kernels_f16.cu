// Kernel instantiations for f16 I/O (see msda_device.cuh): forward kernels,
// the backward with native f16 reductions, the fused operator's reference-point kernel.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_forward<__half>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_forward_tma<__half>(const KernelArgs&, const CUtensorMap&, int, unsigned, cudaStream_t);
template void launch_forward_pointparallel<__half>(const KernelArgs&, unsigned, cudaStream_t);
template void launch_backward<__half, __half>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_fused_ref_grad<__half>(const __half*, __half*, const int64_t*, long long, int, int, int, cudaStream_t);
}  // namespace msda
