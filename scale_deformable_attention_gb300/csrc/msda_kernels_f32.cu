// Kernel instantiations for f32 I/O (see msda_device.cuh): forward kernels,
// the backward with fp32 reductions, the fused operator's reference-point kernel.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_forward<float>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_forward_tma<float>(const KernelArgs&, const CUtensorMap&, int, unsigned, cudaStream_t);
template void launch_forward_pointparallel<float>(const KernelArgs&, unsigned, cudaStream_t);
template void launch_backward<float, float>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_fused_ref_grad<float>(const float*, float*, const int64_t*, long long, int, int, int, cudaStream_t);
}  // namespace msda
