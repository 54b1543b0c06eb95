// Kernel instantiations for bf16 I/O (see msda_device.cuh): forward kernels,
// the backward with native bf16 reductions, the fused operator's reference-point kernel.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_forward<__nv_bfloat16>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_forward_tma<__nv_bfloat16>(const KernelArgs&, const CUtensorMap&, int, unsigned, cudaStream_t);
template void launch_forward_pointparallel<__nv_bfloat16>(const KernelArgs&, unsigned, cudaStream_t);
template void launch_backward<__nv_bfloat16, __nv_bfloat16>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_fused_ref_grad<__nv_bfloat16>(const __nv_bfloat16*, __nv_bfloat16*, const int64_t*, long long, int, int, int, cudaStream_t);
}  // namespace msda
