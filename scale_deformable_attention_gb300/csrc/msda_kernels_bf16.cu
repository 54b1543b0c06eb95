// Kernel instantiations for bf16 I/O (see msda_device.cuh).
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_forward<__nv_bfloat16>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_forward_tma<__nv_bfloat16>(const KernelArgs&, const CUtensorMap&, int, unsigned, cudaStream_t);
template void launch_forward_pointparallel<__nv_bfloat16>(const KernelArgs&, unsigned, cudaStream_t);
template void launch_backward<__nv_bfloat16, __nv_bfloat16>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_backward<__nv_bfloat16, float>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_convert<__nv_bfloat16>(const float*, __nv_bfloat16*, long long, int, int, cudaStream_t);
template void launch_widen<__nv_bfloat16>(const __nv_bfloat16*, float*, long long, int, cudaStream_t);
template void launch_backward<__nv_bfloat16, long long>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_det_max<__nv_bfloat16>(const __nv_bfloat16*, long long, const __nv_bfloat16*, long long, float, DetHeader*, int, cudaStream_t);
template void launch_det_convert<__nv_bfloat16>(const long long*, __nv_bfloat16*, long long, const DetHeader*, long long, int, int,
                                      cudaStream_t);
template void launch_fused_ref_grad<__nv_bfloat16>(const __nv_bfloat16*, __nv_bfloat16*, const int64_t*, long long, int, int, int, cudaStream_t);
}  // namespace msda
