// Kernel instantiations for bf16 I/O (see msda_device.cuh): the backward
// into the fp32 workspace, its widen / convert kernels and the touch count.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_backward<__nv_bfloat16, float>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_convert<__nv_bfloat16>(float*, __nv_bfloat16*, long long, int, int, int, cudaStream_t);
template void launch_touch_count<__nv_bfloat16>(const KernelArgs&, int, cudaStream_t);
template void launch_round_rows<__nv_bfloat16>(const KernelArgs&, int, int, cudaStream_t);
template void launch_widen<__nv_bfloat16>(const __nv_bfloat16*, float*, long long, int, cudaStream_t);
}  // namespace msda
