// Kernel instantiations for f16 I/O (see msda_device.cuh): the backward
// into the fp32 workspace, its widen / convert kernels and the touch count.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_backward<__half, float>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_convert<__half>(float*, __half*, long long, int, int, int, cudaStream_t);
template void launch_touch_count<__half>(const KernelArgs&, int, cudaStream_t);
template void launch_round_rows<__half>(const KernelArgs&, int, int, cudaStream_t);
template void launch_widen<__half>(const __half*, float*, long long, int, cudaStream_t);
}  // namespace msda
