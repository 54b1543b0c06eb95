// Kernel instantiations for bf16 I/O (see msda_tiled.cuh): the on-chip FP32
// accumulator's count, place and accumulate passes and the backward's gather
// phase without its scatter.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_backward_gather<__nv_bfloat16>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_tile_count<__nv_bfloat16>(const TileArgs&, cudaStream_t);
template void launch_tile_place<__nv_bfloat16>(const TileArgs&, cudaStream_t);
template void launch_tile_scan<__nv_bfloat16>(const TileArgs&, cudaStream_t);
template void launch_tile_accum<__nv_bfloat16>(const TileArgs&, int, cudaStream_t);
}  // namespace msda
