// Kernel instantiations for f32 I/O (see msda_tiled.cuh): the on-chip FP32
// accumulator's count, place and accumulate passes and the backward's gather
// phase without its scatter.
#define MSDA_INSTANTIATE
#include "msda_launch.cuh"

namespace msda {
template void launch_backward_gather<float>(const KernelArgs&, const Plan&, cudaStream_t);
template void launch_tile_count<float>(const TileArgs&, cudaStream_t);
template void launch_tile_place<float>(const TileArgs&, cudaStream_t);
template void launch_tile_scan<float>(const TileArgs&, cudaStream_t);
template void launch_tile_accum<float>(const TileArgs&, int, cudaStream_t);
}  // namespace msda
