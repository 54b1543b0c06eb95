// msda_probe.cu -- msda_reduction_ceiling: the L2's throughput for the
// backward's kind of reduction traffic (rows of row_bytes at random places,
// each row taken by row_bytes / 16 adjacent lanes with one 16-byte vector
// reduction each, as a team adds one corner row of grad_value), measured
// alone so that the backward's scatter can be reported against it.
#include <cuda_runtime.h>

#include <cstdint>

#include "msda_internal.h"

namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeIters = 256;

// a 32-bit integer hash (xor-shift-multiply), for scattered sector indices
__device__ __forceinline__ uint32_t scatter_hash(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

// Groups of LPR = row_bytes / 16 adjacent lanes add into one row, a new
// random row per iteration; every address is inside [buf, buf + n_rows * row_bytes).
template <int KIND>
__global__ void __launch_bounds__(kProbeThreads) msda_reduction_probe_kernel(unsigned char* buf, uint32_t n_rows,
                                                                             int lg_lpr) {
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t grp = tid >> lg_lpr, slot = tid & ((1u << lg_lpr) - 1u);
    const size_t row_bytes = (size_t)16 << lg_lpr;
    for (int i = 0; i < kProbeIters; ++i) {
        const uint32_t row = scatter_hash(grp * 1315423911u + (uint32_t)i * 2654435761u) % n_rows;
        unsigned char* p = buf + (size_t)row * row_bytes + slot * 16;
        if constexpr (KIND == 0) {
            const uint32_t one = 0x3f803f80u;  // bf16x2 (1, 1)
            asm volatile("red.relaxed.gpu.global.add.noftz.v4.bf16x2 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(one), "r"(one),
                         "r"(one), "r"(one)
                         : "memory");
        } else if constexpr (KIND == 1) {
            const uint32_t one = 0x3c003c00u;  // f16x2 (1, 1)
            asm volatile("red.relaxed.gpu.global.add.noftz.v4.f16x2 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(one), "r"(one),
                         "r"(one), "r"(one)
                         : "memory");
        } else {
            asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(1.f), "f"(1.f),
                         "f"(1.f), "f"(1.f)
                         : "memory");
        }
    }
}

void launch_probe(int kind, unsigned grid, unsigned char* buf, uint32_t n_rows, int lg_lpr, cudaStream_t st) {
    switch (kind) {
    case 0: msda_reduction_probe_kernel<0><<<grid, kProbeThreads, 0, st>>>(buf, n_rows, lg_lpr); break;
    case 1: msda_reduction_probe_kernel<1><<<grid, kProbeThreads, 0, st>>>(buf, n_rows, lg_lpr); break;
    default: msda_reduction_probe_kernel<2><<<grid, kProbeThreads, 0, st>>>(buf, n_rows, lg_lpr); break;
    }
}

}  // namespace

extern "C" msda_status msda_reduction_ceiling(int kind, int row_bytes, int blocks_per_sm, int repeats, void* scratch,
                                              size_t scratch_bytes, double* sectors_per_second, msda_stream_t stream) {
    msda::clear_error();
    if (!sectors_per_second) return msda::set_error(MSDA_ERR_INVALID_ARG, "sectors_per_second is NULL");
    if (!scratch || scratch_bytes < (1u << 20) || (reinterpret_cast<uintptr_t>(scratch) & 15u))
        return msda::set_error(MSDA_ERR_INVALID_ARG, "scratch must be a 16-byte aligned buffer of at least 1 MiB");
    if (kind < 0 || kind > 2) return msda::set_error(MSDA_ERR_INVALID_ARG, "kind must be 0 (bf16x2), 1 (f16x2) or 2 (f32)");
    if (blocks_per_sm < 1 || blocks_per_sm > 16) return msda::set_error(MSDA_ERR_INVALID_ARG, "blocks_per_sm outside 1..16");
    if (repeats < 1 || repeats > 100) return msda::set_error(MSDA_ERR_INVALID_ARG, "repeats outside 1..100");
    int lg_lpr = -1;
    for (int l = 0; l <= 5; ++l)
        if (row_bytes == (16 << l)) lg_lpr = l;
    if (lg_lpr < 0) return msda::set_error(MSDA_ERR_INVALID_ARG, "row_bytes must be 16, 32, 64, 128, 256 or 512");
    const size_t rows64 = scratch_bytes / (size_t)row_bytes;
    const uint32_t n_rows = (uint32_t)(rows64 > 0xffffffffu ? 0xffffffffu : rows64);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
    const unsigned grid = (unsigned)(sms * blocks_per_sm);
    unsigned char* buf = static_cast<unsigned char*>(scratch);
    cudaEvent_t a = nullptr, b = nullptr;
    if ((e = cudaEventCreate(&a)) != cudaSuccess || (e = cudaEventCreate(&b)) != cudaSuccess) {
        if (a) cudaEventDestroy(a);
        return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
    }
    double best = 0.0;
    launch_probe(kind, grid, buf, n_rows, lg_lpr, st);  // warm-up
    for (int r = 0; r < repeats && e == cudaSuccess; ++r) {
        cudaEventRecord(a, st);
        launch_probe(kind, grid, buf, n_rows, lg_lpr, st);
        cudaEventRecord(b, st);
        e = cudaEventSynchronize(b);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
        if (e == cudaSuccess && ms > 0.f) {
            // one 16-byte reduction per lane and iteration, two per 32-byte sector
            const double sectors = (double)grid * kProbeThreads * kProbeIters / 2.0;
            const double rate = sectors / (ms * 1e-3);
            if (rate > best) best = rate;
        }
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (e != cudaSuccess) return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
    *sectors_per_second = best;
    return MSDA_OK;
}
