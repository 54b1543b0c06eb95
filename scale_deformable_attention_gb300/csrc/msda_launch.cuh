// msda_launch.cuh -- host-side launch of the kernel templates: maps a runtime
// launch plan (vector width, vectors per lane, parameter staging) onto the
// compiled instantiations.  Each dtype's instantiations live in their own
// translation unit (msda_kernels_<dtype>.cu) so they compile in parallel.
#pragma once

#include "msda_device.cuh"
#include "msda_tiled.cuh"

namespace msda {

// Samples per lane whose corner loads are issued together.
constexpr int kSamplesInFlight = 2;

struct Plan {
    dim3 grid, block;
    size_t smem;   // dynamic shared memory (staged parameters)
    int nv;        // vectors per lane, 1..4
    bool vec;      // 16-byte slots (else one element per slot)
    bool wide;     // 64-bit offsets inside a batch slice
    bool spec;     // specialised kernels: C = 4, nvec == 4 * nv, nv <= 4, 32-bit offsets
    bool pdl;      // launched as a programmatic dependent of the kernel ahead of it
    bool fused;    // fused operator (offsets + logits in, offset / logit gradients out)
    bool merge;    // backward: merge the corners a point group's samples share before the scatter
    bool c8;       // backward into the fp32 workspace, 16-bit I/O: eight lanes a unit (msda_bwd8_kernel)
};

#define MSDA_DISPATCH_NV(NVV, ...)                                   \
    switch (NVV) {                                                   \
    case 1: { constexpr int NV = 1; __VA_ARGS__; } break;            \
    case 2: { constexpr int NV = 2; __VA_ARGS__; } break;            \
    case 3: { constexpr int NV = 3; __VA_ARGS__; } break;            \
    default: { constexpr int NV = 4; __VA_ARGS__; } break;           \
    }

template <typename T, typename ACC, int NV, int EPV, bool WIDE>
static void bwd_go(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    msda_bwd_kernel<T, ACC, NV, EPV, WIDE, kSamplesInFlight><<<pl.grid, pl.block, pl.smem, st>>>(a);
}

#define MSDA_DISPATCH_NV3(NVV, ...)                                  \
    switch (NVV) {                                                   \
    case 1: { constexpr int NV = 1; __VA_ARGS__; } break;            \
    case 2: { constexpr int NV = 2; __VA_ARGS__; } break;            \
    default: { constexpr int NV = 3; __VA_ARGS__; } break;           \
    }

// Launch `kernel` with pl's shape; with pl.pdl as a programmatic dependent of
// the kernel ahead of it on the stream (it may start before that kernel has
// finished, and must griddepcontrol.wait before touching what it wrote).
static inline void launch_plan(void (*kernel)(const KernelArgs), const KernelArgs& a, const Plan& pl,
                               cudaStream_t st) {
    if (pl.pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = pl.grid;
        cfg.blockDim = pl.block;
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, kernel, a);
    } else {
        kernel<<<pl.grid, pl.block, pl.smem, st>>>(a);
    }
}

template <typename T, int NV, int EPV, bool WIDE>
static void fwd_go(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    // the kernel waits for the kernel ahead of it before reading anything
    launch_plan(msda_fwd_kernel<T, NV, EPV, WIDE, kSamplesInFlight>, a, pl, st);
}

template <typename T, int NV>
static void fwd4_go(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    // the kernel waits for the kernel ahead of it before reading anything
    if (pl.fused) launch_plan(msda_fwd4_kernel<T, NV, true>, a, pl, st);
    else launch_plan(msda_fwd4_kernel<T, NV, false>, a, pl, st);
}

template <typename T, typename ACC, int NV, bool FUSED>
static void bwd4_go2(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    // with pl.pdl: may start while the zero kernel that precedes it still
    // runs; the kernel waits (griddepcontrol.wait) before its first scatter
    // merge mode: every shared corner for a 16-bit value into the fp32
    // workspace, whole cells otherwise (the faster of the two on GB300 for
    // each accumulator)
    constexpr int MODE = (std::is_same<ACC, float>::value && sizeof(T) == 2) ? kMergeCorners : kMergeCells;
    if constexpr (std::is_same<ACC, float>::value && sizeof(T) == 2 && !FUSED) {
        if (pl.c8) {
            if (a.touch) launch_plan(msda_bwd8_kernel<T, NV, true>, a, pl, st);
            else launch_plan(msda_bwd8_kernel<T, NV, false>, a, pl, st);
            return;
        }
        // the touch classes of the workspace rows: their own kernel (its
        // extra registers stay out of the others), without the corner merge
        if (a.touch) {
            launch_plan(msda_bwd4_kernel<T, ACC, NV, false, 0, true>, a, pl, st);
            return;
        }
    }
    if (!pl.merge) {
        launch_plan(msda_bwd4_kernel<T, ACC, NV, FUSED, 0>, a, pl, st);
    } else {
        // one slot per lane: the 64-register form (the integer accumulator's would spill)
        if constexpr (NV == 1 && !std::is_same<ACC, long long>::value)
            launch_plan(msda_bwd4_merge1_kernel<T, ACC, FUSED, MODE>, a, pl, st);
        else
            launch_plan(msda_bwd4_kernel<T, ACC, NV, FUSED, MODE>, a, pl, st);
    }
}

template <typename T, typename ACC, int NV>
static void bwd4_go(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    if (pl.fused) bwd4_go2<T, ACC, NV, true>(a, pl, st);
    else bwd4_go2<T, ACC, NV, false>(a, pl, st);
}

template <typename T>
void launch_forward(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    constexpr int VE = 16 / sizeof(T);
    if (pl.spec) {
        MSDA_DISPATCH_NV(pl.nv, (fwd4_go<T, NV>(a, pl, st)))
        return;
    }
    if (pl.vec) {
        if (pl.wide) { MSDA_DISPATCH_NV(pl.nv, (fwd_go<T, NV, VE, true>(a, pl, st))) }
        else { MSDA_DISPATCH_NV(pl.nv, (fwd_go<T, NV, VE, false>(a, pl, st))) }
    } else {
        if (pl.wide) { MSDA_DISPATCH_NV(pl.nv, (fwd_go<T, NV, 1, true>(a, pl, st))) }
        else { MSDA_DISPATCH_NV(pl.nv, (fwd_go<T, NV, 1, false>(a, pl, st))) }
    }
}

template <typename T, typename ACC>
void launch_backward(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    constexpr int VE = 16 / sizeof(T);
    if (pl.spec) {
        MSDA_DISPATCH_NV(pl.nv, (bwd4_go<T, ACC, NV>(a, pl, st)))
        return;
    }
    if (pl.vec) {
        if (pl.wide) { MSDA_DISPATCH_NV(pl.nv, (bwd_go<T, ACC, NV, VE, true>(a, pl, st))) }
        else { MSDA_DISPATCH_NV(pl.nv, (bwd_go<T, ACC, NV, VE, false>(a, pl, st))) }
    } else {
        if (pl.wide) { MSDA_DISPATCH_NV(pl.nv, (bwd_go<T, ACC, NV, 1, true>(a, pl, st))) }
        else { MSDA_DISPATCH_NV(pl.nv, (bwd_go<T, ACC, NV, 1, false>(a, pl, st))) }
    }
}

template <typename T, int NV>
static void fwd_tma_go(const KernelArgs& a, const CUtensorMap& map, unsigned grid, cudaStream_t st) {
    constexpr int smem = fwd_tma_smem<T, NV>();
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(msda_fwd_tma_kernel<T, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    msda_fwd_tma_kernel<T, NV><<<grid, kTmaWarps * 32, smem, st>>>(a, map);
}

template <typename T>
void launch_forward_tma(const KernelArgs& a, const CUtensorMap& map, int nv, unsigned grid, cudaStream_t st) {
    MSDA_DISPATCH_NV3(nv, (fwd_tma_go<T, NV>(a, map, grid, st)))
}

template <typename T>
void launch_forward_pointparallel(const KernelArgs& a, unsigned grid, cudaStream_t st) {
    msda_fwd_pointparallel_kernel<T><<<grid, kBlockThreads, 0, st>>>(a);
}

template <typename T>
void launch_fused_ref_grad(const T* goff, T* gref, const int64_t* shapes, long long BQ, int M, int L, int K,
                           cudaStream_t st) {
    const long long n = BQ * L * 2;
    msda_fused_ref_grad_kernel<T><<<(unsigned)((n + kBlockThreads - 1) / kBlockThreads), kBlockThreads, 0, st>>>(
        goff, gref, shapes, BQ, M, L, K);
}

template <typename T>
void launch_det_max(const T* g, long long ng, const T* attn, long long na, float ma0, DetHeader* h, int grid,
                    cudaStream_t st) {
    msda_det_max_kernel<T><<<grid, kBlockThreads, 0, st>>>(g, ng, attn, na, ma0, h);
}

template <typename T>
void launch_det_convert(const long long* ws, T* gv, long long n, const DetHeader* h, long long qlk, int accumulate,
                        int grid, cudaStream_t st) {
    msda_det_convert_kernel<T><<<grid, kBlockThreads, 0, st>>>(ws, gv, n, h, qlk, accumulate);
}

template <typename T>
void launch_convert(float* ws, T* gv, long long n, int vec, int rezero, int grid, cudaStream_t st) {
    msda_convert_kernel<T><<<grid, kBlockThreads, 0, st>>>(ws, gv, n, vec, rezero);
}

template <typename T>
void launch_round_rows(const KernelArgs& a, int nv, int grid, cudaStream_t st) {
    MSDA_DISPATCH_NV(nv, (msda_round_rows_kernel<T, NV><<<grid, kBlockThreads, 0, st>>>(a)));
}

template <typename T>
void launch_touch_count(const KernelArgs& a, int grid, cudaStream_t st) {
    msda_touch_count_kernel<T><<<grid, kBlockThreads, 0, st>>>(a);
}

template <typename T>
void launch_widen(const T* gv, float* ws, long long n, int grid, cudaStream_t st) {
    msda_widen_kernel<T><<<grid, kBlockThreads, 0, st>>>(gv, ws, n);
}

// ---- the on-chip FP32 accumulator (msda_tiled.cuh) ----

// The backward's gather phase alone: grad_sampling_locations and
// grad_attention_weights, no grad_value scatter (specialised plans only).
template <typename T>
void launch_backward_gather(const KernelArgs& a, const Plan& pl, cudaStream_t st) {
    MSDA_DISPATCH_NV3(pl.nv, (launch_plan(msda_bwd4_kernel<T, T, NV, false, kGatherOnly>, a, pl, st)))
}

template <typename T>
void launch_tile_count(const TileArgs& t, cudaStream_t st) {
    const unsigned grid = (unsigned)((t.n_samples + kBlockThreads - 1) / kBlockThreads);
    msda_tile_count_kernel<T><<<grid, kBlockThreads, 0, st>>>(t);
}

template <typename T>
void launch_tile_place(const TileArgs& t, cudaStream_t st) {
    const unsigned grid = (unsigned)((t.n_samples + kBlockThreads - 1) / kBlockThreads);
    msda_tile_place_kernel<T><<<grid, kBlockThreads, 0, st>>>(t);
}

template <typename T>
void launch_tile_scan(const TileArgs& t, cudaStream_t st) {
    msda_tile_scan_kernel<T><<<1, kScanThreads, 0, st>>>(t);
}

// Shared memory of the accumulate pass: (1 << lg_tp) rows of D fp32.
inline size_t tile_smem(int lg_tp, int D) { return ((size_t)1 << lg_tp) * (size_t)D * sizeof(float); }

template <typename T, int NV>
static void tile_accum_go(const TileArgs& t, cudaStream_t st) {
    const size_t smem = tile_smem(t.lg_tp, t.D);
    // the static level table comes on top of the dynamic rows: allow the
    // dynamic size explicitly whenever the two together pass the default 48 KB
    if (smem + sizeof(Level) * MSDA_MAX_LEVELS > 48 * 1024)
        cudaFuncSetAttribute(msda_tile_accum_kernel<T, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    msda_tile_accum_kernel<T, NV><<<(unsigned)t.n_tiles, kBlockThreads, smem, st>>>(t);
}

template <typename T>
void launch_tile_accum(const TileArgs& t, int nv, cudaStream_t st) {
    MSDA_DISPATCH_NV3(nv, (tile_accum_go<T, NV>(t, st)))
}

#ifndef MSDA_INSTANTIATE
// defined in msda_kernels_<dtype>.cu
#define MSDA_EXTERN_IO(T)                                                                  \
    extern template void launch_forward<T>(const KernelArgs&, const Plan&, cudaStream_t); \
    extern template void launch_forward_tma<T>(const KernelArgs&, const CUtensorMap&, int, unsigned, cudaStream_t); \
    extern template void launch_forward_pointparallel<T>(const KernelArgs&, unsigned, cudaStream_t); \
    extern template void launch_fused_ref_grad<T>(const T*, T*, const int64_t*, long long, int, int, int, cudaStream_t); \
    extern template void launch_backward<T, float>(const KernelArgs&, const Plan&, cudaStream_t);             \
    extern template void launch_backward<T, long long>(const KernelArgs&, const Plan&, cudaStream_t);         \
    extern template void launch_det_max<T>(const T*, long long, const T*, long long, float, DetHeader*, int,    \
                                           cudaStream_t);                                                         \
    extern template void launch_det_convert<T>(const long long*, T*, long long, const DetHeader*, long long, int, int, \
                                               cudaStream_t);
MSDA_EXTERN_IO(float)
MSDA_EXTERN_IO(__half)
MSDA_EXTERN_IO(__nv_bfloat16)
#undef MSDA_EXTERN_IO
#define MSDA_EXTERN_HALF(T)                                                                              \
    extern template void launch_backward<T, T>(const KernelArgs&, const Plan&, cudaStream_t);           \
    extern template void launch_convert<T>(float*, T*, long long, int, int, int, cudaStream_t);         \
    extern template void launch_widen<T>(const T*, float*, long long, int, cudaStream_t);                \
    extern template void launch_touch_count<T>(const KernelArgs&, int, cudaStream_t);                \
    extern template void launch_round_rows<T>(const KernelArgs&, int, int, cudaStream_t);
MSDA_EXTERN_HALF(__half)
MSDA_EXTERN_HALF(__nv_bfloat16)
#undef MSDA_EXTERN_HALF
#define MSDA_EXTERN_TILED(T)                                                                     \
    extern template void launch_backward_gather<T>(const KernelArgs&, const Plan&, cudaStream_t); \
    extern template void launch_tile_count<T>(const TileArgs&, cudaStream_t);                    \
    extern template void launch_tile_place<T>(const TileArgs&, cudaStream_t);                    \
    extern template void launch_tile_scan<T>(const TileArgs&, cudaStream_t);                     \
    extern template void launch_tile_accum<T>(const TileArgs&, int, cudaStream_t);
MSDA_EXTERN_TILED(float)
MSDA_EXTERN_TILED(__half)
MSDA_EXTERN_TILED(__nv_bfloat16)
#undef MSDA_EXTERN_TILED
#endif

}  // namespace msda
