// msda_device.cuh -- sm_103a device code of the multi-scale deformable
// attention sampling core: forward gather, backward gather + relaxed
// vector-atomic scatter, and the zero / convert helpers of the backward.
//
// Work decomposition.  One *unit* is one (b, q, m) output vector of D
// channels; units are numbered u = (b*Q + q)*M + m, so consecutive units own
// contiguous rows of out / grad_out and contiguous runs of the sampling
// parameters (both [.., M, L, K, ..] with m innermost before (l, k)).  A *team*
// of C*P lanes (C, P powers of two, C*P <= 32, teams never straddle a warp)
// owns one unit:
//   * C channel lanes split a D-row into 16-byte vectors (8 bf16/fp16 or 4
//     fp32 channels; NV vectors per lane), so each corner row is read with
//     full-width loads over the channel dimension;
//   * P point lanes split the L*K sampling points of the unit.
// A block holds 256 / (C*P) consecutive units.  The forward keeps a private
// fp32 register accumulator per lane and combines the P point lanes with
// warp shuffles at the end (no cross-block combine); the backward reduces the
// per-sample dot products over the C channel lanes with warp shuffles and
// scatters grad_value with relaxed vector reductions (red.global.add.v4.*),
// which return nothing and impose no ordering; the end of the kernel is the
// only synchronisation the sums need.
//
// This differs from the msda-triton query-block kernel (course ch. 4,
// "The design question") in that a block owns consecutive flat (b, q, m)
// units rather than a query block of one (b, m): the parameters of a block
// are then one contiguous byte range, staged into shared memory with one
// bulk copy, and the output tile is one contiguous store.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include <cuda.h>  // CUtensorMap

#include "../../include/msda.h"

namespace msda {

constexpr int kBlockThreads = 256;

// Sampling-parameter staging.
enum ParamMode : int { PARAMS_DIRECT = 0, PARAMS_SMEM_LD = 1, PARAMS_SMEM_BULK = 2 };

// Device error bits (msda_device_errors).
constexpr unsigned kErrBadLevel = 1u;
constexpr unsigned kErrBulkTimeout = 2u;
constexpr unsigned kErrTouch = 8u;   // a corner row the touch count missed (never expected)

// n / d for 0 <= n < 2^31 by a multiply-high and a shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994:
// the round-up multiplier m = floor(2^32 (2^l - d) / d) + 1, l = ceil(log2 d),
// with the 33rd multiplier bit applied as the "+ n").
struct FastDiv {
    uint32_t mul, shift;
};
__device__ __forceinline__ uint32_t fdiv(uint32_t n, FastDiv f) { return (__umulhi(n, f.mul) + n) >> f.shift; }

// One pyramid level in shared memory; offsets are in elements inside the
// [S, M, D] slice of one batch image.
struct Level {
    long long start_md;  // level_start_index * M * D
    long long w_md;      // W * M * D (one image row)
    float fH, fW;
    int ok;              // passed the shape check
    int W;               // level width
    long long start;     // level_start_index
};

struct KernelArgs {
    const void* value;
    const int64_t* shapes;
    const int64_t* starts;
    const void* loc;
    const void* attn;
    void* out;             // forward output
    const void* grad_out;  // backward input
    void* grad_acc;        // backward: grad_value (native) or the fp32 workspace
    void* grad_loc;
    void* grad_attn;
    unsigned* err;         // device error word
    long long S;           // pyramid rows
    long long slice;       // S * M * D: elements of one batch image
    int M, D, L, K, LK;
    int n_units;           // B * Q * M (< 2^31)
    FastDiv div_qm, div_m, div_k;
    FastDiv div_lk, div_d8;  // by L*K and by D/8 (touch classes only)
    int lc, lp;            // log2(C), log2(P)
    int nvec;              // vectors per D-row
    int tpb;               // units (teams) per block
    int param_mode;        // ParamMode
    int Q;                 // queries
    const struct DetHeader* det;  // deterministic accumulator: maxima for the fixed-point scale
    // fused operator: loc / attn above hold sampling offsets / attention logits,
    // grad_loc / grad_attn receive grad_offsets / grad_logits
    const void* ref;       // reference points [B, Q, L, 2]
    int gbuf_off;          // fused backward: byte offset of the per-sample <g, sampled> buffer in shared memory
    int rbuf_off;          // fused backward: byte offset of the per-sample grad_loc buffer, or -1 (separate kernel)
    void* gref;            // fused backward: grad_reference_points [B, Q, L, 2] (with rbuf_off >= 0)
    // backward: the samples [s_begin, s_end) of every unit (all of them, or
    // one level's when the backward runs one pass per level)
    int s_begin, s_end;
    // Rounding of the fp32 workspace folded into a backward pass (FP32
    // accumulator, one pass per level): conv_blocks blocks of the launch,
    // every conv_every-th one, each round one chunk of conv_chunk workspace
    // elements into grad_value (conv_out), restricted to the pyramid rows
    // below the first row of levels >= conv_level, which no pass from
    // conv_level on adds to.  conv_first: this launch's first chunk.
    int conv_blocks, conv_every, conv_level, conv_rezero;
    int conv_lo, conv_hi;  // tail rounding: rows from the first row of the levels >= conv_lo (row 0 when < 0)
                           // up to the first row of the levels >= conv_hi (the end when >= L)
    long long conv_first, conv_chunk, conv_chunks_per_image;
    void* conv_out;
    int n_images;          // B
    // Touch classes of the FP32 workspace's rows (see touch_sparse): 2 bits
    // per (b, pixel, head) row, 16 rows a word, at (b*M + m)*S + pixel;
    // class 0 no contribution, 1 exactly one, 2 (or 3) several.  A row of a
    // sparse level with one contribution is written to touch_out (grad_value)
    // directly and never reaches the workspace; rounding skips it, and writes
    // zeros for an untouched one without reading the workspace.  NULL: off.
    unsigned* touch;
    int touch_tau;
    void* touch_out;
    // TMA-gather forward: L2 size, for the eviction priority of large levels (0: none)
    long long l2_bytes;
};

// Head of the deterministic accumulator's workspace (256 bytes, then the
// int64 sums): bit patterns of max |A| and max |g| (non-negative floats
// order like their bits, so atomicMax on the bits is an order-free max).
struct DetHeader {
    unsigned max_attn_bits;
    unsigned max_g_bits;
    unsigned pad[62];
};
constexpr long long kDetHeaderBytes = 256;

// 2^F with F = 61 - e, where Q*L*K * max|A| * max|g| = f * 2^e, f in [0.5, 1):
// no element of grad_value takes more than Q*L*K contributions, each of
// magnitude <= max|A| * max|g| (bilinear weights are <= 1), so after scaling
// every partial sum stays below 2^61 (plus Q*L*K/2 of rounding), one bit of
// margin for the float rounding of the bound.  A zero bound gives F = 61; a
// non-finite one F = 0.
__device__ __forceinline__ float det_scale(const DetHeader* h, long long qlk) {
    const float bound = (float)qlk * __uint_as_float(h->max_attn_bits) * __uint_as_float(h->max_g_bits);
    int F = 61;
    if (bound > 0.f && bound <= 3.0e38f) {
        int e = 0;
        frexpf(bound, &e);
        F = 61 - e;
    } else if (!(bound == 0.f)) {
        F = 0;
    }
    F = max(-120, min(120, F));
    return ldexpf(1.f, F);
}

__device__ __forceinline__ void red_s64(long long* p, long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"((unsigned long long)v) : "memory");
}

// Deterministic scatter: each fp32 contribution times 2^F (exact) rounded once
// to an integer, summed with integer atomics (exact, so order-free).
template <int EPV>
__device__ __forceinline__ void det_scatter(long long* p, const float (&c)[EPV], float scale) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) red_s64(p + e, __float2ll_rn(c[e] * scale));
}

// ---------------------------------------------------------------------------
// element types

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <typename T>
__device__ __forceinline__ float ldg_f(const T* p) {
    return Elem<T>::to_f(__ldg(p));
}

// Unpack one 16-byte word into fp32 lanes.
__device__ __forceinline__ void unpack16(const uint4& w, float (&f)[4], const float*) {
    f[0] = __uint_as_float(w.x);
    f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z);
    f[3] = __uint_as_float(w.w);
}
__device__ __forceinline__ void unpack16(const uint4& w, float (&f)[8], const __nv_bfloat16*) {
    // bf16 -> fp32 is exact: the bf16 bits are the upper half of the binary32
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4& w, float (&f)[8], const __half*) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<const __half2*>(&u[i]);
        float2 t = __half22float2(h);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b, const __nv_bfloat16*) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, const __half*) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// EPV channels of one vector slot, T storage <-> fp32 registers: one 16-byte
// word (EPV = 16 / sizeof(T)) or one element (EPV = 1).  Loads in flight are
// kept as raw words (Raw) and widened to fp32 only when consumed.
template <typename T, int EPV>
struct Slot {
    static_assert(EPV == 1 || EPV * sizeof(T) == 16, "a slot is one element or one 16-byte word");
    using Raw = typename std::conditional<EPV == 1, T, uint4>::type;
    static __device__ __forceinline__ Raw zero() {
        if constexpr (EPV == 1) return Elem<T>::from_f(0.f);
        else return make_uint4(0u, 0u, 0u, 0u);
    }
    static __device__ __forceinline__ Raw load_raw(const T* p) {
        if constexpr (EPV == 1) return __ldg(p);
        else return __ldg(reinterpret_cast<const uint4*>(p));
    }
    static __device__ __forceinline__ void unpack(const Raw& r, float (&f)[EPV]) {
        if constexpr (EPV == 1) {
            f[0] = Elem<T>::to_f(r);
        } else {
            const T* tag = nullptr;
            unpack16(r, f, tag);
        }
    }
    static __device__ __forceinline__ void load(const T* p, float (&f)[EPV]) { unpack(load_raw(p), f); }
    static __device__ __forceinline__ void store(T* p, const float (&f)[EPV]) {
        if constexpr (EPV == 1) {
            *p = Elem<T>::from_f(f[0]);
        } else if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<uint4*>(p) = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                                      __float_as_uint(f[2]), __float_as_uint(f[3]));
        } else {
            const T* tag = nullptr;
            *reinterpret_cast<uint4*>(p) = make_uint4(pack2(f[0], f[1], tag), pack2(f[2], f[3], tag),
                                                      pack2(f[4], f[5], tag), pack2(f[6], f[7], tag));
        }
    }
};

// ---------------------------------------------------------------------------
// relaxed reductions (fire-and-forget, no ordering; course ch. 5, "sem=relaxed")

__device__ __forceinline__ void red_v4_f32(float* p, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}
__device__ __forceinline__ void red_v4_bf16x2(__nv_bfloat16* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("red.relaxed.gpu.global.add.noftz.v4.bf16x2 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ void red_v4_f16x2(__half* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("red.relaxed.gpu.global.add.noftz.v4.f16x2 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ void red_f32(float* p, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_bf16(__nv_bfloat16* p, float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    unsigned short s = *reinterpret_cast<unsigned short*>(&h);
    asm volatile("red.relaxed.gpu.global.add.noftz.bf16 [%0], %1;" ::"l"(p), "h"(s) : "memory");
}
__device__ __forceinline__ void red_f16(__half* p, float v) {
    __half h = __float2half_rn(v);
    unsigned short s = *reinterpret_cast<unsigned short*>(&h);
    asm volatile("red.relaxed.gpu.global.add.noftz.f16 [%0], %1;" ::"l"(p), "h"(s) : "memory");
}

// Add EPV fp32 contributions c[] to EPV consecutive ACC elements at p.
template <typename ACC, int EPV> struct Scatter;
template <> struct Scatter<float, 4> {
    static __device__ __forceinline__ void add(float* p, const float (&c)[4]) { red_v4_f32(p, c[0], c[1], c[2], c[3]); }
};
template <> struct Scatter<float, 8> {  // fp16/bf16 slot into the fp32 workspace
    static __device__ __forceinline__ void add(float* p, const float (&c)[8]) {
        red_v4_f32(p, c[0], c[1], c[2], c[3]);
        red_v4_f32(p + 4, c[4], c[5], c[6], c[7]);
    }
};
template <> struct Scatter<__nv_bfloat16, 8> {
    static __device__ __forceinline__ void add(__nv_bfloat16* p, const float (&c)[8]) {
        const __nv_bfloat16* t = nullptr;
        red_v4_bf16x2(p, pack2(c[0], c[1], t), pack2(c[2], c[3], t), pack2(c[4], c[5], t), pack2(c[6], c[7], t));
    }
};
template <> struct Scatter<__half, 8> {
    static __device__ __forceinline__ void add(__half* p, const float (&c)[8]) {
        const __half* t = nullptr;
        red_v4_f16x2(p, pack2(c[0], c[1], t), pack2(c[2], c[3], t), pack2(c[4], c[5], t), pack2(c[6], c[7], t));
    }
};
template <> struct Scatter<float, 1> {
    static __device__ __forceinline__ void add(float* p, const float (&c)[1]) { red_f32(p, c[0]); }
};
template <> struct Scatter<__nv_bfloat16, 1> {
    static __device__ __forceinline__ void add(__nv_bfloat16* p, const float (&c)[1]) { red_bf16(p, c[0]); }
};
template <> struct Scatter<__half, 1> {
    static __device__ __forceinline__ void add(__half* p, const float (&c)[1]) { red_f16(p, c[0]); }
};

// ---------------------------------------------------------------------------
// block prologue: level table and parameter staging

// Largest level side for which the binary32 pixel coordinate and the float
// bound checks below are exact.
constexpr long long kMaxSide = 1ll << 24;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done;
}

// Level l of the table: its sizes pass the check (1 <= H, W <= kMaxSide, the
// level inside the S rows) or it has no corner inside (ok = 0).
__device__ __forceinline__ Level level_of(const KernelArgs& a, int l) {
    const long long H = a.shapes[2 * l], W = a.shapes[2 * l + 1], st = a.starts[l];
    const bool ok = H >= 1 && W >= 1 && H <= kMaxSide && W <= kMaxSide && st >= 0 && st <= a.S && H * W <= a.S - st;
    const long long MD = (long long)a.M * a.D;
    Level v;
    v.start_md = ok ? st * MD : 0;
    v.w_md = ok ? W * MD : 0;
    v.fH = ok ? (float)H : 0.f;
    v.fW = ok ? (float)W : 0.f;
    v.ok = ok;
    v.W = ok ? (int)W : 0;
    v.start = ok ? st : 0;
    return v;
}

// Byte offset of the attention-weight chunk in the staged parameters.
template <typename T>
__device__ __forceinline__ int attn_chunk_offset(const KernelArgs& a) {
    return (a.tpb * a.LK * 2 * (int)sizeof(T) + 15) & ~15;
}

// Loads the level table into shared memory and stages the block's sampling
// parameters (loc chunk [nu*LK*2] then the attn chunk, raw dtype) into `sm`:
// thread 0 issues one-dimensional bulk copies completing on an mbarrier
// before the level loads, so the two overlap, and waits for them with a
// bounded number of polls.  Returns the block-uniform verdict (false only if
// the copy did not complete within the limit).
template <typename T>
__device__ __forceinline__ bool prologue(const KernelArgs& a, Level* lv, unsigned char* sm, uint64_t* bar,
                                         int* verdict, uint32_t u0) {
    const int tid = threadIdx.x;
    const int nu = min(a.tpb, a.n_units - (int)u0);
    const int loc_bytes = nu * a.LK * 2 * (int)sizeof(T);
    const int attn_bytes = nu * a.LK * (int)sizeof(T);
    const int attn_off = attn_chunk_offset<T>(a);
    const unsigned char* gloc = (const unsigned char*)a.loc + (long long)u0 * a.LK * 2 * (long long)sizeof(T);
    const unsigned char* gattn = (const unsigned char*)a.attn + (long long)u0 * a.LK * (long long)sizeof(T);
    const uint32_t b = smem_u32(bar);
    if (a.param_mode == PARAMS_SMEM_BULK) {
        // both global ranges and both sizes are multiples of 16 bytes (host check)
        if (tid == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b));
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b),
                         "r"((uint32_t)(loc_bytes + attn_bytes))
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(sm)),
                "l"(gloc), "r"((uint32_t)loc_bytes), "r"(b)
                : "memory");
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(sm + attn_off)),
                "l"(gattn), "r"((uint32_t)attn_bytes), "r"(b)
                : "memory");
        }
    } else if (a.param_mode == PARAMS_SMEM_LD) {
        const T* s1 = reinterpret_cast<const T*>(gloc);
        T* d1 = reinterpret_cast<T*>(sm);
        for (int i = tid; i < nu * a.LK * 2; i += blockDim.x) d1[i] = __ldg(s1 + i);
        const T* s2 = reinterpret_cast<const T*>(gattn);
        T* d2 = reinterpret_cast<T*>(sm + attn_off);
        for (int i = tid; i < nu * a.LK; i += blockDim.x) d2[i] = __ldg(s2 + i);
    }
    if (tid < a.L) {
        lv[tid] = level_of(a, tid);
        if (!lv[tid].ok) atomicOr(a.err, kErrBadLevel);
    }
    if (a.param_mode == PARAMS_SMEM_BULK && tid == 0) {
        uint32_t done = 0;
        for (int it = 0; it < (1 << 22) && !done; ++it) done = mbar_try_wait(b, 0);
        *verdict = (int)done;
        // a copy still in flight gets a second bounded wait before the block exits
        for (int it = 0; it < (1 << 22) && !done; ++it) done = mbar_try_wait(b, 0);
    }
    __syncthreads();
    return a.param_mode != PARAMS_SMEM_BULK || *verdict != 0;
}

// Bilinear setup of one sampling point (course ch. 4, "Bilinear sampling";
// README, "Kernel design": x_im = x * W_l - 0.5, zero padding).  Off is the
// offset type inside one [S, M, D] slice: int when the slice has < 2^31
// elements, else long long.
template <typename Off>
struct Corners {
    Off off[4];   // element offsets of (y0,x0), (y0,x0+1), (y0+1,x0), (y0+1,x0+1)
    float w[4];   // bilinear weights of the four corners
    bool ok[4];   // corner inside the level
    float lx, ly;
};

template <typename Off>
__device__ __forceinline__ void bilinear_setup(const Level& L, float x, float y, int MD, Corners<Off>& cr) {
    // binary32 pixel coordinate, one rounding of x * W - 0.5
    const float xi = __fmaf_rn(x, L.fW, -0.5f);
    const float yi = __fmaf_rn(y, L.fH, -0.5f);
    const float x0f = floorf(xi), y0f = floorf(yi);
    const float lx = xi - x0f, ly = yi - y0f;
    // comparisons are false for NaN: a non-finite location has no corner inside
    const bool vx0 = L.ok && x0f >= 0.f && x0f < L.fW;
    const bool vx1 = L.ok && x0f >= -1.f && x0f < L.fW - 1.f;
    const bool vy0 = y0f >= 0.f && y0f < L.fH;
    const bool vy1 = y0f >= -1.f && y0f < L.fH - 1.f;
    const int x0 = (vx0 || vx1) ? (int)x0f : 0;
    const int y0 = (vy0 || vy1) ? (int)y0f : 0;
    const Off o = (Off)L.start_md + (Off)y0 * (Off)L.w_md + (Off)x0 * (Off)MD;
    cr.off[0] = o;
    cr.off[1] = o + MD;
    cr.off[2] = o + (Off)L.w_md;
    cr.off[3] = o + (Off)L.w_md + MD;
    cr.ok[0] = vy0 && vx0;
    cr.ok[1] = vy0 && vx1;
    cr.ok[2] = vy1 && vx0;
    cr.ok[3] = vy1 && vx1;
    const float hx = 1.f - lx, hy = 1.f - ly;
    cr.w[0] = hx * hy;
    cr.w[1] = lx * hy;
    cr.w[2] = hx * ly;
    cr.w[3] = lx * ly;
    cr.lx = lx;
    cr.ly = ly;
}

template <typename T>
__device__ __forceinline__ void read_params(const KernelArgs& a, const unsigned char* sm, bool staged, int team,
                                            uint32_t u, int s, float& x, float& y, float& w) {
    if (staged) {
        const T* pl = reinterpret_cast<const T*>(sm) + (team * a.LK + s) * 2;
        const T* pa = reinterpret_cast<const T*>(sm + attn_chunk_offset<T>(a)) + team * a.LK + s;
        x = Elem<T>::to_f(pl[0]);
        y = Elem<T>::to_f(pl[1]);
        w = Elem<T>::to_f(pa[0]);
    } else {
        const long long ps = (long long)u * a.LK + s;
        const T* pl = reinterpret_cast<const T*>(a.loc) + 2 * ps;
        x = ldg_f(pl);
        y = ldg_f(pl + 1);
        w = ldg_f(reinterpret_cast<const T*>(a.attn) + ps);
    }
}

template <typename T>
__device__ __forceinline__ float read_weight(const KernelArgs& a, const unsigned char* sm, bool staged, int team,
                                             uint32_t u, int s) {
    if (staged)
        return Elem<T>::to_f(reinterpret_cast<const T*>(sm + attn_chunk_offset<T>(a))[team * a.LK + s]);
    return ldg_f(reinterpret_cast<const T*>(a.attn) + (long long)u * a.LK + s);
}

// Team geometry of this thread.
struct Lane {
    int C, P, TP, team, c, p;
    uint32_t u0, u;
    bool active;
};
__device__ __forceinline__ Lane lane_of(const KernelArgs& a, uint32_t blk) {
    Lane r;
    const int lcp = a.lc + a.lp;
    r.C = 1 << a.lc;
    r.P = 1 << a.lp;
    r.TP = 1 << lcp;
    r.team = threadIdx.x >> lcp;
    const int lt = threadIdx.x & (r.TP - 1);
    r.c = lt & (r.C - 1);
    r.p = lt >> a.lc;
    r.u0 = blk * (uint32_t)a.tpb;
    r.u = r.u0 + r.team;
    r.active = r.u < (uint32_t)a.n_units;
    return r;
}
__device__ __forceinline__ Lane lane_of(const KernelArgs& a) { return lane_of(a, blockIdx.x); }

// ---------------------------------------------------------------------------
// forward (course ch. 4; README "Kernel design" item 1)

template <typename T, int NV, int EPV, bool WIDE, int U>
__global__ void __launch_bounds__(kBlockThreads) msda_fwd_kernel(const KernelArgs a) {
    using Off = typename std::conditional<WIDE, long long, int>::type;
    using S_ = Slot<T, EPV>;
    __shared__ Level lv[MSDA_MAX_LEVELS];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int verdict;
    extern __shared__ __align__(16) unsigned char sm[];

    // launched as a programmatic dependent: wait for the kernel ahead of it
    // (which may have written its inputs) before reading anything; launched
    // normally, the wait returns at once
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const Lane ln = lane_of(a);
    if (!prologue<T>(a, lv, sm, &bar, &verdict, ln.u0)) {
        if (threadIdx.x == 0) atomicOr(a.err, kErrBulkTimeout);
        return;  // nothing was written; the host reports the error bit
    }
    const bool staged = a.param_mode != PARAMS_DIRECT;
    const uint32_t b = fdiv(ln.u, a.div_qm);
    const uint32_t m = ln.u - fdiv(ln.u, a.div_m) * (uint32_t)a.M;
    const T* vbase = reinterpret_cast<const T*>(a.value) + (long long)b * a.slice + (long long)m * a.D;
    const int MD = a.M * a.D;

    float acc[NV][EPV];
#pragma unroll
    for (int n = 0; n < NV; ++n)
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[n][e] = 0.f;

    for (int s0 = 0; s0 < a.LK; s0 += ln.P * U) {
        typename S_::Raw vals[U][4][NV];
        float coef[U][4];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int s = s0 + ln.p + i * ln.P;
            const bool live = ln.active && s < a.LK;
            float x = -4.f, y = -4.f, w = 0.f;
            int l = 0;
            if (live) {
                read_params<T>(a, sm, staged, ln.team, ln.u, s, x, y, w);
                l = (int)fdiv((uint32_t)s, a.div_k);
            }
            Level lev = lv[l];
            if (!live) lev.ok = 0;
            Corners<Off> cr;
            bilinear_setup<Off>(lev, x, y, MD, cr);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                coef[i][k] = cr.ok[k] ? w * cr.w[k] : 0.f;
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    const int j = n * ln.C + ln.c;
                    vals[i][k][n] = (cr.ok[k] && j < a.nvec) ? S_::load_raw(vbase + cr.off[k] + j * EPV) : S_::zero();
                }
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    float v[EPV];
                    S_::unpack(vals[i][k][n], v);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) acc[n][e] = fmaf(coef[i][k], v[e], acc[n][e]);
                }
    }

    // combine the P point lanes of the team
    for (int o = ln.C; o < ln.TP; o <<= 1) {
#pragma unroll
        for (int n = 0; n < NV; ++n)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[n][e] += __shfl_xor_sync(0xffffffffu, acc[n][e], o);
    }
    if (ln.active && ln.p == 0) {
        T* o = reinterpret_cast<T*>(a.out) + (long long)ln.u * a.D;
#pragma unroll
        for (int n = 0; n < NV; ++n) {
            const int j = n * ln.C + ln.c;
            if (j < a.nvec) S_::store(o + j * EPV, acc[n]);
        }
    }
}

// ---------------------------------------------------------------------------
// backward (course ch. 5; README "Kernel design" items 2, 3)

template <typename T, typename ACC, int NV, int EPV, bool WIDE, int U>
__global__ void __launch_bounds__(kBlockThreads) msda_bwd_kernel(const KernelArgs a) {
    using Off = typename std::conditional<WIDE, long long, int>::type;
    using S_ = Slot<T, EPV>;
    __shared__ Level lv[MSDA_MAX_LEVELS];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int verdict;
    extern __shared__ __align__(16) unsigned char sm[];

    const Lane ln = lane_of(a);
    if (!prologue<T>(a, lv, sm, &bar, &verdict, ln.u0)) {
        if (threadIdx.x == 0) atomicOr(a.err, kErrBulkTimeout);
        return;
    }
    const bool staged = a.param_mode != PARAMS_DIRECT;
    const uint32_t b = fdiv(ln.u, a.div_qm);
    const uint32_t m = ln.u - fdiv(ln.u, a.div_m) * (uint32_t)a.M;
    const long long vofs = (long long)b * a.slice + (long long)m * a.D;
    const T* vbase = reinterpret_cast<const T*>(a.value) + vofs;
    ACC* gbase = reinterpret_cast<ACC*>(a.grad_acc) + vofs;
    const int MD = a.M * a.D;

    // this lane's slots of g = grad_out[b, q, m, :]
    float g[NV][EPV];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        const int j = n * ln.C + ln.c;
        if (ln.active && j < a.nvec) {
            S_::load(reinterpret_cast<const T*>(a.grad_out) + (long long)ln.u * a.D + j * EPV, g[n]);
        } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) g[n][e] = 0.f;
        }
    }

    T* gl = reinterpret_cast<T*>(a.grad_loc);
    T* ga = reinterpret_cast<T*>(a.grad_attn);
    float dscale = 0.f;
    if constexpr (std::is_same<ACC, long long>::value) dscale = det_scale(a.det, (long long)a.Q * a.LK);

    for (int s0 = 0; s0 < a.LK; s0 += ln.P * U) {
        typename S_::Raw vals[U][4][NV];
        Corners<Off> cr[U];
        float wa[U], fW[U], fH[U];
        bool live[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int s = s0 + ln.p + i * ln.P;
            live[i] = ln.active && s < a.LK;
            float x = -4.f, y = -4.f, w = 0.f;
            int l = 0;
            if (live[i]) {
                read_params<T>(a, sm, staged, ln.team, ln.u, s, x, y, w);
                l = (int)fdiv((uint32_t)s, a.div_k);
            }
            Level lev = lv[l];
            if (!live[i]) lev.ok = 0;
            bilinear_setup<Off>(lev, x, y, MD, cr[i]);
            wa[i] = w;
            fW[i] = lev.fW;
            fH[i] = lev.fH;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    const int j = n * ln.C + ln.c;
                    vals[i][k][n] = (cr[i].ok[k] && j < a.nvec) ? S_::load_raw(vbase + cr[i].off[k] + j * EPV)
                                                                : S_::zero();
                }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            // per-lane partial <g, v_corner> over this lane's channels
            float d[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float t = 0.f;
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    float v[EPV];
                    S_::unpack(vals[i][k][n], v);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) t = fmaf(g[n][e], v[e], t);
                }
                d[k] = t;
            }
            const bool any = cr[i].ok[0] || cr[i].ok[1] || cr[i].ok[2] || cr[i].ok[3];
            const float lx = cr[i].lx, ly = cr[i].ly;
            // <g, sampled>, <g, d sampled / d x_im>, <g, d sampled / d y_im>
            float r_a = any ? (cr[i].w[0] * d[0] + cr[i].w[1] * d[1] + cr[i].w[2] * d[2] + cr[i].w[3] * d[3]) : 0.f;
            float r_x = any ? ((1.f - ly) * (d[1] - d[0]) + ly * (d[3] - d[2])) : 0.f;
            float r_y = any ? ((1.f - lx) * (d[2] - d[0]) + lx * (d[3] - d[1])) : 0.f;
            for (int o = 1; o < ln.C; o <<= 1) {
                r_a += __shfl_xor_sync(0xffffffffu, r_a, o);
                r_x += __shfl_xor_sync(0xffffffffu, r_x, o);
                r_y += __shfl_xor_sync(0xffffffffu, r_y, o);
            }
            const int s = s0 + ln.p + i * ln.P;
            if (live[i] && ln.c == 0) {
                const long long ps = (long long)ln.u * a.LK + s;
                ga[ps] = Elem<T>::from_f(r_a);
                gl[2 * ps] = Elem<T>::from_f(wa[i] * fW[i] * r_x);
                gl[2 * ps + 1] = Elem<T>::from_f(wa[i] * fH[i] * r_y);
            }
            // grad_value scatter: A * w_corner * g into the inside corners
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (!cr[i].ok[k]) continue;
                const float cf = wa[i] * cr[i].w[k];
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    const int j = n * ln.C + ln.c;
                    if (j < a.nvec) {
                        float t[EPV];
#pragma unroll
                        for (int e = 0; e < EPV; ++e) t[e] = cf * g[n][e];
                        if constexpr (std::is_same<ACC, long long>::value)
                            det_scatter<EPV>(gbase + cr[i].off[k] + j * EPV, t, dscale);
                        else
                            Scatter<ACC, EPV>::add(gbase + cr[i].off[k] + j * EPV, t);
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Specialised kernels for rows of whole 16-byte vectors: C = 4 channel lanes
// with NV vectors each (D = 32 * NV bf16/fp16 or 16 * NV fp32 channels),
// 32-bit slice offsets, runtime P.
//
// One bilinear setup per sample.  The samples of a unit are taken in rounds
// of 4P; in a round starting at r0 the lane (c, p) of a team sets up sample
// r0 + p + c*P, and the four channel lanes of point group p take it in turn
// (iteration j uses the setup of lane (j, p)), reading it with warp shuffles
// instead of recomputing it.  The producer lane also writes that sample's
// grad_attn / grad_loc, since it holds the level sizes and the weight.

constexpr int kC = 4;

struct SampleSetup {
    int o;          // element offset of corner (y0, x0) in the slice
    int wmd;        // W * M * D of the sample's level
    unsigned mask;  // bit k: corner k inside the level
    float lx, ly;   // fractional offsets in the cell
    int pix;        // pyramid row (pixel) of corner (y0, x0); not carried by shfl_setup
};

__device__ __forceinline__ SampleSetup sample_setup(const Level& L, float x, float y, int MD) {
    // binary32 pixel coordinate, one rounding of x * W - 0.5 (as bilinear_setup)
    const float xi = __fmaf_rn(x, L.fW, -0.5f);
    const float yi = __fmaf_rn(y, L.fH, -0.5f);
    const float x0f = floorf(xi), y0f = floorf(yi);
    const bool vx0 = L.ok && x0f >= 0.f && x0f < L.fW;
    const bool vx1 = L.ok && x0f >= -1.f && x0f < L.fW - 1.f;
    const bool vy0 = y0f >= 0.f && y0f < L.fH;
    const bool vy1 = y0f >= -1.f && y0f < L.fH - 1.f;
    const int x0 = (vx0 || vx1) ? (int)x0f : 0;
    const int y0 = (vy0 || vy1) ? (int)y0f : 0;
    SampleSetup r;
    r.wmd = (int)L.w_md;
    r.o = (int)L.start_md + y0 * r.wmd + x0 * MD;
    r.mask = (unsigned)(vy0 && vx0) | ((unsigned)(vy0 && vx1) << 1) | ((unsigned)(vy1 && vx0) << 2) |
             ((unsigned)(vy1 && vx1) << 3);
    r.lx = xi - x0f;
    r.ly = yi - y0f;
    r.pix = (int)L.start + y0 * L.W + x0;
    return r;
}

__device__ __forceinline__ SampleSetup shfl_setup(const SampleSetup& s, int src) {
    SampleSetup r;
    r.o = __shfl_sync(0xffffffffu, s.o, src);
    r.wmd = __shfl_sync(0xffffffffu, s.wmd, src);
    r.mask = __shfl_sync(0xffffffffu, s.mask, src);
    r.lx = __shfl_sync(0xffffffffu, s.lx, src);
    r.ly = __shfl_sync(0xffffffffu, s.ly, src);
    r.pix = 0;
    return r;
}

// bilinear weights of the four corners
__device__ __forceinline__ void corner_weights(float lx, float ly, float (&w)[4]) {
    const float hx = 1.f - lx, hy = 1.f - ly;
    w[0] = hx * hy;
    w[1] = lx * hy;
    w[2] = hx * ly;
    w[3] = lx * ly;
}

// acc[e] += c * v[e] on pairs of lanes with the packed fp32x2 FMA
template <int EPV>
__device__ __forceinline__ void axpy2(float (&acc)[EPV], float c, const float (&v)[EPV]) {
    const float2 cc = make_float2(c, c);
#pragma unroll
    for (int e = 0; e < EPV; e += 2) {
        float2 r = __ffma2_rn(cc, make_float2(v[e], v[e + 1]), make_float2(acc[e], acc[e + 1]));
        acc[e] = r.x;
        acc[e + 1] = r.y;
    }
}

// sum over e of g[e] * v[e], pairwise then folded
template <int EPV>
__device__ __forceinline__ float dot2(const float (&g)[EPV], const float (&v)[EPV]) {
    float2 t = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < EPV; e += 2) t = __ffma2_rn(make_float2(g[e], g[e + 1]), make_float2(v[e], v[e + 1]), t);
    return t.x + t.y;
}

// Samples whose corners a lane loads in one batch before using them.
// Measured on GB300: in the forward, all four samples of a round for one
// 16-byte slot per lane (encoder forward 122 -> 111 us), else two; the
// fused forward keeps two (four: decoder 12.7 -> 16.1 us, encoder
// 129 -> 150 us, its per-sample location and softmax work in between); in the
// backward, two for every slot count: four slowed the encoder backward
// (344 -> 367 us), and one halved the registers at three slots but slowed
// the fp32 D=48 backward (211 -> 248 us).  Loads in flight per lane matter
// more than occupancy here.
template <int NV, bool FUSED>
constexpr int kGatherBatchFwd = (NV == 1 && !FUSED) ? 4 : 2;
constexpr int kGatherBatchBwd = 2;

// Channels [0, 4) and [16, 20) from p (16-bit elements, 8-byte aligned), as
// one 16-byte word in that order.
template <typename T>
__device__ __forceinline__ uint4 split_load_raw(const T* p) {
    static_assert(sizeof(T) == 2, "split slots hold 16-bit elements");
    const uint2 lo = __ldg(reinterpret_cast<const uint2*>(p));
    const uint2 hi = __ldg(reinterpret_cast<const uint2*>(p + 16));
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

// Lane index (within the warp) of lane (c, p) of this thread's team.
__device__ __forceinline__ int team_lane(const Lane& ln, int c, int p) {
    return ((threadIdx.x & 31) & ~(ln.TP - 1)) + c + p * kC;
}

// Fused operator (msda-triton README, "The operator": softmax-normalised
// weights over the L*K (level, point) pairs, locations = reference point plus
// offset).  Offsets are in pixels of the sample's level: loc = ref + off / W
// (x) and ref + off / H (y), one binary32 rounding per operation.

// max and sum of exp(logit - max) over the unit's L*K logits, reduced over
// the team (all lanes of the warp take part; inactive teams get (0, 1))
template <typename T>
__device__ __forceinline__ void softmax_stats(const KernelArgs& a, const unsigned char* sm, bool staged,
                                              const Lane& ln, float& mx, float& sum) {
    const int lt = ln.c + ln.p * ln.C;
    float m = -INFINITY;
    if (ln.active)
        for (int s = lt; s < a.LK; s += ln.TP) m = fmaxf(m, read_weight<T>(a, sm, staged, ln.team, ln.u, s));
    for (int o = 1; o < ln.TP; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float t = 0.f;
    if (ln.active)
        for (int s = lt; s < a.LK; s += ln.TP) t += expf(read_weight<T>(a, sm, staged, ln.team, ln.u, s) - m);
    for (int o = 1; o < ln.TP; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    mx = ln.active ? m : 0.f;
    sum = ln.active ? t : 1.f;
}

// location of a fused sample from its offset (x, y in pixels) and the
// reference point of (b*Q + q, level l)
template <typename T>
__device__ __forceinline__ void fused_location(const KernelArgs& a, uint32_t bq, int l, const Level& lev, float& x,
                                               float& y) {
    const T* rp = reinterpret_cast<const T*>(a.ref) + ((long long)bq * a.L + l) * 2;
    x = __fadd_rn(ldg_f(rp), __fdiv_rn(x, lev.fW));
    y = __fadd_rn(ldg_f(rp + 1), __fdiv_rn(y, lev.fH));
}

template <typename T, int NV, bool FUSED>
__global__ void __launch_bounds__(kBlockThreads) msda_fwd4_kernel(const KernelArgs a) {
    constexpr int EPV = 16 / sizeof(T);
    constexpr int JB = kGatherBatchFwd<NV, FUSED>;
    using S_ = Slot<T, EPV>;
    __shared__ Level lv[MSDA_MAX_LEVELS];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int verdict;
    extern __shared__ __align__(16) unsigned char sm[];

    // Launched as a programmatic dependent, this grid may start before the
    // kernel ahead of it (which may have written its inputs) has finished:
    // wait for it before reading anything.  Launched normally, the wait
    // returns at once.  The grid never lets the next kernel launch early:
    // measured on GB300, an early trigger gained nothing for the core
    // forward and cost the fused decoder step 13 us (its dependents' waiting
    // blocks hold SM slots); the next kernel's own programmatic launch still
    // overlaps this grid's completion.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const Lane ln = lane_of(a);
    if (!prologue<T>(a, lv, sm, &bar, &verdict, ln.u0)) {
        if (threadIdx.x == 0) atomicOr(a.err, kErrBulkTimeout);
        return;
    }
    const bool staged = a.param_mode != PARAMS_DIRECT;
    const uint32_t b = fdiv(ln.u, a.div_qm);
    const uint32_t m = ln.u - fdiv(ln.u, a.div_m) * (uint32_t)a.M;
    const T* vbase = reinterpret_cast<const T*>(a.value) + (long long)b * a.slice + (long long)m * a.D + ln.c * EPV;
    const int MD = a.M * a.D;
    float smx = 0.f, ssum = 1.f;
    if constexpr (FUSED) softmax_stats<T>(a, sm, staged, ln, smx, ssum);

    float acc[NV][EPV];
#pragma unroll
    for (int n = 0; n < NV; ++n)
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[n][e] = 0.f;

    for (int r0 = 0; r0 < a.LK; r0 += ln.TP) {
        // this lane's sample of the round
        const int s_own = r0 + ln.p + ln.c * ln.P;
        const bool live = ln.active && s_own < a.LK;
        float x = -4.f, y = -4.f, w = 0.f;
        int l = 0;
        if (live) {
            read_params<T>(a, sm, staged, ln.team, ln.u, s_own, x, y, w);
            l = (int)fdiv((uint32_t)s_own, a.div_k);
        }
        Level lev = lv[l];
        if (!live) lev.ok = 0;
        if constexpr (FUSED) {
            if (live) {
                fused_location<T>(a, fdiv(ln.u, a.div_m), l, lev, x, y);
                w = expf(w - smx) / ssum;
            }
        }
        SampleSetup me = sample_setup(lev, x, y, MD);
        float mw[4];
        corner_weights(me.lx, me.ly, mw);
        float mc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mc[k] = ((me.mask >> k) & 1u) ? w * mw[k] : 0.f;

#pragma unroll
        for (int j0 = 0; j0 < kC; j0 += JB) {
            typename S_::Raw raw[JB][4][NV];
            float cf[JB][4];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                const int src = team_lane(ln, j0 + jj, ln.p);
                const int o = __shfl_sync(0xffffffffu, me.o, src);
                const int wmd = __shfl_sync(0xffffffffu, me.wmd, src);
                const unsigned mask = __shfl_sync(0xffffffffu, me.mask, src);
#pragma unroll
                for (int k = 0; k < 4; ++k) cf[jj][k] = __shfl_sync(0xffffffffu, mc[k], src);
                const int off[4] = {o, o + MD, o + wmd, o + wmd + MD};
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int n = 0; n < NV; ++n)
                        raw[jj][k][n] = ((mask >> k) & 1u) ? S_::load_raw(vbase + off[k] + n * kC * EPV) : S_::zero();
            }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj)
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int n = 0; n < NV; ++n) {
                        float v[EPV];
                        S_::unpack(raw[jj][k][n], v);
                        axpy2(acc[n], cf[jj][k], v);
                    }
        }
    }

    // combine the P point lanes of the team
    for (int o = kC; o < ln.TP; o <<= 1) {
#pragma unroll
        for (int n = 0; n < NV; ++n)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[n][e] += __shfl_xor_sync(0xffffffffu, acc[n][e], o);
    }
    if (ln.active && ln.p == 0) {
        T* o = reinterpret_cast<T*>(a.out) + (long long)ln.u * a.D + ln.c * EPV;
#pragma unroll
        for (int n = 0; n < NV; ++n) S_::store(o + n * kC * EPV, acc[n]);
    }
}

// ---------------------------------------------------------------------------
// Touch classes of the FP32 workspace's rows (course ch. 5, "The fix:
// accumulate in FP32, downcast at the end": the sum of one contribution,
// rounded once, is that contribution rounded once).
//
// A level is sparse when its rows take few corner contributions: the 4*Q*K
// corners of one (b, m) image over its H*W rows, at most touch_tau a row on
// average.  For the large levels of a big pyramid most touched rows then
// take exactly one contribution (for uniformly spread samples a fraction
// e^-r of the rows is untouched and r*e^-r touched once, r = 4QK/HW), and
// going through the workspace costs such a row a line fetch, a write-back
// and a read by the rounding, where writing it directly costs one store.
// A count pass before the sampling passes gives every row of the sparse
// levels its class (0, 1 or 2 = several); the sampling pass then stores a
// class-1 row's contribution to grad_value, rounded once, and reduces the
// others into the workspace; rounding skips class-1 rows and writes zeros
// for class-0 rows without reading the workspace.

__device__ __forceinline__ bool touch_sparse(const KernelArgs& a, const Level& L) {
    return L.ok && 4ll * a.Q * a.K <= (long long)a.touch_tau * (long long)L.fH * (long long)L.W;
}

// Class index of (image b, pixel, head m): (b*M + m)*S + pixel (< 2^31, host
// check), head-major so that horizontally adjacent corners are adjacent
// classes, mostly in one word.
__device__ __forceinline__ unsigned touch_row(const KernelArgs& a, uint32_t b, int pix, uint32_t m) {
    return ((unsigned)b * (unsigned)a.M + m) * (unsigned)a.S + (unsigned)pix;
}

__device__ __forceinline__ unsigned touch_bits(unsigned word, unsigned row) { return (word >> ((row & 15u) * 2u)) & 3u; }

// grad_value[p..p+3] = (a, b, c, d), rounded once (8-byte aligned p)
template <typename T>
__device__ __forceinline__ void store4(T* p, float a, float b, float c, float d) {
    const T* tag = nullptr;
    *reinterpret_cast<uint2*>(p) = make_uint2(pack2(a, b, tag), pack2(c, d, tag));
}

// The count pass: one thread per sample (samples of dense levels return at
// once).  A corner row's low bit is set by an atomic OR; a row whose low bit
// was already set gets the high bit too.  The four ORs of a sample are
// issued before any of their old values is used.  The bilinear setup is
// sample_setup's, as in the sampling pass, so both see the same corners.
template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_touch_count_kernel(const KernelArgs a) {
    __shared__ Level lv[MSDA_MAX_LEVELS];
    __shared__ int sparse[MSDA_MAX_LEVELS];
    if (threadIdx.x < a.L) {
        lv[threadIdx.x] = level_of(a, threadIdx.x);
        sparse[threadIdx.x] = touch_sparse(a, lv[threadIdx.x]);
    }
    __syncthreads();
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (uint32_t)a.n_units * (uint32_t)a.LK) return;
    const uint32_t u = fdiv(i, a.div_lk);
    const int s = (int)(i - u * (uint32_t)a.LK);
    const int l = (int)fdiv((uint32_t)s, a.div_k);
    if (!sparse[l]) return;
    const T* pl = reinterpret_cast<const T*>(a.loc) + 2ll * i;
    const SampleSetup st = sample_setup(lv[l], ldg_f(pl), ldg_f(pl + 1), a.M * a.D);
    if (!st.mask) return;
    const uint32_t b = fdiv(u, a.div_qm);
    const uint32_t m = u - fdiv(u, a.div_m) * (uint32_t)a.M;
    // corners (0, 1) and (2, 3) are adjacent classes: one OR per word
    const unsigned r0 = touch_row(a, b, st.pix, m), r2 = r0 + (unsigned)lv[l].W;
    const unsigned rows[4] = {r0, r0 + 1u, r2, r2 + 1u};
    unsigned* w[4];
    unsigned bit[4], old[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        w[k] = a.touch + (rows[k] >> 4);
        bit[k] = ((st.mask >> k) & 1u) << ((rows[k] & 15u) * 2u);
    }
#pragma unroll
    for (int k = 0; k < 4; k += 2)
        if (w[k] == w[k + 1]) {   // the pair in one word
            bit[k] |= bit[k + 1];
            bit[k + 1] = 0u;
        }
#pragma unroll
    for (int k = 0; k < 4; ++k) old[k] = bit[k] ? atomicOr(w[k], bit[k]) : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (old[k] & bit[k]) atomicOr(w[k], (old[k] & bit[k]) << 1);
}

// Row ranges [begin, end) of the sparse levels in one image's rows
// (pixel * M + m), in shared memory for the rounding kernels.
struct TouchRanges {
    unsigned begin[MSDA_MAX_LEVELS], end[MSDA_MAX_LEVELS];
    int n;
};

__device__ __forceinline__ void touch_ranges(const KernelArgs& a, TouchRanges* r) {
    if (threadIdx.x == 0) {
        int n = 0;
        for (int l = 0; l < a.L; ++l) {
            const Level v = level_of(a, l);
            if (!touch_sparse(a, v)) continue;
            r->begin[n] = (unsigned)v.start * (unsigned)a.M;
            r->end[n] = (unsigned)(v.start + (long long)v.fH * v.W) * (unsigned)a.M;
            ++n;
        }
        r->n = n;
    }
    __syncthreads();
}

// Eight workspace elements from index 8*i: rounded once into grad_value; with
// rezero, the 32 bytes written back as zeros when any of them is non-zero.
template <typename T>
__device__ __forceinline__ void round8(float* ws, T* gv, long long i, int rezero) {
    float4* s = reinterpret_cast<float4*>(ws);
    const float4 x = __ldcs(s + 2 * i);
    const float4 y = __ldcs(s + 2 * i + 1);
    const float f[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
    Slot<T, 8>::store(gv + 8 * i, f);
    if (rezero) {
        const uint32_t nz = __float_as_uint(x.x) | __float_as_uint(x.y) | __float_as_uint(x.z) | __float_as_uint(x.w) |
                            __float_as_uint(y.x) | __float_as_uint(y.y) | __float_as_uint(y.z) | __float_as_uint(y.w);
        if (nz) {
            __stcs(s + 2 * i, make_float4(0.f, 0.f, 0.f, 0.f));
            __stcs(s + 2 * i + 1, make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
}

// The first pyramid row of the levels >= l0 that pass the shape check (S if
// none): rows below it receive nothing from those levels.
__device__ __forceinline__ long long first_row_from(const KernelArgs& a, int l0) {
    long long p = a.S;
    for (int l = l0; l < a.L; ++l) {
        const long long H = a.shapes[2 * l], W = a.shapes[2 * l + 1], st = a.starts[l];
        const bool ok = H >= 1 && W >= 1 && H <= kMaxSide && W <= kMaxSide && st >= 0 && st <= a.S &&
                        H * W <= a.S - st;
        if (ok && st < p) p = st;
    }
    return p;
}

// round8 under the touch classes: group i (eight elements) of image img.  A
// row of a sparse level with one contribution already holds it in grad_value;
// one with none gets zeros, its workspace row unread.
template <typename T>
__device__ __forceinline__ void round8_touch(const KernelArgs& a, const TouchRanges& tr, float* ws, T* gv,
                                             long long i, unsigned img) {
    static_assert(sizeof(T) == 2, "eight 16-bit elements are one 16-byte store");
    const unsigned row = fdiv((uint32_t)i, a.div_d8);
    bool sp = false;
    for (int j = 0; j < tr.n; ++j) sp |= row >= tr.begin[j] && row < tr.end[j];
    if (sp) {
        const unsigned pix = fdiv(row, a.div_m);
        const unsigned id = (img * (unsigned)a.M + (row - pix * (unsigned)a.M)) * (unsigned)a.S + pix;
        const unsigned c = touch_bits(__ldg(a.touch + (id >> 4)), id);
        if (c == 1u) return;
        if (c == 0u) {
            *reinterpret_cast<uint4*>(gv + 8 * i) = make_uint4(0u, 0u, 0u, 0u);
            return;
        }
    }
    round8<T>(ws, gv, i, a.conv_rezero);
}

// One folded chunk: workspace elements [k*conv_chunk, (k+1)*conv_chunk) of
// batch image img, cut at the first row of the levels >= conv_level.
template <typename T>
__device__ __noinline__ void fold_round_chunk(const KernelArgs& a, long long c) {
    __shared__ long long cut;
    __shared__ TouchRanges tr;
    if (threadIdx.x == 0) cut = first_row_from(a, a.conv_level) * a.M * a.D;
    if (a.touch) touch_ranges(a, &tr);
    else __syncthreads();
    const long long img = c / a.conv_chunks_per_image, k = c - img * a.conv_chunks_per_image;
    const long long e0 = k * a.conv_chunk, e1 = min(e0 + a.conv_chunk, cut);
    float* ws = reinterpret_cast<float*>(a.grad_acc) + img * a.slice;
    T* gv = reinterpret_cast<T*>(a.conv_out) + img * a.slice;
    if (a.touch) {
        for (long long i = e0 / 8 + threadIdx.x; i < e1 / 8; i += blockDim.x)
            round8_touch<T>(a, tr, ws, gv, i, (unsigned)img);
    } else {
        for (long long i = e0 / 8 + threadIdx.x; i < e1 / 8; i += blockDim.x) round8<T>(ws, gv, i, a.conv_rezero);
    }
}

// Backward, same decomposition.  Each round first gathers the corners of its
// samples and reduces <g, corner> to grad_attn / grad_loc (reads only), then
// scatters grad_value.  When launched as a programmatic dependent of the
// zero kernel, griddepcontrol.wait before the first scatter lets the gather
// phase of the first round overlap the zeroing of grad_value; launched
// normally, the wait returns at once.
// MERGE: 0 none, kMergeCells whole cells only, kMergeCorners every shared corner;
// kGatherOnly: no scatter at all (grad_attn / grad_loc only; grad_value is
// accumulated on chip by the tiled passes of msda_tiled.cuh).
constexpr int kMergeCells = 1;
constexpr int kMergeCorners = 2;
constexpr int kGatherOnly = -1;

template <typename T, typename ACC, int NV, bool FUSED, int MERGE, bool TOUCH>
__device__ __forceinline__ void bwd4_body(const KernelArgs& a) {
    constexpr int EPV = 16 / sizeof(T);
    constexpr int JB = kGatherBatchBwd;
    using S_ = Slot<T, EPV>;
    __shared__ Level lv[MSDA_MAX_LEVELS];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int verdict;
    extern __shared__ __align__(16) unsigned char sm[];

    // Blocks that round finished workspace rows instead of sampling (the
    // rounding pass folded into this launch; see KernelArgs::conv_blocks):
    // every conv_every-th block, so they run alongside the sampling blocks.
    uint32_t blk = blockIdx.x;
    if constexpr (std::is_same<ACC, float>::value && sizeof(T) == 2 && !FUSED) {
        if (a.conv_blocks > 0) {
            const uint32_t R = (uint32_t)a.conv_every;
            if (blk % R == R - 1 && blk / R < (uint32_t)a.conv_blocks) {
                fold_round_chunk<T>(a, a.conv_first + blk / R);
                return;
            }
            blk -= min((blk + 1) / R, (uint32_t)a.conv_blocks);
        }
    }
    const Lane ln = lane_of(a, blk);
    if (!prologue<T>(a, lv, sm, &bar, &verdict, ln.u0)) {
        if (threadIdx.x == 0) atomicOr(a.err, kErrBulkTimeout);
        return;
    }
    const bool staged = a.param_mode != PARAMS_DIRECT;
    const uint32_t b = fdiv(ln.u, a.div_qm);
    const uint32_t m = ln.u - fdiv(ln.u, a.div_m) * (uint32_t)a.M;
    // Lane channels.  A lane owns EPV channels of each group of kC * EPV:
    // normally the 16-byte slot [c*EPV, c*EPV + EPV).  A 16-bit value
    // accumulated into the fp32 workspace splits the slot instead: channels
    // [4c, 4c+4) and [16+4c, 16+4c+4) of the 32-channel group.  Each corner
    // then takes two 8-byte loads (still one whole sector per four lanes),
    // and each 16-byte fp32 reduction of a warp instruction lands with those
    // of the team's other lanes in whole 32-byte sectors; with whole slots,
    // every instruction half-fills four sectors and the L2 takes twice the
    // reduction operations.
    constexpr bool SPLIT = std::is_same<ACC, float>::value && EPV == 8;
    const int lane_ch = ln.c * (SPLIT ? 4 : EPV);
    const long long vofs = (long long)b * a.slice + (long long)m * a.D + lane_ch;
    const T* vbase = reinterpret_cast<const T*>(a.value) + vofs;
    ACC* gbase = reinterpret_cast<ACC*>(a.grad_acc) + vofs;
    const int MD = a.M * a.D;
    // TOUCH: the touch classes (FP32 workspace, 16-bit I/O, no merge): a
    // sparse level's rows with one contribution are written directly
    static_assert(!TOUCH || (SPLIT && !FUSED && MERGE == 0), "touch classes: FP32 workspace, unfused, no merge");
    T* tbase = TOUCH ? reinterpret_cast<T*>(a.touch_out) + vofs : nullptr;
    auto load_raw = [&](const T* p) -> typename S_::Raw {
        if constexpr (SPLIT) return split_load_raw(p);
        else return S_::load_raw(p);
    };

    // this lane's channels of g = grad_out[b, q, m, :]
    float g[NV][EPV];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        if (ln.active) {
            const T* go = reinterpret_cast<const T*>(a.grad_out) + (long long)ln.u * a.D + lane_ch + n * kC * EPV;
            S_::unpack(load_raw(go), g[n]);
        } else {
#pragma unroll
            for (int e = 0; e < EPV; ++e) g[n][e] = 0.f;
        }
    }
    // Deterministic accumulator: its reductions are 8-byte integers, one per
    // channel.  For them a lane takes channel kC*e + c of each group (a second
    // copy of g in that order), so the team's four lanes add four adjacent
    // integers, one whole 32-byte sector, per instruction; in slot order each
    // instruction would touch a quarter of four sectors.
    constexpr bool ILV = std::is_same<ACC, long long>::value;
    float gi[ILV ? NV : 1][ILV ? EPV : 1];
    long long* ibase = nullptr;
    if constexpr (ILV) {
        const T* go = reinterpret_cast<const T*>(a.grad_out) + (long long)ln.u * a.D + ln.c;
#pragma unroll
        for (int n = 0; n < NV; ++n)
#pragma unroll
            for (int e = 0; e < EPV; ++e)
                gi[n][e] = ln.active ? Elem<T>::to_f(__ldg(go + n * kC * EPV + kC * e)) : 0.f;
        ibase = reinterpret_cast<long long*>(a.grad_acc) + (long long)b * a.slice + (long long)m * a.D + ln.c;
    }
    T* gl = reinterpret_cast<T*>(a.grad_loc);
    T* ga = reinterpret_cast<T*>(a.grad_attn);
    bool waited = false;
    float dscale = 0.f;  // deterministic accumulator: 2^F, read after the wait
    float smx = 0.f, ssum = 1.f, pdot = 0.f;
    if constexpr (FUSED) softmax_stats<T>(a, sm, staged, ln, smx, ssum);
    float* gbuf = reinterpret_cast<float*>(sm + a.gbuf_off) + ln.team * a.LK;  // fused: <g, sampled> per sample

    for (int r0 = a.s_begin; r0 < a.s_end; r0 += ln.TP) {
        // lane (c, p) owns sample r0 + p*kC + c: a point group's kC samples
        // are consecutive (one level's points when K = kC)
        const int s_own = r0 + ln.p * kC + ln.c;
        const bool live = ln.active && s_own < a.s_end;
        float x = -4.f, y = -4.f, wa = 0.f;
        int l = 0;
        if (live) {
            read_params<T>(a, sm, staged, ln.team, ln.u, s_own, x, y, wa);
            l = (int)fdiv((uint32_t)s_own, a.div_k);
        }
        Level lev = lv[l];
        if (!live) lev.ok = 0;
        if constexpr (FUSED) {
            if (live) {
                fused_location<T>(a, fdiv(ln.u, a.div_m), l, lev, x, y);
                wa = expf(wa - smx) / ssum;
            }
        }
        const SampleSetup me = sample_setup(lev, x, y, MD);
        // touch words of this lane's sample's corner rows, loaded now and
        // read after the gather (sparse levels only; else every corner is
        // reduced into the workspace)
        unsigned tw[4] = {0u, 0u, 0u, 0u};
        bool tsp = false;
        if constexpr (TOUCH) {
            tsp = live && touch_sparse(a, lev);
            if (tsp) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if ((me.mask >> k) & 1u)
                        tw[k] = __ldg(a.touch + (touch_row(a, b, me.pix + (k & 1) + (k >> 1) * lev.W, m) >> 4));
            }
        }

        // gather + reduce: the lane with c == j keeps the totals of sample j
        float ra = 0.f, rx = 0.f, ry = 0.f;
#pragma unroll
        for (int j0 = 0; j0 < kC; j0 += JB) {
            typename S_::Raw raw[JB][4][NV];
            SampleSetup st[JB];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                st[jj] = shfl_setup(me, team_lane(ln, j0 + jj, ln.p));
                const int off[4] = {st[jj].o, st[jj].o + MD, st[jj].o + st[jj].wmd, st[jj].o + st[jj].wmd + MD};
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int n = 0; n < NV; ++n)
                        raw[jj][k][n] = ((st[jj].mask >> k) & 1u) ? load_raw(vbase + off[k] + n * kC * EPV)
                                                                  : S_::zero();
            }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                float d[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float t = 0.f;
#pragma unroll
                    for (int n = 0; n < NV; ++n) {
                        float v[EPV];
                        S_::unpack(raw[jj][k][n], v);
                        t += dot2(g[n], v);
                    }
                    d[k] = t;
                }
                float w[4];
                corner_weights(st[jj].lx, st[jj].ly, w);
                const bool any = st[jj].mask != 0u;
                const float lx = st[jj].lx, ly = st[jj].ly;
                // <g, sampled>, <g, d sampled / d x_im>, <g, d sampled / d y_im>
                float pa = any ? (w[0] * d[0] + w[1] * d[1] + w[2] * d[2] + w[3] * d[3]) : 0.f;
                float px = any ? ((1.f - ly) * (d[1] - d[0]) + ly * (d[3] - d[2])) : 0.f;
                float py = any ? ((1.f - lx) * (d[2] - d[0]) + lx * (d[3] - d[1])) : 0.f;
#pragma unroll
                for (int o = 1; o < kC; o <<= 1) {
                    pa += __shfl_xor_sync(0xffffffffu, pa, o);
                    px += __shfl_xor_sync(0xffffffffu, px, o);
                    py += __shfl_xor_sync(0xffffffffu, py, o);
                }
                if (ln.c == j0 + jj) {
                    ra = pa;
                    rx = px;
                    ry = py;
                }
            }
        }
        if (live) {
            const long long ps = (long long)ln.u * a.LK + s_own;
            if constexpr (FUSED) {
                // d loc / d offset = (1/W, 1/H): the level size cancels
                gl[2 * ps] = Elem<T>::from_f(wa * rx);
                gl[2 * ps + 1] = Elem<T>::from_f(wa * ry);
                gbuf[s_own] = ra;
                pdot += wa * ra;
                if (a.rbuf_off >= 0) {  // grad_loc, summed into grad_reference_points below
                    float* rb = reinterpret_cast<float*>(sm + a.rbuf_off) + ((long long)ln.team * a.LK + s_own) * 2;
                    rb[0] = wa * rx * lev.fW;
                    rb[1] = wa * ry * lev.fH;
                }
            } else {
                ga[ps] = Elem<T>::from_f(ra);
                gl[2 * ps] = Elem<T>::from_f(wa * lev.fW * rx);
                gl[2 * ps + 1] = Elem<T>::from_f(wa * lev.fH * ry);
            }
        }

        if constexpr (MERGE >= 0) {
            // Corner merge (MERGE).  Samples of the point group that add some of
            // the same rows merge first: each shared row is added once, by the
            // last sample holding it, with the sum of their coefficients
            // A * w_k, and the others skip that corner.  A corner merges only
            // when it is inside the level for both samples, so equal offsets mean
            // the same row.  Whole cells: samples with the same cell offset and
            // level width (an equivalence, so every holder is found).  Every
            // shared corner: also cells that touch, by edge or corner, on a level
            // at least three pixels wide.  Two cells sharing a corner row are
            // within one pixel of each other, and for W >= 3 the nine such offsets
            // are distinct, so every pair holding a row is found (a missed pair
            // could lose a coefficient: an intermediate sample would absorb it and
            // then skip the row for a later holder that did not).
            // The reductions bound this kernel when samples cluster.  Measured on
            // GB300, encoder backward: native 346 -> 281 us with whole cells
            // (17% fewer reductions; 306 us with every corner, whose extra
            // instructions cost more than its extra 12%); fp32 workspace
            // 601 -> 454 us with every corner (479 with whole cells).  With
            // uniformly spread samples (decoder) nothing merges and the code
            // costs ~2 us, so it is compiled only into the merging kernels.
            float mc[4];
            unsigned smask = me.mask;
            {
                float w0[4];
                corner_weights(me.lx, me.ly, w0);
                float oc[4];
    #pragma unroll
                for (int k = 0; k < 4; ++k) mc[k] = oc[k] = wa * w0[k];
    #pragma unroll
                for (int jj = 0; jj < kC; ++jj) {
                    if constexpr (MERGE == 0) break;
                    const int src = team_lane(ln, jj, ln.p);
                    const int o2 = __shfl_sync(0xffffffffu, me.o, src);
                    const int w2 = __shfl_sync(0xffffffffu, me.wmd, src);
                    const unsigned m2 = __shfl_sync(0xffffffffu, me.mask, src);
                    float c2[4];
    #pragma unroll
                    for (int k = 0; k < 4; ++k) c2[k] = __shfl_sync(0xffffffffu, oc[k], src);
                    if (jj == ln.c || w2 != me.wmd) continue;
                    const bool earlier = jj < ln.c;
                    // my corner k is the other sample's corner k2
                    auto share = [&](int k, int k2) {
                        if (((me.mask >> k) & 1u) && ((m2 >> k2) & 1u)) {
                            if (earlier) mc[k] += c2[k2];
                            else smask &= ~(1u << k);
                        }
                    };
                    const int dd = o2 - me.o;  // the other cell relative to mine
                    if constexpr (MERGE == kMergeCells) {
                        if (dd == 0) {
                            share(0, 0); share(1, 1); share(2, 2); share(3, 3);
                        }
                    } else {
                        if (me.wmd < 3 * MD) continue;
                        if (dd == 0) {
                            share(0, 0); share(1, 1); share(2, 2); share(3, 3);
                        } else if (dd == MD) {                  // one pixel right
                            share(1, 0); share(3, 2);
                        } else if (dd == -MD) {                 // one pixel left
                            share(0, 1); share(2, 3);
                        } else if (dd == me.wmd) {              // one row down
                            share(2, 0); share(3, 1);
                        } else if (dd == -me.wmd) {             // one row up
                            share(0, 2); share(1, 3);
                        } else if (dd == me.wmd + MD) {         // down-right
                            share(3, 0);
                        } else if (dd == me.wmd - MD) {         // down-left
                            share(2, 1);
                        } else if (dd == MD - me.wmd) {         // up-right
                            share(1, 2);
                        } else if (dd == -MD - me.wmd) {        // up-left
                            share(0, 3);
                        }
                    }
                }
            }

            // the sample's corner classes, 2 bits each (2 = reduce into the workspace)
            unsigned tcls = 0xAAu;
            if constexpr (TOUCH) {
                if (tsp) {
                    tcls = 0u;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        unsigned c = 2u;
                        if ((me.mask >> k) & 1u) {
                            c = touch_bits(tw[k], touch_row(a, b, me.pix + (k & 1) + (k >> 1) * lev.W, m));
                            if (c == 0u) {   // the count pass missed it: never expected
                                atomicOr(a.err, kErrTouch);
                                c = 2u;
                            }
                        }
                        tcls |= c << (2 * k);
                    }
                }
            }

            // scatter: A * w_corner * g into the inside corners
            if (!waited) {
                asm volatile("griddepcontrol.wait;" ::: "memory");
                waited = true;
                if constexpr (std::is_same<ACC, long long>::value) dscale = det_scale(a.det, (long long)a.Q * a.LK);
            }
    #pragma unroll
            for (int j = 0; j < kC; ++j) {
                const int src = team_lane(ln, j, ln.p);
                const int so = __shfl_sync(0xffffffffu, me.o, src);
                const int swmd = __shfl_sync(0xffffffffu, me.wmd, src);
                const unsigned smk = __shfl_sync(0xffffffffu, smask, src);
                const unsigned scls = TOUCH ? __shfl_sync(0xffffffffu, tcls, src) : 0xAAu;
                float cj[4];
    #pragma unroll
                for (int k = 0; k < 4; ++k) cj[k] = __shfl_sync(0xffffffffu, mc[k], src);
                const int off[4] = {so, so + MD, so + swmd, so + swmd + MD};
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (!((smk >> k) & 1u)) continue;
                    const float2 cf = make_float2(cj[k], cj[k]);
    #pragma unroll
                    for (int n = 0; n < NV; ++n) {
                        if constexpr (ILV) {
                            // each contribution times 2^F (exact), rounded once to an integer
                            long long* q = ibase + off[k] + n * kC * EPV;
    #pragma unroll
                            for (int e = 0; e < EPV; ++e) red_s64(q + kC * e, __float2ll_rn(cf.x * gi[n][e] * dscale));
                        } else {
                            float t[EPV];
    #pragma unroll
                            for (int e = 0; e < EPV; e += 2) {
                                const float2 r = __fmul2_rn(cf, make_float2(g[n][e], g[n][e + 1]));
                                t[e] = r.x;
                                t[e + 1] = r.y;
                            }
                            if constexpr (SPLIT) {
                                if (TOUCH && ((scls >> (2 * k)) & 3u) == 1u) {
                                    // the row's one contribution, rounded once
                                    T* q = tbase + off[k] + n * kC * EPV;
                                    store4<T>(q, t[0], t[1], t[2], t[3]);
                                    store4<T>(q + 16, t[4], t[5], t[6], t[7]);
                                } else {
                                    float* q = gbase + off[k] + n * kC * EPV;
                                    red_v4_f32(q, t[0], t[1], t[2], t[3]);
                                    red_v4_f32(q + 16, t[4], t[5], t[6], t[7]);
                                }
                            } else {
                                Scatter<ACC, EPV>::add(gbase + off[k] + n * kC * EPV, t);
                            }
                        }
                    }
                }
            }
        }
    }
    if constexpr (FUSED) {
        // softmax backward: grad_logit_s = A_s * (<g, sampled_s> - sum_j A_j <g, sampled_j>)
        for (int o = 1; o < ln.TP; o <<= 1) pdot += __shfl_xor_sync(0xffffffffu, pdot, o);
        __syncwarp();
        for (int r0 = 0; r0 < a.LK; r0 += ln.TP) {
            const int s_own = r0 + ln.p * kC + ln.c;
            if (ln.active && s_own < a.LK) {
                const float A = expf(read_weight<T>(a, sm, staged, ln.team, ln.u, s_own) - smx) / ssum;
                ga[(long long)ln.u * a.LK + s_own] = Elem<T>::from_f(A * (gbuf[s_own] - pdot));
            }
        }
        // grad_reference_points[b, q, l] = sum over (m, k) of grad_loc, when
        // the block holds whole queries (units per block a multiple of M):
        // one thread per output, a fixed summation order
        if (a.rbuf_off >= 0) {
            __syncthreads();
            const float* rb = reinterpret_cast<const float*>(sm + a.rbuf_off);
            const int nq = min(a.tpb, a.n_units - (int)ln.u0) / a.M;
            for (int t = threadIdx.x; t < nq * a.L * 2; t += blockDim.x) {
                const int c = t & 1, l = (t >> 1) % a.L, ql = (t >> 1) / a.L;
                float acc = 0.f;
                for (int m = 0; m < a.M; ++m) {
                    const float* r = rb + ((ql * a.M + m) * a.LK + l * a.K) * 2 + c;
                    for (int k = 0; k < a.K; ++k) acc += r[2 * k];
                }
                const long long bq = (long long)(ln.u0 / (uint32_t)a.M) + ql;
                reinterpret_cast<T*>(a.gref)[(bq * a.L + l) * 2 + c] = Elem<T>::from_f(acc);
            }
        }
    }
}

template <typename T, typename ACC, int NV, bool FUSED, int MERGE, bool TOUCH = false>
__global__ void __launch_bounds__(kBlockThreads) msda_bwd4_kernel(const KernelArgs a) {
    bwd4_body<T, ACC, NV, FUSED, MERGE, TOUCH>(a);
}

// The merging backward for one slot per lane, held to four resident blocks
// per SM (64 registers): merging every corner would take it to 76 registers
// and three blocks, and on GB300 the native encoder backward then keeps none
// of the merge gains (344 us at three blocks, 306 us at four).
template <typename T, typename ACC, bool FUSED, int MERGE>
__global__ void __launch_bounds__(kBlockThreads, 4) msda_bwd4_merge1_kernel(const KernelArgs a) {
    bwd4_body<T, ACC, 1, FUSED, MERGE, false>(a);
}

// ---------------------------------------------------------------------------
// Backward into the FP32 workspace for 16-bit I/O, eight channel lanes a unit
// (one pass per level, no corner merge).  Lane c owns channels [4c, 4c + 4)
// of each 32-channel group: its corner loads are 8 bytes and its reductions
// 16 bytes of fp32, so the eight lanes of a team read a corner row's 64 bytes
// with one request and add its 128 bytes of sums with one, where the four
// lanes of msda_bwd4_kernel take two of each (split slots).  The passes of
// dense levels, whose corner rows mostly hit in the L2, are bound by the
// L1's requests to the L2.  Setup, gather, touch classes and scatter as in
// bwd4_body: lane c sets up sample r0 + c of the round, the team reads it
// with warp shuffles.

// four 16-bit channels (8 bytes) -> fp32
__device__ __forceinline__ void unpack8(const uint2& w, float (&f)[4], const __nv_bfloat16*) {
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
}
__device__ __forceinline__ void unpack8(const uint2& w, float (&f)[4], const __half*) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
}

constexpr int kC8 = 8;

template <typename T, int NV, bool TOUCH>
__global__ void __launch_bounds__(kBlockThreads) msda_bwd8_kernel(const KernelArgs a) {
    static_assert(sizeof(T) == 2, "16-bit I/O into the fp32 workspace");
    constexpr int JB = 2;   // samples whose corners are loaded together (stress backward 4.12 ms; 4 or 1: 4.26)
    const T* tag = nullptr;
    __shared__ Level lv[MSDA_MAX_LEVELS];
    if (threadIdx.x < a.L) {
        lv[threadIdx.x] = level_of(a, threadIdx.x);
        if (!lv[threadIdx.x].ok) atomicOr(a.err, kErrBadLevel);
    }
    __syncthreads();
    // launched as a programmatic dependent of the workspace's clearing: wait
    // for it before anything (returns at once otherwise)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int team = threadIdx.x / kC8, c = threadIdx.x % kC8;
    const int lane0 = (threadIdx.x & 31) & ~(kC8 - 1);
    const uint32_t u = blockIdx.x * (uint32_t)(kBlockThreads / kC8) + (uint32_t)team;
    const bool active = u < (uint32_t)a.n_units;
    const uint32_t b = active ? fdiv(u, a.div_qm) : 0u;
    const uint32_t m = active ? u - fdiv(u, a.div_m) * (uint32_t)a.M : 0u;
    const int MD = a.M * a.D;
    const long long vofs = (long long)b * a.slice + (long long)m * a.D + 4 * c;
    const T* vbase = reinterpret_cast<const T*>(a.value) + vofs;
    float* gbase = reinterpret_cast<float*>(a.grad_acc) + vofs;
    T* tbase = TOUCH ? reinterpret_cast<T*>(a.touch_out) + vofs : nullptr;
    float g[NV][4];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
        if (active) {
            const T* go = reinterpret_cast<const T*>(a.grad_out) + (long long)u * a.D + 32 * n + 4 * c;
            unpack8(__ldg(reinterpret_cast<const uint2*>(go)), g[n], tag);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) g[n][e] = 0.f;
        }
    }
    T* gl = reinterpret_cast<T*>(a.grad_loc);
    T* ga = reinterpret_cast<T*>(a.grad_attn);

    for (int r0 = a.s_begin; r0 < a.s_end; r0 += kC8) {
        const int nj = min(kC8, a.s_end - r0);   // samples of this round (the same for the whole warp)
        const int s_own = r0 + c;
        const bool live = active && c < nj;
        float x = -4.f, y = -4.f, wa = 0.f;
        int l = 0;
        if (live) {
            const long long ps = (long long)u * a.LK + s_own;
            const T* pl = reinterpret_cast<const T*>(a.loc) + 2 * ps;
            x = ldg_f(pl);
            y = ldg_f(pl + 1);
            wa = ldg_f(reinterpret_cast<const T*>(a.attn) + ps);
            l = (int)fdiv((uint32_t)s_own, a.div_k);
        }
        Level lev = lv[l];
        if (!live) lev.ok = 0;
        const SampleSetup me = sample_setup(lev, x, y, MD);
        unsigned tw[4] = {0u, 0u, 0u, 0u};
        bool tsp = false;
        if constexpr (TOUCH) {
            tsp = live && touch_sparse(a, lev);
            if (tsp) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if ((me.mask >> k) & 1u)
                        tw[k] = __ldg(a.touch + (touch_row(a, b, me.pix + (k & 1) + (k >> 1) * lev.W, m) >> 4));
            }
        }

        // gather + reduce over the team: lane j keeps the totals of sample j
        float ra = 0.f, rx = 0.f, ry = 0.f;
        for (int j0 = 0; j0 < nj; j0 += JB) {
            uint2 raw[JB][4][NV];
            SampleSetup st[JB];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                st[jj] = shfl_setup(me, lane0 + min(j0 + jj, kC8 - 1));
                if (j0 + jj >= nj) st[jj].mask = 0u;
                const int off[4] = {st[jj].o, st[jj].o + MD, st[jj].o + st[jj].wmd, st[jj].o + st[jj].wmd + MD};
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int n = 0; n < NV; ++n)
                        raw[jj][k][n] = ((st[jj].mask >> k) & 1u)
                                            ? __ldg(reinterpret_cast<const uint2*>(vbase + off[k] + 32 * n))
                                            : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                float d[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float t = 0.f;
#pragma unroll
                    for (int n = 0; n < NV; ++n) {
                        float v[4];
                        unpack8(raw[jj][k][n], v, tag);
                        t = __fmaf_rn(g[n][0], v[0], t);
                        t = __fmaf_rn(g[n][1], v[1], t);
                        t = __fmaf_rn(g[n][2], v[2], t);
                        t = __fmaf_rn(g[n][3], v[3], t);
                    }
                    d[k] = t;
                }
                float w[4];
                corner_weights(st[jj].lx, st[jj].ly, w);
                const bool any = st[jj].mask != 0u;
                const float lx = st[jj].lx, ly = st[jj].ly;
                float pa = any ? (w[0] * d[0] + w[1] * d[1] + w[2] * d[2] + w[3] * d[3]) : 0.f;
                float px = any ? ((1.f - ly) * (d[1] - d[0]) + ly * (d[3] - d[2])) : 0.f;
                float py = any ? ((1.f - lx) * (d[2] - d[0]) + lx * (d[3] - d[1])) : 0.f;
#pragma unroll
                for (int o = 1; o < kC8; o <<= 1) {
                    pa += __shfl_xor_sync(0xffffffffu, pa, o);
                    px += __shfl_xor_sync(0xffffffffu, px, o);
                    py += __shfl_xor_sync(0xffffffffu, py, o);
                }
                if (c == j0 + jj) {
                    ra = pa;
                    rx = px;
                    ry = py;
                }
            }
        }
        if (live) {
            const long long ps = (long long)u * a.LK + s_own;
            ga[ps] = Elem<T>::from_f(ra);
            gl[2 * ps] = Elem<T>::from_f(wa * lev.fW * rx);
            gl[2 * ps + 1] = Elem<T>::from_f(wa * lev.fH * ry);
        }

        // the sample's corner classes, 2 bits each (2 = reduce into the workspace)
        unsigned tcls = 0xAAu;
        if constexpr (TOUCH) {
            if (tsp) {
                tcls = 0u;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    unsigned cl = 2u;
                    if ((me.mask >> k) & 1u) {
                        cl = touch_bits(tw[k], touch_row(a, b, me.pix + (k & 1) + (k >> 1) * lev.W, m));
                        if (cl == 0u) {   // the count pass missed it: never expected
                            atomicOr(a.err, kErrTouch);
                            cl = 2u;
                        }
                    }
                    tcls |= cl << (2 * k);
                }
            }
        }
        float w0[4];
        corner_weights(me.lx, me.ly, w0);
        float mc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mc[k] = wa * w0[k];

        // scatter: A * w_corner * g into the inside corners
        for (int j = 0; j < nj; ++j) {
            const int src = lane0 + j;
            const int so = __shfl_sync(0xffffffffu, me.o, src);
            const int swmd = __shfl_sync(0xffffffffu, me.wmd, src);
            const unsigned smk = __shfl_sync(0xffffffffu, me.mask, src);
            const unsigned scls = TOUCH ? __shfl_sync(0xffffffffu, tcls, src) : 0xAAu;
            float cj[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) cj[k] = __shfl_sync(0xffffffffu, mc[k], src);
            const int off[4] = {so, so + MD, so + swmd, so + swmd + MD};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (!((smk >> k) & 1u)) continue;
                const float2 cf = make_float2(cj[k], cj[k]);
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    const float2 t0 = __fmul2_rn(cf, make_float2(g[n][0], g[n][1]));
                    const float2 t1 = __fmul2_rn(cf, make_float2(g[n][2], g[n][3]));
                    if (TOUCH && ((scls >> (2 * k)) & 3u) == 1u)
                        store4<T>(tbase + off[k] + 32 * n, t0.x, t0.y, t1.x, t1.y);   // the row's one contribution
                    else
                        red_v4_f32(gbase + off[k] + 32 * n, t0.x, t0.y, t1.x, t1.y);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Forward with TMA gathers (rows of whole 16-byte vectors, L*K in {4, 8, 16,
// 32}, B*S*M < 2^31).  `value` is seen as a 2-D tensor of B*S*M rows of D
// channels; one cp.async.bulk.tensor ... tile::gather4 brings the four
// corner rows of a sample into shared memory, so a warp keeps 32 samples
// (32 x 4 rows) in flight without holding registers or L1 miss slots for
// them.  Each warp takes 32 / (L*K) units: lane t sets up sample t, writes
// its four coefficients (A * w_corner, 0 outside) to shared memory and
// issues the gather; a corner outside the level gets row -1, which the
// copy fills with zeros.  The copies complete on the warp's mbarrier, waited
// with a bounded number of polls; then the same lanes, as C = 4 channel
// lanes x P = L*K/4 point lanes per unit, accumulate from shared memory.

constexpr int kTmaWarps = 4;

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int col, int r0, int r1, int r2,
                                            int r3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(map), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}

// The same with an L2 eviction priority (a createpolicy cache policy).
__device__ __forceinline__ void tma_gather4_hint(uint32_t dst, const CUtensorMap* map, int col, int r0, int r1,
                                                 int r2, int r3, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(map), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar), "l"(policy)
        : "memory");
}

// bytes of dynamic shared memory of msda_fwd_tma_kernel<T, NV>
template <typename T, int NV>
constexpr int fwd_tma_smem() {
    return kTmaWarps * (32 * 4 * kC * NV * 16 + 32 * 16) + 128;
}

template <typename T, int NV>
__global__ void __launch_bounds__(kTmaWarps * 32) msda_fwd_tma_kernel(const KernelArgs a,
                                                                      const __grid_constant__ CUtensorMap tmap) {
    constexpr int EPV = 16 / sizeof(T);
    constexpr int ROWB = kC * NV * 16;  // bytes of one D-row
    constexpr int SAMPLEB = 4 * ROWB;   // four corner rows
    constexpr int STAGEB = 32 * SAMPLEB;
    using S_ = Slot<T, EPV>;
    __shared__ Level lv[MSDA_MAX_LEVELS];
    __shared__ __align__(8) uint64_t wbar[kTmaWarps];
    extern __shared__ unsigned char sm_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(sm_raw) + 127) & ~(uintptr_t)127);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < a.L) {
        const int l = threadIdx.x;
        const long long H = a.shapes[2 * l], W = a.shapes[2 * l + 1], st = a.starts[l];
        const bool ok = H >= 1 && W >= 1 && H <= kMaxSide && W <= kMaxSide && st >= 0 && st <= a.S &&
                        H * W <= a.S - st;
        const long long MD = (long long)a.M * a.D;
        Level v;
        v.start_md = ok ? st * MD : 0;
        v.w_md = ok ? W * MD : 0;
        v.fH = ok ? (float)H : 0.f;
        v.fW = ok ? (float)W : 0.f;
        v.ok = ok;
        v.W = ok ? (int)W : 0;
        v.start = ok ? st : 0;
        lv[l] = v;
        if (!ok) atomicOr(a.err, kErrBadLevel);
    }
    const uint32_t bar = smem_u32(&wbar[warp]);
    if (lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int lgLK = a.lp + 2;  // L*K = 4P lanes per unit
    const int LK = 1 << lgLK;
    const int G = 32 >> lgLK;   // units per warp
    const uint32_t n_groups = ((uint32_t)a.n_units + G - 1) / G;
    const uint32_t grp = blockIdx.x * (uint32_t)kTmaWarps + warp;
    if (grp >= n_groups) return;  // the whole warp leaves together

    unsigned char* stage = sm + warp * STAGEB;
    float4* coef = reinterpret_cast<float4*>(sm + kTmaWarps * STAGEB) + warp * 32;

    // ---- setup: lane = (unit ul, sample s)
    const int ul = lane >> lgLK;
    const int s = lane & (LK - 1);
    const uint32_t u = grp * G + ul;
    const bool live = u < (uint32_t)a.n_units;
    const uint32_t b = live ? fdiv(u, a.div_qm) : 0u;
    const uint32_t m = live ? u - fdiv(u, a.div_m) * (uint32_t)a.M : 0u;
    float x = -4.f, y = -4.f, w = 0.f;
    int l = 0;
    if (live) {
        const long long ps = (long long)u * LK + s;
        const T* pl = reinterpret_cast<const T*>(a.loc) + 2 * ps;
        x = ldg_f(pl);
        y = ldg_f(pl + 1);
        w = ldg_f(reinterpret_cast<const T*>(a.attn) + ps);
        l = (int)fdiv((uint32_t)s, a.div_k);
    }
    Level lev = lv[l];
    if (!live) lev.ok = 0;
    const float xi = __fmaf_rn(x, lev.fW, -0.5f);
    const float yi = __fmaf_rn(y, lev.fH, -0.5f);
    const float x0f = floorf(xi), y0f = floorf(yi);
    const bool vx0 = lev.ok && x0f >= 0.f && x0f < lev.fW;
    const bool vx1 = lev.ok && x0f >= -1.f && x0f < lev.fW - 1.f;
    const bool vy0 = y0f >= 0.f && y0f < lev.fH;
    const bool vy1 = y0f >= -1.f && y0f < lev.fH - 1.f;
    const int x0 = (vx0 || vx1) ? (int)x0f : 0;
    const int y0 = (vy0 || vy1) ? (int)y0f : 0;
    // row of corner (y0, x0) in the [B*S*M, D] view: (b*S + pixel)*M + m
    const int row0 = (int)(((long long)b * a.S + lev.start + (long long)y0 * lev.W + x0) * a.M + m);
    const int wm = lev.W * a.M;
    const bool ok[4] = {vy0 && vx0, vy0 && vx1, vy1 && vx0, vy1 && vx1};
    float wk[4];
    corner_weights(xi - x0f, yi - y0f, wk);
    coef[lane] = make_float4(ok[0] ? w * wk[0] : 0.f, ok[1] ? w * wk[1] : 0.f, ok[2] ? w * wk[2] : 0.f,
                             ok[3] ? w * wk[3] : 0.f);
    const unsigned issuing = __ballot_sync(0xffffffffu, live);
    if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)(__popc(issuing) * SAMPLEB))
                     : "memory");
    __syncwarp();
    // L2 priority by the size of the sample's level (its rows in one image):
    // the rows of a level over twice the L2 are read about once each and evict
    // first.  Measured on GB300 (stress forward): 0.843 -> 0.825 ms; evict-first
    // from half the L2 on (levels 0 and 1) 0.859 ms, from an eighth 1.07 ms;
    // evict-last for the levels of at most a quarter of the L2 gave nothing
    // (0.839 ms), at a fraction of 0.25 0.872 ms, and with both priorities 1.10 ms.
    const long long lvb = (long long)lev.fH * lev.W * a.M * a.D * (long long)sizeof(T);
    const bool evict_first = a.l2_bytes > 0 && lvb >= 2 * a.l2_bytes;
    if (live) {
        const int r0 = ok[0] ? row0 : -1, r1 = ok[1] ? row0 + a.M : -1;
        const int r2 = ok[2] ? row0 + wm : -1, r3 = ok[3] ? row0 + wm + a.M : -1;
        if (!evict_first) {
            tma_gather4(smem_u32(stage + lane * SAMPLEB), &tmap, 0, r0, r1, r2, r3, bar);
        } else {
            uint64_t pol;
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
            tma_gather4_hint(smem_u32(stage + lane * SAMPLEB), &tmap, 0, r0, r1, r2, r3, bar, pol);
        }
    }

    uint32_t done = 0;
    for (int it = 0; it < (1 << 22) && !done; ++it) done = mbar_try_wait(bar, 0);
    if (!__all_sync(0xffffffffu, done)) {
        if (lane == 0) atomicOr(a.err, kErrBulkTimeout);
        for (int it = 0; it < (1 << 22) && !done; ++it) done = mbar_try_wait(bar, 0);
        return;
    }

    // ---- accumulate: lane = (unit ul, channel lane c, point lane p)
    const int c = s & (kC - 1), p = s >> 2, P = LK >> 2;
    float acc[NV][EPV];
#pragma unroll
    for (int n = 0; n < NV; ++n)
#pragma unroll
        for (int e = 0; e < EPV; ++e) acc[n][e] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int slot = (ul << lgLK) + p + i * P;
        const float4 cf4 = coef[slot];
        const float cf[4] = {cf4.x, cf4.y, cf4.z, cf4.w};
        const unsigned char* base = stage + slot * SAMPLEB + c * 16;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int n = 0; n < NV; ++n) {
                const uint4 raw = *reinterpret_cast<const uint4*>(base + k * ROWB + n * kC * 16);
                float v[EPV];
                S_::unpack(raw, v);
                axpy2(acc[n], cf[k], v);
            }
    }
    for (int o = kC; o < LK; o <<= 1) {
#pragma unroll
        for (int n = 0; n < NV; ++n)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[n][e] += __shfl_xor_sync(0xffffffffu, acc[n][e], o);
    }
    if (live && p == 0) {
        T* o = reinterpret_cast<T*>(a.out) + (long long)u * a.D + c * EPV;
#pragma unroll
        for (int n = 0; n < NV; ++n) S_::store(o + n * kC * EPV, acc[n]);
    }
}

// ---------------------------------------------------------------------------
// Point-parallel forward (ablation only, selected with MSDA_TUNE=pointparallel):
// the decomposition the course calls the obvious port (ch. 4, "The design
// question"): one thread per sampling point (b, q, m, l, k) reads its four
// corners channel by channel on its own and keeps a D-float partial sum; the
// L*K threads of a unit then combine their partials through shared memory.
// Threads of a warp read unrelated rows, so each scalar load uses a few
// bytes of its sector.  Kept to compare occupancy and bandwidth with the
// team decomposition above; D = 32, L*K dividing 256.

constexpr int kPpD = 32;

template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_fwd_pointparallel_kernel(const KernelArgs a) {
    __shared__ Level lv[MSDA_MAX_LEVELS];
    __shared__ float part[kBlockThreads][kPpD + 1];
    if (threadIdx.x < a.L) {
        const int l = threadIdx.x;
        const long long H = a.shapes[2 * l], W = a.shapes[2 * l + 1], st = a.starts[l];
        const bool ok = H >= 1 && W >= 1 && H <= kMaxSide && W <= kMaxSide && st >= 0 && st <= a.S &&
                        H * W <= a.S - st;
        const long long MD = (long long)a.M * a.D;
        Level v;
        v.start_md = ok ? st * MD : 0;
        v.w_md = ok ? W * MD : 0;
        v.fH = ok ? (float)H : 0.f;
        v.fW = ok ? (float)W : 0.f;
        v.ok = ok;
        v.W = ok ? (int)W : 0;
        v.start = ok ? st : 0;
        lv[l] = v;
        if (!ok) atomicOr(a.err, kErrBadLevel);
    }
    __syncthreads();
    const int LK = a.LK;
    const int upb = kBlockThreads / LK;  // units per block
    const int t = threadIdx.x;
    const uint32_t u = blockIdx.x * (uint32_t)upb + t / LK;
    const int s = t % LK;
    const bool live = t < upb * LK && u < (uint32_t)a.n_units;
    float acc[kPpD];
#pragma unroll
    for (int d = 0; d < kPpD; ++d) acc[d] = 0.f;
    if (live) {
        const uint32_t b = fdiv(u, a.div_qm);
        const uint32_t m = u - fdiv(u, a.div_m) * (uint32_t)a.M;
        const T* vbase = reinterpret_cast<const T*>(a.value) + (long long)b * a.slice + (long long)m * a.D;
        const long long ps = (long long)u * LK + s;
        const float x = ldg_f(reinterpret_cast<const T*>(a.loc) + 2 * ps);
        const float y = ldg_f(reinterpret_cast<const T*>(a.loc) + 2 * ps + 1);
        const float w = ldg_f(reinterpret_cast<const T*>(a.attn) + ps);
        const Level lev = lv[fdiv((uint32_t)s, a.div_k)];
        Corners<int> cr;
        bilinear_setup<int>(lev, x, y, a.M * a.D, cr);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (!cr.ok[k]) continue;
            const float c = w * cr.w[k];
#pragma unroll
            for (int d = 0; d < kPpD; ++d) acc[d] = fmaf(c, ldg_f(vbase + cr.off[k] + d), acc[d]);
        }
    }
#pragma unroll
    for (int d = 0; d < kPpD; ++d) part[t][d] = acc[d];
    __syncthreads();
    // combine: thread t sums channel t % 32 of unit t / 32 over its L*K partials
    for (int i = t; i < upb * kPpD; i += kBlockThreads) {
        const int ul = i / kPpD, d = i % kPpD;
        const uint32_t uu = blockIdx.x * (uint32_t)upb + ul;
        if (uu >= (uint32_t)a.n_units) continue;
        float sum = 0.f;
        for (int j = 0; j < LK; ++j) sum += part[ul * LK + j][d];
        reinterpret_cast<T*>(a.out)[(long long)uu * a.D + d] = Elem<T>::from_f(sum);
    }
}

// ---------------------------------------------------------------------------
// fused operator: gradient of the reference points, d loc / d ref = 1:
// grad_ref[bq, l, c] = sum over (m, k) of grad_loc = grad_offsets * (W_l | H_l)

template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_fused_ref_grad_kernel(const T* goff, T* gref,
                                                                            const int64_t* shapes, long long BQ,
                                                                            int M, int L, int K) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BQ * L * 2) return;
    const int c = (int)(i & 1);
    const int l = (int)((i >> 1) % L);
    const long long bq = (i >> 1) / L;
    const long long side = shapes[2 * l + (c == 0 ? 1 : 0)];   // W for x, H for y
    const float scale = (side >= 1 && side <= kMaxSide) ? (float)side : 0.f;
    float acc = 0.f;
    for (int m = 0; m < M; ++m) {
        const T* p = goff + ((((bq * M + m) * L + l) * (long long)K) * 2) + c;
        for (int k = 0; k < K; ++k) acc += Elem<T>::to_f(p[2 * k]) * scale;
    }
    gref[i] = Elem<T>::from_f(acc);
}

// ---------------------------------------------------------------------------
// deterministic accumulator: maxima and conversion

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// max |g| and max |A| into the header (order-free: atomicMax on the bits of
// non-negative floats; NaN compares false and is skipped).  max |A| starts at
// ma0: 1 for softmax-normalised weights, which then need no scan (na = 0).
template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_det_max_kernel(const T* g, long long ng, const T* attn,
                                                                     long long na, float ma0, DetHeader* h) {
    // the backward (a programmatic dependent) may start its gather phase now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float red[2][kBlockThreads / 32];
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nth = (long long)gridDim.x * blockDim.x;
    float mg = 0.f, ma = ma0;
    for (long long i = tid; i < ng; i += nth) mg = fmaxf(mg, fabsf(Elem<T>::to_f(g[i])));
    for (long long i = tid; i < na; i += nth) ma = fmaxf(ma, fabsf(Elem<T>::to_f(attn[i])));
    mg = warp_max(mg);
    ma = warp_max(ma);
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = mg;
        red[1][threadIdx.x >> 5] = ma;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        mg = threadIdx.x < kBlockThreads / 32 ? red[0][threadIdx.x] : 0.f;
        ma = threadIdx.x < kBlockThreads / 32 ? red[1][threadIdx.x] : 0.f;
        mg = warp_max(mg);
        ma = warp_max(ma);
        if (threadIdx.x == 0) {
            atomicMax(&h->max_g_bits, __float_as_uint(mg));
            atomicMax(&h->max_attn_bits, __float_as_uint(ma));
        }
    }
}

// grad_value[i] = dtype(sum[i] * 2^-F (+ grad_value[i] when accumulating)),
// the integer converted to double and scaled exactly, then one rounding.
template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_det_convert_kernel(const long long* ws, T* gv, long long n,
                                                                         const DetHeader* h, long long qlk,
                                                                         int accumulate) {
    const double inv = 1.0 / (double)det_scale(h, qlk);
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nth = (long long)gridDim.x * blockDim.x;
    for (long long i = tid; i < n; i += nth) {
        double v = __ll2double_rn(ws[i]) * inv;
        if (accumulate) v += (double)Elem<T>::to_f(gv[i]);
        if constexpr (sizeof(T) == 4) gv[i] = __double2float_rn(v);
        else if constexpr (std::is_same<T, __half>::value) gv[i] = __double2half(v);
        else gv[i] = __double2bfloat16(v);
    }
}

// ---------------------------------------------------------------------------
// zero / convert helpers of the backward

// grad_value[i] = round(ws[i]) for i < n (8 elements per step when aligned).
// rezero: write zeros back over every 32-byte piece of ws found non-zero, so
// a workspace that held zeros before the backward holds zeros again (the
// pieces no sample touched are left alone, unwritten).
template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_convert_kernel(float* ws, T* gv, long long n, int vec,
                                                                     int rezero) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nth = (long long)gridDim.x * blockDim.x;
    long long done = 0;
    if (vec) {
        const long long n8 = n / 8;
        for (long long i = tid; i < n8; i += nth) round8<T>(ws, gv, i, rezero);
        done = n8 * 8;
    }
    for (long long i = done + tid; i < n; i += nth) {
        const float v = ws[i];
        gv[i] = Elem<T>::from_f(v);
        if (rezero && __float_as_uint(v)) ws[i] = 0.f;
    }
}

// The rounding pass for the rows the backward passes did not round
// themselves: in every batch image, the rows from the first row of the levels
// >= a.conv_lo (row 0 when a.conv_lo < 0) up to the first row of the levels
// >= a.conv_hi, which no pass of those levels adds to (16-byte aligned
// workspace and grad_value; rows of 32*NV channels, the specialised plans).  A warp takes 32 consecutive rows (pixel,
// head) of one image; lane L works out the class of row base + L once (touch
// classes: 0 untouched, 1 written by its pass, 2 in the workspace), then the
// warp rounds the rows four at a time, eight lanes a row and 16 bytes of fp32
// a lane (each 32-channel group of a row is one 128-byte line), reading a
// row's class from its lane with a shuffle.  Loads of four rows are issued
// before their stores; the rows read are re-zeroed without looking (with
// MSDA_BWD_WORKSPACE_ZEROED).  Measured on GB300 (stress rounding, 8.6 GB of
// workspace): 1.36 ms, against 1.41 ms for one thread per group of eight
// elements (two groups in flight, eight blocks an SM; four groups 1.53 ms,
// eight 1.92 ms; with a test of the values before re-zeroing 1.49 ms).  Held
// to six blocks an SM (one 16-byte slot a lane: wider rows would spill), with
// the classes worked out an iteration ahead: 1.32 ms alone, and the stress
// backward with the rounding beside the coarse passes 4.23 -> 4.13 ms.
template <typename T, int NV>
__global__ void __launch_bounds__(kBlockThreads, NV == 1 ? 6 : 1) msda_round_rows_kernel(const KernelArgs a) {
    static_assert(sizeof(T) == 2, "16-bit grad_value");
    const T* tag = nullptr;
    __shared__ long long lo_hi[2];
    __shared__ TouchRanges tr;
    if (threadIdx.x == 0) {
        lo_hi[0] = a.conv_lo < 0 ? 0 : first_row_from(a, a.conv_lo) * a.M;
        lo_hi[1] = first_row_from(a, a.conv_hi) * a.M;   // S * M for conv_hi >= L
    }
    if (a.touch) touch_ranges(a, &tr);
    else __syncthreads();
    const long long r_lo = lo_hi[0], r_hi = lo_hi[1];
    const int lane = threadIdx.x & 31, j = lane & 7, sub = lane >> 3;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    constexpr int D = 32 * NV;
    for (int img = 0; img < a.n_images; ++img) {
        const float* ws = reinterpret_cast<const float*>(a.grad_acc) + img * a.slice;
        float* wz = reinterpret_cast<float*>(a.grad_acc) + img * a.slice;
        T* gv = reinterpret_cast<T*>(a.conv_out) + img * a.slice;
        // class of row bb + lane: 0 untouched (sparse level), 1 written by its
        // pass, 2 in the workspace (every row of a dense level); 1 past the range.
        // Worked out one iteration ahead, so that its touch word's load overlaps
        // the rows of the iteration before.
        auto class_of = [&](long long bb) -> unsigned {
            const long long r = bb + lane;
            unsigned c = r < r_hi ? 2u : 1u;
            if (a.touch && r < r_hi) {
                const unsigned row = (unsigned)r;
                bool sp = false;
                for (int q = 0; q < tr.n; ++q) sp |= row >= tr.begin[q] && row < tr.end[q];
                if (sp) {
                    const unsigned pix = fdiv(row, a.div_m);
                    const unsigned id = ((unsigned)img * (unsigned)a.M + (row - pix * (unsigned)a.M)) * (unsigned)a.S + pix;
                    c = min(touch_bits(__ldg(a.touch + (id >> 4)), id), 2u);
                }
            }
            return c;
        };
        unsigned cls_next = class_of(r_lo + warp * 32);
        for (long long base = r_lo + warp * 32; base < r_hi; base += nwarps * 32) {
            const unsigned cls = cls_next;
            cls_next = class_of(base + nwarps * 32);
#pragma unroll
            for (int q0 = 0; q0 < 8; q0 += 4) {
                unsigned c4[4];
                float4 x[4][NV];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int rl = 4 * (q0 + q) + sub;   // the row's lane
                    c4[q] = __shfl_sync(0xffffffffu, cls, rl);
                    const long long e = (base + rl) * D + 4 * j;
#pragma unroll
                    for (int n = 0; n < NV; ++n)
                        x[q][n] = c4[q] == 2u ? __ldcs(reinterpret_cast<const float4*>(ws + e + 32 * n))
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (c4[q] == 1u) continue;
                    const long long e = (base + 4 * (q0 + q) + sub) * D + 4 * j;
#pragma unroll
                    for (int n = 0; n < NV; ++n) {
                        *reinterpret_cast<uint2*>(gv + e + 32 * n) =
                            make_uint2(pack2(x[q][n].x, x[q][n].y, tag), pack2(x[q][n].z, x[q][n].w, tag));
                        if (c4[q] == 2u && a.conv_rezero)
                            __stcs(reinterpret_cast<float4*>(wz + e + 32 * n), make_float4(0.f, 0.f, 0.f, 0.f));
                    }
                }
            }
        }
    }
}

// ws[i] = grad_value[i] (accumulating backward with the fp32 workspace)
template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_widen_kernel(const T* gv, float* ws, long long n) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nth = (long long)gridDim.x * blockDim.x;
    for (long long i = tid; i < n; i += nth) ws[i] = Elem<T>::to_f(gv[i]);
}

}  // namespace msda
