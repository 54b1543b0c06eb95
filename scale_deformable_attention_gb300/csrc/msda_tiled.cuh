// msda_tiled.cuh -- the FP32 grad_value accumulator kept on chip.
//
// The pages accumulate grad_value in an FP32 buffer in memory and round it
// to the I/O dtype afterwards (course ch. 5, "The fix: accumulate in FP32,
// downcast at the end").  In memory that buffer is twice the size of
// grad_value and costs a zeroing pass, a read-modify-write by the L2 for every
// reduction, and a rounding pass: for the encoder-scale pyramid (4.3 GB of
// bf16 grad_value) about 38 GB of DRAM traffic.  Here the FP32 sums live in
// shared memory instead, one tile of the pyramid at a time (the shared-memory
// pre-reduction idea the README credits mmcv with, "Benchmarks"), and
// grad_value is written exactly once:
//
//   1. count:  every sampling point adds 1 to the counter of each tile its
//              inside corners fall in (a tile is TP consecutive pyramid rows
//              of one (b, m) image, so a point touches 1 to 4 tiles);
//   2. scan:   exclusive prefix sum of the counters: each tile's range in an
//              entry array;
//   3. place:  every point writes one entry (point index << 4 | corner mask)
//              into the range of each of its tiles;
//   4. accum:  one block per tile zeroes TP x D fp32 in shared memory, adds
//              A * w_corner * g for every entry of its range (shared-memory
//              atomics; the bilinear setup is recomputed from the point's
//              location with the same binary32 arithmetic), and writes its
//              TP rows of grad_value once, rounded once to the dtype (plus
//              the old value when accumulating).
//
// grad_sampling_locations and grad_attention_weights come from the gather
// kernel of the backward, run without its scatter.  The corner and cell
// decisions of the three passes are the same function of the same inputs,
// so a point's corners land in the tiles its entries name; the accumulate
// pass still checks every row against its tile and drops (and reports) one
// that is not, and the place pass drops an entry beyond its tile's range.
#pragma once

#include "msda_device.cuh"

namespace msda {

struct TileArgs {
    const void* loc;         // [B, Q, M, L, K, 2]
    const void* attn;        // [B, Q, M, L, K]
    const void* grad_out;    // [B, Q, M*D]
    void* grad_value;        // [B, S, M, D]
    const int64_t* shapes;
    const int64_t* starts;
    unsigned* err;
    unsigned* counts;        // [n_tiles]
    unsigned* offsets;       // [n_tiles + 1]
    unsigned* cursor;        // [n_tiles]
    unsigned* entries;       // [<= 4 * n_samples]
    long long S;
    int M, D, L, K, LK, Q;
    int n_samples;           // B*Q*M*L*K  (< 2^28)
    FastDiv div_lk, div_k, div_qm, div_m;
    int lg_tp;               // log2 of the rows per tile
    int tiles;               // tiles per (b, m) image: ceil(S / TP)
    int n_tiles;             // B * tiles * M
    int accumulate;          // add the old grad_value before rounding
};

constexpr unsigned kErrTile = 4u;   // an entry outside its tile or range (never expected)

// Level table of the block, as the other kernels check it.
__device__ __forceinline__ void tile_levels(const TileArgs& a, Level* lv) {
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
}

// The cell of a point (binary32 pixel coordinate, floor, validity; as
// sample_setup): the pyramid row of corner (y0, x0), the level width, the
// inside-corner mask and the fractional offsets.
struct Cell {
    int pix;        // start + y0 * W + x0 (meaningful for the inside corners)
    int W;
    unsigned mask;  // bit k: corner k = (y0 + k/2, x0 + k%2) inside the level
    float lx, ly;
};

__device__ __forceinline__ Cell point_cell(const Level& L, float x, float y) {
    const float xi = __fmaf_rn(x, L.fW, -0.5f);
    const float yi = __fmaf_rn(y, L.fH, -0.5f);
    const float x0f = floorf(xi), y0f = floorf(yi);
    const bool vx0 = L.ok && x0f >= 0.f && x0f < L.fW;
    const bool vx1 = L.ok && x0f >= -1.f && x0f < L.fW - 1.f;
    const bool vy0 = y0f >= 0.f && y0f < L.fH;
    const bool vy1 = y0f >= -1.f && y0f < L.fH - 1.f;
    const int x0 = (vx0 || vx1) ? (int)x0f : 0;
    const int y0 = (vy0 || vy1) ? (int)y0f : 0;
    Cell c;
    c.W = L.W;
    c.pix = (int)L.start + y0 * L.W + x0;
    c.mask = (unsigned)(vy0 && vx0) | ((unsigned)(vy0 && vx1) << 1) | ((unsigned)(vy1 && vx0) << 2) |
             ((unsigned)(vy1 && vx1) << 3);
    c.lx = xi - x0f;
    c.ly = yi - y0f;
    return c;
}

__device__ __forceinline__ int corner_row(const Cell& c, int k) { return c.pix + (k & 1) + (k >> 1) * c.W; }

// Point p's location, weight, level and unit u = (b*Q + q)*M + m.
template <typename T>
__device__ __forceinline__ void tile_point(const TileArgs& a, int p, float& x, float& y, float& w, int& l,
                                           uint32_t& u) {
    u = fdiv((uint32_t)p, a.div_lk);
    const int s = p - (int)u * a.LK;
    l = (int)fdiv((uint32_t)s, a.div_k);
    const T* pl = reinterpret_cast<const T*>(a.loc) + 2ll * p;
    x = ldg_f(pl);
    y = ldg_f(pl + 1);
    w = ldg_f(reinterpret_cast<const T*>(a.attn) + p);
}

// Global index of tile t of image (b, m): tiles are ordered (b, t, m), so the
// M blocks of one row range are neighbours and together write one contiguous
// range of grad_value.
__device__ __forceinline__ int tile_index(const TileArgs& a, uint32_t b, uint32_t m, int t) {
    return ((int)b * a.tiles + t) * a.M + (int)m;
}

// The distinct tiles of a cell's inside corners, with the corners in each.
__device__ __forceinline__ int cell_tiles(const Cell& c, int lg_tp, int (&t)[4], unsigned (&mk)[4]) {
    int n = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (!((c.mask >> k) & 1u)) continue;
        const int tk = corner_row(c, k) >> lg_tp;
        int j = 0;
        while (j < n && t[j] != tk) ++j;
        if (j == n) {
            t[n] = tk;
            mk[n] = 0u;
            ++n;
        }
        mk[j] |= 1u << k;
    }
    return n;
}

// 1. count (one thread per point)
template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_tile_count_kernel(const TileArgs a) {
    __shared__ Level lv[MSDA_MAX_LEVELS];
    tile_levels(a, lv);
    __syncthreads();
    const int p = blockIdx.x * kBlockThreads + threadIdx.x;
    if (p >= a.n_samples) return;
    float x, y, w;
    int l;
    uint32_t u;
    tile_point<T>(a, p, x, y, w, l, u);
    const Cell c = point_cell(lv[l], x, y);
    if (!c.mask) return;
    const uint32_t b = fdiv(u, a.div_qm), m = u - fdiv(u, a.div_m) * (uint32_t)a.M;
    int t[4];
    unsigned mk[4];
    const int n = cell_tiles(c, a.lg_tp, t, mk);
    for (int j = 0; j < n; ++j)
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(a.counts + tile_index(a, b, m, t[j]))
                     : "memory");
}

// 2. exclusive scan of the counters (one block of 1024 threads): offsets[i] =
// sum of counts[0..i), offsets[n] = total; the cursors start at the offsets.
constexpr int kScanThreads = 1024;

template <typename T>   // instantiated once per dtype's translation unit (T is unused)
__global__ void __launch_bounds__(kScanThreads) msda_tile_scan_kernel(const TileArgs a) {
    __shared__ unsigned wsum[kScanThreads / 32];
    const int n = a.n_tiles;
    const int per = (n + kScanThreads - 1) / kScanThreads;
    const int i0 = min(n, threadIdx.x * per), i1 = min(n, i0 + per);
    unsigned s = 0;
    for (int i = i0; i < i1; ++i) s += a.counts[i];
    // block-wide exclusive scan of the per-thread sums
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned v = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        wsum[lane] = v;   // inclusive over warps
    }
    __syncthreads();
    unsigned run = (warp ? wsum[warp - 1] : 0u) + incl - s;
    for (int i = i0; i < i1; ++i) {
        a.offsets[i] = run;
        a.cursor[i] = run;
        run += a.counts[i];
    }
    if (threadIdx.x == kScanThreads - 1) a.offsets[n] = wsum[31];
}

// 3. place (one thread per point)
template <typename T>
__global__ void __launch_bounds__(kBlockThreads) msda_tile_place_kernel(const TileArgs a) {
    __shared__ Level lv[MSDA_MAX_LEVELS];
    tile_levels(a, lv);
    __syncthreads();
    const int p = blockIdx.x * kBlockThreads + threadIdx.x;
    if (p >= a.n_samples) return;
    float x, y, w;
    int l;
    uint32_t u;
    tile_point<T>(a, p, x, y, w, l, u);
    const Cell c = point_cell(lv[l], x, y);
    if (!c.mask) return;
    const uint32_t b = fdiv(u, a.div_qm), m = u - fdiv(u, a.div_m) * (uint32_t)a.M;
    int t[4];
    unsigned mk[4];
    const int n = cell_tiles(c, a.lg_tp, t, mk);
    for (int j = 0; j < n; ++j) {
        const int ti = tile_index(a, b, m, t[j]);
        const unsigned slot = atomicAdd(a.cursor + ti, 1u);
        if (slot < a.offsets[ti + 1]) a.entries[slot] = ((unsigned)p << 4) | mk[j];
        else atomicOr(a.err, kErrTile);
    }
}

// Entry batches a warp keeps in flight in the accumulate pass (8 entries
// per batch: a team of kC lanes per entry).
constexpr int kTileBatches = 4;

// Column of channel ch of shared-memory row r: rotated by r inside its group
// of 32, so that the teams of a warp, adding to different rows, spread over
// the banks.
__device__ __forceinline__ int tile_col(int ch, int r) { return (ch & ~31) | ((ch + r) & 31); }

// 4. accumulate + write (one block per tile)
template <typename T, int NV>
__global__ void __launch_bounds__(kBlockThreads) msda_tile_accum_kernel(const TileArgs a) {
    constexpr int EPV = 16 / sizeof(T);
    constexpr int D = kC * NV * EPV;
    using S_ = Slot<T, EPV>;
    __shared__ Level lv[MSDA_MAX_LEVELS];
    extern __shared__ __align__(16) float acc[];   // [TP][D]
    const int TP = 1 << a.lg_tp;
    tile_levels(a, lv);
    {
        float4* a4 = reinterpret_cast<float4*>(acc);
        for (int i = threadIdx.x; i < TP * D / 4; i += kBlockThreads) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    const int ti = blockIdx.x;
    const uint32_t m = (uint32_t)(ti % a.M);
    const int bt = ti / a.M;
    const int tt = bt % a.tiles;
    const uint32_t b = (uint32_t)(bt / a.tiles);
    const int row0 = tt << a.lg_tp;
    const int e0 = (int)a.offsets[ti], e1 = (int)a.offsets[ti + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = lane & (kC - 1), es = lane >> 2;   // channel lane, entry slot of the warp's batch
    constexpr int kWarps = kBlockThreads / 32;
    for (int base = e0 + warp * 8 * kTileBatches; base < e1; base += kWarps * 8 * kTileBatches) {
        unsigned ent[kTileBatches];
#pragma unroll
        for (int i = 0; i < kTileBatches; ++i) {
            const int j = base + i * 8 + es;
            ent[i] = j < e1 ? __ldg(a.entries + j) : 0u;   // mask 0: nothing to add
        }
        float xs[kTileBatches], ys[kTileBatches], ws[kTileBatches];
        int ls[kTileBatches];
        typename S_::Raw graw[kTileBatches][NV];
#pragma unroll
        for (int i = 0; i < kTileBatches; ++i) {
            const int p = (int)(ent[i] >> 4);
            uint32_t u;
            tile_point<T>(a, p, xs[i], ys[i], ws[i], ls[i], u);
            const T* go = reinterpret_cast<const T*>(a.grad_out) + (long long)u * D + c * EPV;
#pragma unroll
            for (int n = 0; n < NV; ++n) graw[i][n] = S_::load_raw(go + n * kC * EPV);
        }
#pragma unroll
        for (int i = 0; i < kTileBatches; ++i) {
            const unsigned mask = ent[i] & 15u;
            if (!mask) continue;
            const Cell cl = point_cell(lv[ls[i]], xs[i], ys[i]);
            float wk[4];
            corner_weights(cl.lx, cl.ly, wk);
            float g[NV][EPV];
#pragma unroll
            for (int n = 0; n < NV; ++n) S_::unpack(graw[i][n], g[n]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (!((mask >> k) & 1u)) continue;
                const int r = corner_row(cl, k) - row0;
                if (r < 0 || r >= TP || !((cl.mask >> k) & 1u)) {
                    atomicOr(a.err, kErrTile);
                    continue;
                }
                const float cf = ws[i] * wk[k];
                float* rowp = acc + r * D;
#pragma unroll
                for (int n = 0; n < NV; ++n)
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        const int ch = n * kC * EPV + c * EPV + e;
                        atomicAdd(rowp + tile_col(ch, r), cf * g[n][e]);
                    }
            }
        }
    }
    __syncthreads();
    // write the tile's rows of grad_value, rounded once
    constexpr int SL = D / EPV;   // 16-byte slots per row
    T* gv = reinterpret_cast<T*>(a.grad_value);
    for (int i = threadIdx.x; i < TP * SL; i += kBlockThreads) {
        const int r = i / SL, sl = i - r * SL;
        const long long gp = (long long)row0 + r;
        if (gp >= a.S) break;   // rows beyond the pyramid: nothing to write (i grows with r)
        float v[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[e] = acc[r * D + tile_col(sl * EPV + e, r)];
        T* dst = gv + (((long long)b * a.S + gp) * a.M + m) * D + sl * EPV;
        if (a.accumulate) {
            float old[EPV];
            S_::load(dst, old);
#pragma unroll
            for (int e = 0; e < EPV; ++e) v[e] += old[e];
        }
        S_::store(dst, v);
    }
}

}  // namespace msda
