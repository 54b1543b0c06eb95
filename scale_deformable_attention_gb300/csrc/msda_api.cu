// msda_api.cu -- the C ABI declared in include/msda.h: host-side validation,
// launch planning and kernel launches on the caller's stream.  No call here
// synchronises, allocates device memory or reads device memory, except
// msda_device_errors() and msda_trace_read(), which are documented to wait.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "msda_internal.h"
#include "msda_launch.cuh"

using msda::KernelArgs;
using msda::Plan;

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;

thread_local char g_msg[512];

msda_status fail(msda_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

msda_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MSDA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

size_t esize(msda_dtype dt) { return dt == MSDA_F32 ? 4 : 2; }

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// ---- per-device state ----

struct DeviceInfo {
    bool init = false;
    unsigned long long ctx = 0;   // id of the context the fields below belong to (0: unknown)
    int sms = 0;
    int l2_bytes = 0;
    unsigned* err = nullptr;  // device address of g_msda_err on this device
    // second stream of the backward's overlapped rounding (created on first
    // use) and its fork / join events; side_mu serialises their use
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex side_mu;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

}  // namespace

// Device error word (see msda_device_errors).  One copy per device; its device
// address is looked up once per device context with cudaGetSymbolAddress.
__device__ unsigned int g_msda_err;

namespace {

// Id of the calling thread's current context (cuCtxGetId: never reused in a
// process), or 0 when the driver does not give one.
unsigned long long current_context_id() {
    using GetCurrent = PFN_cuCtxGetCurrent_v4000;
    using GetId = PFN_cuCtxGetId_v12000;
    static GetCurrent get_current = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? (GetCurrent)p
                   : (GetCurrent) nullptr;
    }();
    static GetId get_id = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? (GetId)p
                   : (GetId) nullptr;
    }();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&c) == CUDA_SUCCESS && c && get_id(c, &id) == CUDA_SUCCESS) return id;
    return 0;
}

msda_status device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MSDA_ERR_CUDA, "device ordinal %d out of range", dev);
    // a device reset (cudaDeviceReset) gives the device a new context: the
    // error word's address, the second stream and its events of the old one
    // are then stale and are looked up or created again (the old handles are
    // gone with their context and are not released)
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.init && ctx != 0 && ctx != d.ctx) {
        std::lock_guard<std::mutex> sl(d.side_mu);
        d.init = false;
        d.err = nullptr;
        d.side = nullptr;
        d.fork = d.join = nullptr;
    }
    if (!d.init) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_msda_err);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
        d.err = static_cast<unsigned*>(p);
        d.ctx = ctx;
        d.init = true;
    }
    *out = &d;
    return MSDA_OK;
}

// The device's second stream and fork / join events (created on first use).
msda_status side_stream(DeviceInfo* di) {
    if (di->side) return MSDA_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&di->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&di->fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&di->join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        if (di->join) cudaEventDestroy(di->join);
        if (di->fork) cudaEventDestroy(di->fork);
        if (di->side) cudaStreamDestroy(di->side);
        di->side = nullptr;
        di->fork = di->join = nullptr;
        return cuda_fail(e, "second stream of the backward");
    }
    return MSDA_OK;
}

// ---- kernel trace ----

struct Trace {
    int cap = 0, n = 0, dropped = 0, device = -1;
    bool paused = false;
    std::vector<cudaEvent_t> ev;
    std::vector<int> kernel;
    std::vector<int64_t> work;
};
Trace g_trace;
std::mutex g_trace_mu;

bool trace_active() {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    return g_trace.cap > 0 && !g_trace.paused;
}

struct TraceScope {
    int slot = -1;
    cudaStream_t st;
    TraceScope(cudaStream_t s) : st(s) {
        if (g_trace.cap == 0 || g_trace.paused) return;
        std::lock_guard<std::mutex> lk(g_trace_mu);
        if (g_trace.n >= g_trace.cap) {
            ++g_trace.dropped;
            return;
        }
        slot = g_trace.n++;
        cudaEventRecord(g_trace.ev[2 * slot], st);
    }
    void end(int kernel, int64_t work) {
        if (slot < 0) return;
        cudaEventRecord(g_trace.ev[2 * slot + 1], st);
        g_trace.kernel[slot] = kernel;
        g_trace.work[slot] = work;
    }
};

int ilog2_floor(int v) {
    int r = 0;
    while (v > 1) v >>= 1, ++r;
    return r;
}

// ---- tuning overrides (sweeps and tests), read once per process ----
// MSDA_TUNE is a comma-separated list of: C=<lanes>, P=<lanes>,
// params=bulk|ld|direct, generic, spec, notma, tma, pointparallel, nopdl,
// merge, nomerge, tiled, notiled, tp=<rows>, levelpass, nolevelpass, touch, notouch, tau=<n>, fold, nofold,
// overlap, nooverlap, nol2hint, c8, noc8.
// None of them changes results beyond the rounding order of the grad_value sums.

struct Tune {
    int C = 0, P = 0, params = -1;
    bool generic = false;  // force the generic kernels
    bool notma = false;    // no TMA-gather forward
    bool tma = false;      // TMA-gather forward whatever the size
    bool pointparallel = false;  // the point-parallel ablation forward (D = 32 only)
    bool pdl = true;       // forward and zero kernel as programmatic dependents (off: nopdl)
    bool spec = false;     // the specialised forward even where the generic one is faster
    int merge = -1;        // backward corner merge: -1 by density, 0 off (nomerge), 1 on (merge)
    int tiled = 0;         // FP32 accumulator on chip: 0 off (notiled, the default), 1 where the shape allows (tiled)
    int lg_tp = 0;         // rows per tile of the on-chip accumulator (tp=<power of two>; 0: by D)
    int levelpass = -1;    // backward one level at a time: -1 by size, 0 off (nolevelpass), 1 on (levelpass)
    int touch = 1;         // touch classes of the FP32 workspace's rows: 1 where they apply (touch), 0 off (notouch)
    int tau = 0;           // sparse-level bound of the touch classes (tau=<n>; 0: the default)
    int fold = -1;         // rounding folded into the level passes: -1 unless the touch classes apply, 0 off (nofold), 1 on (fold)
    int overlap = -1;      // touch classes: rounding of the finished rows on a second stream: -1 default, 0 off (nooverlap), 1 on (overlap)
    bool l2hint = true;    // TMA-gather forward: evict-first for levels over twice the L2 (off: nol2hint)
    int c8 = -1;           // backward into the FP32 workspace, eight lanes a unit: -1 default, 0 off (noc8), 1 on (c8)
};
const Tune& tune() {
    static Tune t = [] {
        Tune r;
        const char* s = getenv("MSDA_TUNE");
        if (!s) return r;
        char buf[256];
        snprintf(buf, sizeof(buf), "%s", s);
        for (char* tok = strtok(buf, ","); tok; tok = strtok(nullptr, ",")) {
            if (!strncmp(tok, "C=", 2)) r.C = atoi(tok + 2);
            else if (!strncmp(tok, "P=", 2)) r.P = atoi(tok + 2);
            else if (!strcmp(tok, "params=bulk")) r.params = msda::PARAMS_SMEM_BULK;
            else if (!strcmp(tok, "params=ld")) r.params = msda::PARAMS_SMEM_LD;
            else if (!strcmp(tok, "params=direct")) r.params = msda::PARAMS_DIRECT;
            else if (!strcmp(tok, "generic")) r.generic = true;
            else if (!strcmp(tok, "notma")) r.notma = true;
            else if (!strcmp(tok, "tma")) r.tma = true;
            else if (!strcmp(tok, "pointparallel")) r.pointparallel = true;
            else if (!strcmp(tok, "nopdl")) r.pdl = false;
            else if (!strcmp(tok, "spec")) r.spec = true;
            else if (!strcmp(tok, "merge")) r.merge = 1;
            else if (!strcmp(tok, "nomerge")) r.merge = 0;
            else if (!strcmp(tok, "tiled")) r.tiled = 1;
            else if (!strcmp(tok, "levelpass")) r.levelpass = 1;
            else if (!strcmp(tok, "nolevelpass")) r.levelpass = 0;
            else if (!strcmp(tok, "notiled")) r.tiled = 0;
            else if (!strncmp(tok, "tp=", 3)) r.lg_tp = ilog2_floor(atoi(tok + 3));
            else if (!strcmp(tok, "touch")) r.touch = 1;
            else if (!strcmp(tok, "notouch")) r.touch = 0;
            else if (!strncmp(tok, "tau=", 4)) r.tau = atoi(tok + 4);
            else if (!strcmp(tok, "nofold")) r.fold = 0;
            else if (!strcmp(tok, "fold")) r.fold = 1;
            else if (!strcmp(tok, "overlap")) r.overlap = 1;
            else if (!strcmp(tok, "nooverlap")) r.overlap = 0;
            else if (!strcmp(tok, "nol2hint")) r.l2hint = false;
            else if (!strcmp(tok, "c8")) r.c8 = 1;
            else if (!strcmp(tok, "noc8")) r.c8 = 0;
        }
        return r;
    }();
    return t;
}

// Multiplier and shift of msda::fdiv for divisor d >= 1 (numerators < 2^31).
msda::FastDiv fast_div(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return msda::FastDiv{(uint32_t)m, l};
}

int ilog2(int v) {
    int r = 0;
    while ((1 << r) < v) ++r;
    return r;
}

// ---- validation ----

struct Dims {
    int64_t B, S, M, D, L, K, Q;
    int64_t units;    // B*Q*M
    int64_t n_value;  // B*S*M*D
    int64_t n_param;  // B*Q*M*L*K
};

msda_status check_dims(msda_dtype dt, Dims& d) {
    if (dt != MSDA_F32 && dt != MSDA_F16 && dt != MSDA_BF16) return fail(MSDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    if (d.B < 0 || d.S < 0 || d.M < 0 || d.D < 0 || d.L < 0 || d.K < 0 || d.Q < 0)
        return fail(MSDA_ERR_INVALID_ARG, "negative size (B=%lld S=%lld M=%lld D=%lld L=%lld K=%lld Q=%lld)",
                    (long long)d.B, (long long)d.S, (long long)d.M, (long long)d.D, (long long)d.L, (long long)d.K,
                    (long long)d.Q);
    if (d.L == 0 || d.K == 0) return fail(MSDA_ERR_INVALID_ARG, "L and K must be at least 1");
    if (d.L > MSDA_MAX_LEVELS) return fail(MSDA_ERR_UNSUPPORTED, "L=%lld above %d", (long long)d.L, MSDA_MAX_LEVELS);
    if (d.K > MSDA_MAX_POINTS) return fail(MSDA_ERR_UNSUPPORTED, "K=%lld above %d", (long long)d.K, MSDA_MAX_POINTS);
    if (d.L * d.K > MSDA_MAX_SAMPLES)
        return fail(MSDA_ERR_UNSUPPORTED, "L*K=%lld above %d", (long long)(d.L * d.K), MSDA_MAX_SAMPLES);
    if (d.D > MSDA_MAX_CHANNELS) return fail(MSDA_ERR_UNSUPPORTED, "D=%lld above %d", (long long)d.D, MSDA_MAX_CHANNELS);
    int64_t t;
    if (!mul_ok(d.B, d.Q, &t) || !mul_ok(t, d.M, &d.units) || !mul_ok(d.units, d.L * d.K * 2, &t) ||
        !mul_ok(t, 8, &t) || !mul_ok(d.units, d.D, &t) || !mul_ok(t, 8, &t))
        return fail(MSDA_ERR_INVALID_ARG, "B*Q*M*L*K overflows 64 bits");
    d.n_param = d.units * d.L * d.K;
    if (!mul_ok(d.B, d.S, &t) || !mul_ok(t, d.M, &t) || !mul_ok(t, d.D, &d.n_value) || !mul_ok(d.n_value, 8, &t))
        return fail(MSDA_ERR_INVALID_ARG, "B*S*M*D overflows 64 bits");
    return MSDA_OK;
}

msda_status check_ptr(const void* p, bool needed, size_t align, const char* name) {
    if (!needed) return MSDA_OK;
    if (!p) return fail(MSDA_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, align)) return fail(MSDA_ERR_MISALIGNED, "%s is not aligned to %zu bytes", name, align);
    return MSDA_OK;
}

// ---- the FP32 accumulator on chip (msda_tiled.cuh) ----

// Layout of the on-chip FP32 accumulator's passes for a problem: rows per
// tile, tile counts, and its workspace (tile counters, offsets, cursors and
// the entry array, each 16-byte aligned).
struct TileLayout {
    int lg_tp = 0;
    int64_t tiles = 0, n_tiles = 0, n_entries = 0;
    size_t off_counts = 0, off_offsets = 0, off_cursor = 0, off_entries = 0, bytes = 0;
};

// Whether a backward with the FP32 accumulator takes the on-chip path, by its
// sizes alone (pointer alignment is checked at the call): 16-bit I/O, rows of
// 2..6 16-byte vectors of 8 channels (D = 32, 64 or 96), 32-bit offsets inside a
// batch image, fewer than 2^28 sampling points, sparse samples, the unfused
// operator -- and only when asked for (MSDA_TUNE=tiled).  Measured on GB300
// it is slower than the fp32 workspace in memory (encoder-scale stress
// backward 11.0 ms against 6.9 ms; decoder 152 us against 56 us): the
// accumulate pass is bound by the shared-memory atomic pipe (scalar fp32
// atomics, L1/shared throughput at 69% of peak), which does fewer channel
// additions per second than the L2 does with its 16-byte vector reductions,
// and the count and place passes wait on the counters of the coarse levels'
// few tiles.  Its workspace is ~26x smaller (329 MB against 8.56 GB there).
// Touch classes of the FP32 workspace's rows (msda_device.cuh, touch_sparse):
// 2 bits per (b, pixel, head) row, placed after the B*S*M*D fp32 sums at a
// 16-byte boundary.  A level is sparse at most kTouchTau corner contributions
// a row on average (tau=<n> overrides).
constexpr int kTouchTau = 4;
size_t touch_map_offset(int64_t n_value) { return ((size_t)n_value * 4 + 15) & ~(size_t)15; }
size_t touch_map_bytes(int64_t B, int64_t S, int64_t M) { return (size_t)((B * S * M + 63) / 64) * 16; }

bool tiled_layout(msda_dtype dt, msda_accum acc, const Dims& d, bool fused, TileLayout* tl) {
    const Tune& t = tune();
    if (t.tiled != 1 || fused || acc != MSDA_ACCUM_FP32 || (dt != MSDA_F16 && dt != MSDA_BF16)) return false;
    if (d.D != 32 && d.D != 64 && d.D != 96) return false;
    if (d.units <= 0 || d.n_value <= 0 || d.S * d.M * d.D > (1ll << 30)) return false;
    const int64_t n_samples = d.units * d.L * d.K;
    if (n_samples >= (1ll << 28)) return false;
    // rows per tile: 64 KB of fp32 sums (512 rows of D = 32)
    int lg = t.lg_tp > 0 ? t.lg_tp : ilog2_floor((int)(16384 / d.D));
    if (lg < 4) lg = 4;
    if (lg > 12) lg = 12;
    const int64_t tiles = (d.S + (1ll << lg) - 1) >> lg;
    const int64_t n_tiles = d.B * tiles * d.M;
    if (n_tiles >= (1ll << 31) - 1) return false;
    TileLayout r;
    r.lg_tp = lg;
    r.tiles = tiles;
    r.n_tiles = n_tiles;
    r.n_entries = 4 * n_samples;   // a point touches at most four tiles
    auto up16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
    r.off_counts = 0;
    r.off_offsets = up16(r.off_counts + (size_t)n_tiles * 4);
    r.off_cursor = up16(r.off_offsets + (size_t)(n_tiles + 1) * 4);
    r.off_entries = up16(r.off_cursor + (size_t)n_tiles * 4);
    r.bytes = up16(r.off_entries + (size_t)r.n_entries * 4);
    *tl = r;
    return true;
}

// ---- launch planning ----

// Lanes per row C and vectors per lane NV for nvec slots per row: the
// smallest lane waste with NV <= 4, ties towards C = 4.
void pick_c(int nvec, int* C, int* NV) {
    int bestC = 32, bestNV = (nvec + 31) / 32, bestWaste = 1 << 30, bestDist = 1 << 30;
    for (int c = 1; c <= 32; c <<= 1) {
        const int nv = (nvec + c - 1) / c;
        if (nv > 4) continue;
        const int waste = c * nv - nvec;
        const int dist = abs(ilog2(c) - 2);
        if (waste < bestWaste || (waste == bestWaste && dist < bestDist)) {
            bestC = c, bestNV = nv, bestWaste = waste, bestDist = dist;
        }
    }
    *C = bestC;
    *NV = bestNV;
}

msda_status make_plan(msda_dtype dt, const Dims& d, bool vec, int sms, bool backward, const void* loc,
                      const void* attn, Plan& pl, KernelArgs& a, bool fused = false, int lane_scale = 1,
                      bool nv4 = false) {
    const int es = (int)esize(dt);
    const int epv = vec ? 16 / es : 1;
    const int nvec = (int)(d.D / epv);
    int C, NV;
    pick_c(nvec, &C, &NV);
    if ((int64_t)C * NV * epv < d.D)
        return fail(MSDA_ERR_UNSUPPORTED, "D=%lld too large for %s rows (at most %d channels)", (long long)d.D,
                    vec ? "16-byte" : "unaligned", 32 * 4 * epv);
    const int LK = (int)(d.L * d.K);
    const Tune& t = tune();
    if (t.C > 0 && (t.C & (t.C - 1)) == 0 && t.C <= 32 && (int64_t)t.C * 4 * epv >= d.D) {
        C = t.C;
        NV = (nvec + C - 1) / C;
    }
    // point lanes: enough lanes to fill the GPU, within one warp (C*P <= 32)
    // and L*K.  Measured on GB300: ~768 lanes per SM (one resident wave at
    // these register counts) for both kernels, at least two point lanes per
    // unit for the backward, and twice the lanes for a forward whose gathers
    // come from DRAM (value larger than the L2: more loads in flight; odd-D
    // fp32 forward 108 -> 91 us).
    int P = 1;
    const int64_t target = (int64_t)sms * 768 * lane_scale;
    while (P * C < 32 && P * 2 <= LK && d.units * C * P < target) P *= 2;
    if (backward && P == 1 && C < 32 && LK >= 2) P = 2;
    if (t.P > 0 && (t.P & (t.P - 1)) == 0 && t.P * C <= 32) P = t.P;
    // fused backward: a block keeps <g, sampled> of all its samples in shared
    // memory (256 / (C*P) units * L*K floats): at most 32 KB
    if (fused && backward)
        while ((int64_t)(msda::kBlockThreads / (C * P)) * LK * 4 > 32768 && C * P < 32) P *= 2;
    const int tp = C * P;
    const int tpb = msda::kBlockThreads / tp;
    // parameter staging: one bulk copy when both chunks are 16-byte pieces
    const int64_t loc_unit = (int64_t)LK * 2 * es, attn_unit = (int64_t)LK * es;
    const bool v16 = (loc_unit % 16 == 0) && (attn_unit % 16 == 0) && aligned(loc, 16) && aligned(attn, 16);
    if (d.units >= (1ll << 31) || (d.Q * d.M) >= (1ll << 31))
        return fail(MSDA_ERR_UNSUPPORTED, "B*Q*M=%lld (b,q,m) units: at most 2^31-1 per call", (long long)d.units);
    const size_t smem = (size_t)(((tpb * loc_unit) + 15) / 16 * 16 + tpb * attn_unit + 16);
    int mode = v16 ? msda::PARAMS_SMEM_BULK : msda::PARAMS_SMEM_LD;
    if (t.params >= 0) mode = t.params;
    if (mode == msda::PARAMS_SMEM_BULK && !v16) mode = msda::PARAMS_SMEM_LD;
    if (smem > 48 * 1024) mode = msda::PARAMS_DIRECT;

    a.S = d.S;
    a.slice = d.S * d.M * d.D;
    a.M = (int)d.M;
    a.D = (int)d.D;
    a.L = (int)d.L;
    a.K = (int)d.K;
    a.LK = LK;
    a.n_units = (int)d.units;
    a.div_qm = fast_div((uint32_t)(d.Q * d.M));
    a.div_m = fast_div((uint32_t)d.M);
    a.div_k = fast_div((uint32_t)d.K);
    a.lc = ilog2(C);
    a.lp = ilog2(P);
    a.nvec = nvec;
    a.tpb = tpb;
    a.param_mode = mode;
    a.Q = (int)d.Q;
    a.det = nullptr;
    a.s_begin = 0;
    a.s_end = LK;

    pl.block = dim3(msda::kBlockThreads);
    const int64_t blocks = (d.units + tpb - 1) / tpb;
    if (blocks > 0x7fffffffLL) return fail(MSDA_ERR_UNSUPPORTED, "too many units (%lld)", (long long)d.units);
    pl.grid = dim3((unsigned)blocks);
    pl.smem = mode != msda::PARAMS_DIRECT ? smem : 0;
    // 32-bit element offsets inside one batch slice, with a row of margin
    pl.wide = a.slice > (1ll << 30);
    pl.nv = NV;
    pl.vec = vec;
    // four vectors a lane (256-byte rows) take the specialised kernels where
    // they were measured faster than the generic ones: the fp32 forward and
    // a backward into the fp32 workspace (the native 16-bit reductions are
    // faster in the generic kernel); the fused operator has no generic kernel
    pl.spec = vec && !pl.wide && C == msda::kC && nvec == C * NV && !t.generic &&
              (NV <= 3 || (NV == 4 && (fused || nv4)));
    pl.pdl = false;
    pl.fused = fused;
    a.ref = nullptr;
    a.gbuf_off = 0;
    // backward same-cell merge when samples are dense on the pyramid: on
    // average at least two corner contributions per pixel and head
    // (4*Q*L*K / S; measured: encoder 64 -> backward -19%, odd-D 2.6 -> -1.5%,
    // decoder 0.86 -> +10%)
    const double density = d.S > 0 ? 4.0 * (double)d.Q * (double)LK / (double)d.S : 0.0;
    pl.merge = t.merge >= 0 ? t.merge != 0 : density >= 2.0;
    a.rbuf_off = -1;
    if (fused && backward) {
        const int64_t gbuf = (int64_t)tpb * LK * 4;
        int64_t off = mode != msda::PARAMS_DIRECT ? (int64_t)((pl.smem + 15) / 16 * 16) : 0;
        if (off + gbuf > 48 * 1024) {  // drop the parameter staging
            a.param_mode = msda::PARAMS_DIRECT;
            off = 0;
        }
        a.gbuf_off = (int)off;
        pl.smem = (size_t)(off + gbuf);
        // grad_reference_points reduced in the kernel when a block holds
        // whole queries and the per-sample grad_loc buffer fits
        const int64_t rbuf = (int64_t)tpb * LK * 8, roff = (int64_t)((pl.smem + 15) / 16 * 16);
        if (tpb % d.M == 0 && roff + rbuf <= 48 * 1024) {
            a.rbuf_off = (int)roff;
            pl.smem = (size_t)(roff + rbuf);
        }
    }
    if (fused && !pl.spec)
        return fail(MSDA_ERR_UNSUPPORTED,
                    "the fused operator needs rows of whole 16-byte vectors with 16-byte aligned value / grad "
                    "pointers and D*esize in {64, 128, 192, 256} bytes (D = %lld)",
                    (long long)d.D);
    return MSDA_OK;
}

// Inputs / outputs of the fused operator that the plain one does not have.
struct Fused {
    const void* ref;  // reference points [B, Q, L, 2]
    void* grad_ref;   // their gradient (backward)
};

msda_status launch_ref_grad(msda_dtype dt, const Dims& d, const int64_t* shapes, const void* grad_off, void* grad_ref,
                            cudaStream_t st) {
    const long long BQ = d.B * d.Q;
    if (BQ * d.L == 0) return MSDA_OK;
    TraceScope ts(st);
    switch (dt) {
    case MSDA_F32:
        msda::launch_fused_ref_grad<float>(static_cast<const float*>(grad_off), static_cast<float*>(grad_ref), shapes,
                                           BQ, (int)d.M, (int)d.L, (int)d.K, st);
        break;
    case MSDA_F16:
        msda::launch_fused_ref_grad<__half>(static_cast<const __half*>(grad_off), static_cast<__half*>(grad_ref),
                                            shapes, BQ, (int)d.M, (int)d.L, (int)d.K, st);
        break;
    default:
        msda::launch_fused_ref_grad<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(grad_off),
                                                   static_cast<__nv_bfloat16*>(grad_ref), shapes, BQ, (int)d.M,
                                                   (int)d.L, (int)d.K, st);
        break;
    }
    ts.end(MSDA_KERNEL_CONVERT, BQ * d.L * 2);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MSDA_OK : cuda_fail(e, "reference-point gradient kernel launch");
}

// ---- tensor map of value for the TMA-gather forward ----

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encode_tiled() {
    static EncodeTiled fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiled) nullptr;
        return (EncodeTiled)p;
    }();
    return fn;
}

// value as a 2-D tensor of `rows` rows of D elements; one-row boxes of D
// elements (the gather4 box); coordinates outside read zeros.
bool value_tensor_map(msda_dtype dt, const void* value, int64_t rows, int64_t D, CUtensorMap* map) {
    EncodeTiled f = encode_tiled();
    if (!f) return false;
    const CUtensorMapDataType t = dt == MSDA_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : dt == MSDA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(D * (int64_t)esize(dt))};
    const cuuint32_t box[2] = {(cuuint32_t)D, 1u};
    const cuuint32_t estr[2] = {1u, 1u};
    return f(map, t, 2, const_cast<void*>(value), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int grid_for(int64_t n, int sms) {
    const int64_t want = (n + msda::kBlockThreads - 1) / msda::kBlockThreads;
    const int64_t cap = (int64_t)sms * 8;
    return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

// ---------------------------------------------------------------------------
// zero kernel (non-template; lives here, its only user)

namespace msda {
__global__ void __launch_bounds__(kBlockThreads) msda_zero_kernel(unsigned char* p, long long nbytes) {
    // Launched as a programmatic dependent, this grid may start before the
    // kernel ahead of it has finished: wait for it (and its memory) first.
    // Only then may the backward that depends on this grid start its gather
    // phase, so that phase never reads inputs an earlier kernel is still
    // writing; it waits for this grid before its first scatter.  Launched
    // normally, the wait returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // head up to 16-byte alignment, 16-byte body, tail
    const uintptr_t addr = reinterpret_cast<uintptr_t>(p);
    const long long head = min((long long)((16 - (addr & 15)) & 15), nbytes);
    const long long body = (nbytes - head) / 16;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nth = (long long)gridDim.x * blockDim.x;
    if (tid < head) p[tid] = 0;
    uint4* q = reinterpret_cast<uint4*>(p + head);
    for (long long i = tid; i < body; i += nth) q[i] = make_uint4(0u, 0u, 0u, 0u);
    const long long tail0 = head + body * 16;
    if (tid < nbytes - tail0) p[tail0 + tid] = 0;
}
}  // namespace msda

namespace {
msda_status launch_zero(void* p, int64_t nbytes, int sms, cudaStream_t st) {
    if (nbytes <= 0) return MSDA_OK;
    TraceScope ts(st);
    // two blocks per SM: stores need no registers in flight, and the rest of
    // the SM stays free for a backward that starts early (programmatic launch)
    const int64_t want = nbytes / 16 / msda::kBlockThreads + 1;
    const int grid = (int)(want < 2 * (int64_t)sms ? want : 2 * (int64_t)sms);
    unsigned char* ptr = static_cast<unsigned char*>(p);
    if (tune().pdl && !trace_active()) {
        // may start while the kernel ahead of it runs: it waits for that
        // kernel before storing, and only then lets its dependents start
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(msda::kBlockThreads);
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, msda::msda_zero_kernel, ptr, nbytes);
    } else {
        msda::msda_zero_kernel<<<grid, msda::kBlockThreads, 0, st>>>(ptr, nbytes);
    }
    ts.end(MSDA_KERNEL_ZERO, nbytes);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MSDA_OK : cuda_fail(e, "zero kernel launch");
}
}  // namespace

namespace msda {
msda_status set_error(msda_status s, const char* message) { return fail(s, "%s", message); }
void clear_error() { g_msg[0] = 0; }

size_t fp32_workspace_bytes(msda_dtype dt, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, int64_t K,
                            int64_t Q, bool touch) {
    Dims d{B, S, M, D, L, K, Q, 0, 0, 0};
    TileLayout tl;
    if (L >= 0 && K >= 0 && check_dims(dt, d) == MSDA_OK && tiled_layout(dt, MSDA_ACCUM_FP32, d, false, &tl))
        return tl.bytes;
    int64_t n;
    if (!mul_ok(B, S, &n) || !mul_ok(n, M, &n) || !mul_ok(n, D, &n) || !mul_ok(n, 4, &n)) return SIZE_MAX;
    // the fp32 sums, then the touch classes of their rows
    return touch ? touch_map_offset(n / 4) + touch_map_bytes(B, S, M) : (size_t)n;
}
}  // namespace msda

namespace {

// Deterministic accumulator: zero the workspace (header + int64 sums), take
// max |g| and max |A| into the header, run the backward into the int64 sums
// (launched as a programmatic dependent of the maxima kernel: its gather
// phase overlaps; the scale is read after griddepcontrol.wait), then convert.
msda_status backward_deterministic(msda_dtype dt, bool accumulate, const Dims& d, const void* value,
                                   const int64_t* shapes, const int64_t* starts, const void* loc, const void* attn,
                                   const void* grad_out, void* grad_value, void* grad_loc, void* grad_attn,
                                   void* workspace, size_t workspace_bytes, cudaStream_t st, const Fused* fz) {
    const size_t need = (size_t)d.n_value * 8 + (size_t)msda::kDetHeaderBytes;
    if (!workspace || workspace_bytes < need)
        return fail(MSDA_ERR_WORKSPACE, "the deterministic accumulator needs a %zu-byte workspace (got %zu at %p)",
                    need, workspace_bytes, workspace);
    if (!aligned(workspace, 16)) return fail(MSDA_ERR_WORKSPACE, "workspace is not 16-byte aligned");
    DeviceInfo* di = nullptr;
    msda_status s = device_info(&di);
    if (s) return s;
    const size_t es = esize(dt);
    msda::DetHeader* hdr = static_cast<msda::DetHeader*>(workspace);
    long long* sums = reinterpret_cast<long long*>(static_cast<unsigned char*>(workspace) + msda::kDetHeaderBytes);
    // the plan first: a call it rejects enqueues nothing
    const bool vec = (d.D * (int64_t)es) % 16 == 0 && aligned(value, 16) && aligned(grad_out, 16);
    KernelArgs a{};
    Plan pl{};
    if ((s = make_plan(dt, d, vec, di->sms, true, loc, attn, pl, a, fz != nullptr))) return s;
    if ((s = launch_zero(workspace, (int64_t)need, di->sms, st))) return s;
    {
        TraceScope ts(st);
        // softmax-normalised weights (fused operator) are at most 1: no scan
        const int64_t ng = d.units * d.D, na = fz ? 0 : d.n_param;
        const float ma0 = fz ? 1.f : 0.f;
        const int grid = grid_for((ng > na ? ng : na) / 8 + 1, di->sms);
        switch (dt) {
        case MSDA_F32:
            msda::launch_det_max<float>(static_cast<const float*>(grad_out), ng, static_cast<const float*>(attn), na,
                                        ma0, hdr, grid, st);
            break;
        case MSDA_F16:
            msda::launch_det_max<__half>(static_cast<const __half*>(grad_out), ng, static_cast<const __half*>(attn), na,
                                         ma0, hdr, grid, st);
            break;
        default:
            msda::launch_det_max<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(grad_out), ng,
                                                static_cast<const __nv_bfloat16*>(attn), na, ma0, hdr, grid, st);
            break;
        }
        ts.end(MSDA_KERNEL_CONVERT, ng + na);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "maxima kernel launch");
    }
    a.value = value;
    a.shapes = shapes;
    a.starts = starts;
    a.loc = loc;
    a.attn = attn;
    a.grad_out = grad_out;
    a.grad_acc = sums;
    a.grad_loc = grad_loc;
    a.grad_attn = grad_attn;
    a.err = di->err;
    a.det = hdr;
    if (fz) {
        a.ref = fz->ref;
        a.gref = fz->grad_ref;
    }
    pl.pdl = pl.spec && !trace_active();
    {
        TraceScope ts(st);
        switch (dt) {
        case MSDA_F32: msda::launch_backward<float, long long>(a, pl, st); break;
        case MSDA_F16: msda::launch_backward<__half, long long>(a, pl, st); break;
        default: msda::launch_backward<__nv_bfloat16, long long>(a, pl, st); break;
        }
        ts.end(MSDA_KERNEL_BACKWARD, d.units);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "backward kernel launch");
    }
    {
        TraceScope ts(st);
        const int grid = grid_for(d.n_value, di->sms);
        const long long qlk = d.Q * d.L * d.K;
        const int acc = accumulate ? 1 : 0;
        switch (dt) {
        case MSDA_F32:
            msda::launch_det_convert<float>(sums, static_cast<float*>(grad_value), d.n_value, hdr, qlk, acc, grid, st);
            break;
        case MSDA_F16:
            msda::launch_det_convert<__half>(sums, static_cast<__half*>(grad_value), d.n_value, hdr, qlk, acc, grid, st);
            break;
        default:
            msda::launch_det_convert<__nv_bfloat16>(sums, static_cast<__nv_bfloat16*>(grad_value), d.n_value, hdr, qlk,
                                                    acc, grid, st);
            break;
        }
        ts.end(MSDA_KERNEL_CONVERT, d.n_value);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "convert kernel launch");
    }
    if (fz && a.rbuf_off < 0) return launch_ref_grad(dt, d, shapes, grad_loc, fz->grad_ref, st);
    return MSDA_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI

extern "C" {

int msda_version(void) { return kVersion; }

const char* msda_last_error(void) { return g_msg; }

const char* msda_status_string(msda_status s) {
    switch (s) {
    case MSDA_OK: return "MSDA_OK";
    case MSDA_ERR_INVALID_ARG: return "MSDA_ERR_INVALID_ARG";
    case MSDA_ERR_UNSUPPORTED: return "MSDA_ERR_UNSUPPORTED";
    case MSDA_ERR_MISALIGNED: return "MSDA_ERR_MISALIGNED";
    case MSDA_ERR_WORKSPACE: return "MSDA_ERR_WORKSPACE";
    case MSDA_ERR_CUDA: return "MSDA_ERR_CUDA";
    }
    return "MSDA_STATUS_UNKNOWN";
}

const char* msda_kernel_name(int k) {
    switch (k) {
    case MSDA_KERNEL_FORWARD: return "forward";
    case MSDA_KERNEL_BACKWARD: return "backward";
    case MSDA_KERNEL_ZERO: return "zero";
    case MSDA_KERNEL_CONVERT: return "convert";
    case MSDA_KERNEL_TILE_COUNT: return "tile_count";
    case MSDA_KERNEL_TILE_SCAN: return "tile_scan";
    case MSDA_KERNEL_TILE_PLACE: return "tile_place";
    case MSDA_KERNEL_TILE_ACCUM: return "tile_accum";
    case MSDA_KERNEL_TOUCH: return "touch_count";
    }
    return "unknown";
}

}  // extern "C"

namespace {

// Forward after argument validation; `ref` non-NULL selects the fused operator
// (loc / attn then hold sampling offsets / attention logits).
msda_status forward_core(msda_dtype dt, const Dims& d, const void* value, const int64_t* spatial_shapes,
                         const int64_t* level_start_index, const void* loc, const void* attn, void* out,
                         cudaStream_t st, const void* ref) {
    msda_status s;
    const size_t es = esize(dt);
    DeviceInfo* di = nullptr;
    if ((s = device_info(&di))) return s;
    const bool vec = (d.D * (int64_t)es) % 16 == 0 && aligned(value, 16) && aligned(out, 16);
    // value larger than the L2: the gathers are served by DRAM
    const bool big = d.n_value * (int64_t)es > (int64_t)di->l2_bytes;
    KernelArgs a{};
    Plan pl{};
    if ((s = make_plan(dt, d, vec, di->sms, false, loc, attn, pl, a, ref != nullptr, big ? 2 : 1, dt == MSDA_F32)))
        return s;
    // One 16-bit slot per lane and few samples (at most 2^20): the generic
    // forward, whose lanes each set up their own samples, is faster than the
    // specialised one, whose setup-then-shuffle chain lengthens a latency-bound
    // wave.  Measured on GB300, bf16 D=32 decoder: B=1 10.3 -> 8.2 us,
    // B=4 14.2 -> 12.3 us, B=16 31.5 -> 28.7 us.  With many samples the forward
    // is issue-bound and the redundant setups cost more (encoder 111 -> 131 us);
    // with two slots or more the specialised one stays ahead (D=64 bf16 or
    // D=32 fp32: +3-4% generic).
    const int64_t samples = d.units * d.L * d.K;
    if (!ref && pl.spec && pl.nv == 1 && es == 2 && samples <= (1ll << 20) && !tune().spec && !tune().tma)
        pl.spec = false;
    a.value = value;
    a.shapes = spatial_shapes;
    a.starts = level_start_index;
    a.loc = loc;
    a.attn = attn;
    a.out = out;
    a.err = di->err;
    a.ref = ref;
    // TMA-gather forward: whole 16-byte rows of one slot per channel lane
    // (64-byte rows of bf16/fp16 D=32, fp32 D=16), L*K in {4, 8, 16, 32},
    // row coordinates of the [B*S*M, D] view below 2^31, and a value tensor
    // larger than the L2.  Measured on GB300: with value far above the L2
    // (gathers served by DRAM) the gathers are faster than 16-byte loads
    // (stress workload forward -24%); with value inside the L2 the load path
    // is faster (encoder workload forward +59% with gathers); with 192-byte
    // rows the staged corners limit a block to 12% occupancy and the load
    // path is faster (odd-D fp32 forward 107 us with gathers, 91 us without).
    const int LK = (int)(d.L * d.K);
    CUtensorMap map;
    const bool tma = !ref && pl.spec && pl.nv == 1 && !tune().notma && (big || tune().tma) &&
                     (LK == 4 || LK == 8 || LK == 16 || LK == 32) && d.B * d.S * d.M < (1ll << 31) &&
                     value_tensor_map(dt, value, d.B * d.S * d.M, d.D, &map);
    TraceScope ts(st);
    if (!ref && tune().pointparallel && d.D == msda::kPpD && msda::kBlockThreads % LK == 0 && !pl.wide) {
        const int upb = msda::kBlockThreads / LK;
        const unsigned grid = (unsigned)((d.units + upb - 1) / upb);
        switch (dt) {
        case MSDA_F32: msda::launch_forward_pointparallel<float>(a, grid, st); break;
        case MSDA_F16: msda::launch_forward_pointparallel<__half>(a, grid, st); break;
        default: msda::launch_forward_pointparallel<__nv_bfloat16>(a, grid, st); break;
        }
    } else if (tma) {
        a.lc = 2;
        a.lp = ilog2(LK / 4);
        a.l2_bytes = tune().l2hint ? di->l2_bytes : 0;
        const int64_t groups = (d.units * LK + 31) / 32;
        const unsigned grid = (unsigned)((groups + msda::kTmaWarps - 1) / msda::kTmaWarps);
        switch (dt) {
        case MSDA_F32: msda::launch_forward_tma<float>(a, map, pl.nv, grid, st); break;
        case MSDA_F16: msda::launch_forward_tma<__half>(a, map, pl.nv, grid, st); break;
        default: msda::launch_forward_tma<__nv_bfloat16>(a, map, pl.nv, grid, st); break;
        }
    } else {
        pl.pdl = tune().pdl && !trace_active();
        switch (dt) {
        case MSDA_F32: msda::launch_forward<float>(a, pl, st); break;
        case MSDA_F16: msda::launch_forward<__half>(a, pl, st); break;
        default: msda::launch_forward<__nv_bfloat16>(a, pl, st); break;
        }
    }
    ts.end(MSDA_KERNEL_FORWARD, d.units);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MSDA_OK : cuda_fail(e, "forward kernel launch");
}

}  // namespace

extern "C" {

msda_status msda_forward(msda_dtype dt, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, int64_t K, int64_t Q,
                         const void* value, const int64_t* spatial_shapes, const int64_t* level_start_index,
                         const void* sampling_locations, const void* attention_weights, void* out,
                         msda_stream_t stream) {
    g_msg[0] = 0;
    Dims d{B, S, M, D, L, K, Q, 0, 0, 0};
    msda_status s = check_dims(dt, d);
    if (s != MSDA_OK) return s;
    if (d.units == 0 || D == 0) return MSDA_OK;  // empty output: nothing to launch
    const size_t es = esize(dt);
    if ((s = check_ptr(value, d.n_value > 0, es, "value")) ||
        (s = check_ptr(spatial_shapes, true, 8, "spatial_shapes")) ||
        (s = check_ptr(level_start_index, true, 8, "level_start_index")) ||
        (s = check_ptr(sampling_locations, true, es, "sampling_locations")) ||
        (s = check_ptr(attention_weights, true, es, "attention_weights")) || (s = check_ptr(out, true, es, "out")))
        return s;
    return forward_core(dt, d, value, spatial_shapes, level_start_index, sampling_locations, attention_weights, out,
                        reinterpret_cast<cudaStream_t>(stream), nullptr);
}

msda_status msda_forward_fused(msda_dtype dt, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, int64_t K,
                               int64_t Q, const void* value, const int64_t* spatial_shapes,
                               const int64_t* level_start_index, const void* reference_points,
                               const void* sampling_offsets, const void* attention_logits, void* out,
                               msda_stream_t stream) {
    g_msg[0] = 0;
    Dims d{B, S, M, D, L, K, Q, 0, 0, 0};
    msda_status s = check_dims(dt, d);
    if (s != MSDA_OK) return s;
    if (d.units == 0 || D == 0) return MSDA_OK;
    const size_t es = esize(dt);
    if ((s = check_ptr(value, d.n_value > 0, es, "value")) ||
        (s = check_ptr(spatial_shapes, true, 8, "spatial_shapes")) ||
        (s = check_ptr(level_start_index, true, 8, "level_start_index")) ||
        (s = check_ptr(reference_points, true, es, "reference_points")) ||
        (s = check_ptr(sampling_offsets, true, es, "sampling_offsets")) ||
        (s = check_ptr(attention_logits, true, es, "attention_logits")) || (s = check_ptr(out, true, es, "out")))
        return s;
    return forward_core(dt, d, value, spatial_shapes, level_start_index, sampling_offsets, attention_logits, out,
                        reinterpret_cast<cudaStream_t>(stream), reference_points);
}

msda_accum msda_resolve_accum(msda_dtype dt, msda_accum mode, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L,
                              int64_t K, int64_t Q) {
    (void)B, (void)M, (void)D;
    if (mode == MSDA_ACCUM_DETERMINISTIC) return mode;
    if (dt == MSDA_F32) return MSDA_ACCUM_NATIVE;
    if (mode == MSDA_ACCUM_NATIVE || mode == MSDA_ACCUM_FP32) return mode;
    // AUTO: native 16-bit reductions unless many samples land on each pixel,
    // where per-add rounding of bf16 would dominate the error.
    const double contrib = S > 0 ? 4.0 * (double)Q * (double)L * (double)K / (double)S : 0.0;
    if (dt == MSDA_BF16 && contrib > 8.0) return MSDA_ACCUM_FP32;
    return MSDA_ACCUM_NATIVE;
}

size_t msda_backward_workspace_size(msda_dtype dt, msda_accum mode, int64_t B, int64_t S, int64_t M, int64_t D,
                                    int64_t L, int64_t K, int64_t Q) {
    if (B < 0 || S < 0 || M < 0 || D < 0) return 0;
    if (mode == MSDA_ACCUM_DETERMINISTIC) {
        int64_t n;
        if (!mul_ok(B, S, &n) || !mul_ok(n, M, &n) || !mul_ok(n, D, &n) || !mul_ok(n, 8, &n)) return SIZE_MAX;
        return (size_t)(n + msda::kDetHeaderBytes);
    }
    if (dt != MSDA_F16 && dt != MSDA_BF16) return 0;
    const msda_accum acc = msda_resolve_accum(dt, mode, B, S, M, D, L, K, Q);
    if (acc != MSDA_ACCUM_FP32) return 0;
    return msda::fp32_workspace_bytes(dt, B, S, M, D, L, K, Q, true);
}

}  // extern "C"

namespace {

// Whether the backward runs one pass per pyramid level: the specialised
// kernels of the unfused operator, several levels, value or the grad_value
// accumulator larger than the L2, and enough units that each pass still
// fills the GPU many times over (a pass gives each unit's level one team of
// kC lanes).  Measured on GB300: encoder-scale stress backward 3.52 -> 3.15 ms
// (FP32 accumulator) and 2.54 -> 2.19 ms (native); the odd-D workload (value
// 267 MB, 57,600 units: under one wave per pass) 178 -> 232 us, hence the
// unit rule.  MSDA_TUNE=levelpass / nolevelpass override both rules.
bool level_passes(msda_dtype dt, const Dims& d, const Plan& pl, bool fused, bool use_ws, int l2_bytes, int sms) {
    const int t = tune().levelpass;
    if (t == 0 || !pl.spec || fused || d.L < 2) return false;
    if (t == 1) return true;
    const int64_t es = (int64_t)esize(dt);
    const int64_t value_bytes = d.n_value * es, acc_bytes = d.n_value * (use_ws ? 4 : es);
    const bool big = value_bytes > (int64_t)l2_bytes || acc_bytes > (int64_t)l2_bytes;
    return big && d.units * msda::kC >= (int64_t)sms * 768 * 8;
}

// Launch shape of a level pass: K samples per unit, so P point lanes with
// P * kC >= K (one lane per sample when K <= kC), and direct parameter loads
// (a pass reads one level's parameters of each unit: a strided subset).
void level_pass_plan(const Dims& d, Plan& pl, KernelArgs& a) {
    const int C = 1 << a.lc;
    int P = 1;
    while (P * msda::kC < (int)d.K && C * P < 32) P *= 2;
    a.lp = ilog2(P);
    a.tpb = msda::kBlockThreads / (C * P);
    a.param_mode = msda::PARAMS_DIRECT;
    pl.smem = 0;
    pl.grid = dim3((unsigned)((d.units + a.tpb - 1) / a.tpb));
}

// Backward with the FP32 accumulator on chip (msda_tiled.cuh): the gather
// kernel without its scatter (grad_sampling_locations, grad_attention_weights),
// then count, scan, place and accumulate for grad_value.  Nothing is enqueued
// unless the workspace and the plan pass.
msda_status backward_tiled(msda_dtype dt, bool accumulate, const Dims& d, const TileLayout& tl, const void* value,
                           const int64_t* shapes, const int64_t* starts, const void* loc, const void* attn,
                           const void* grad_out, void* grad_value, void* grad_loc, void* grad_attn, void* workspace,
                           size_t workspace_bytes, cudaStream_t st) {
    if (!workspace || workspace_bytes < tl.bytes)
        return fail(MSDA_ERR_WORKSPACE,
                    "FP32 accumulation needs a %zu-byte workspace (got %zu at %p; with 16-byte aligned value, "
                    "grad_out and grad_value)", tl.bytes, workspace_bytes, workspace);
    if (!aligned(workspace, 16)) return fail(MSDA_ERR_WORKSPACE, "workspace is not 16-byte aligned");
    msda_status s;
    DeviceInfo* di = nullptr;
    if ((s = device_info(&di))) return s;
    KernelArgs a{};
    Plan pl{};
    if ((s = make_plan(dt, d, true, di->sms, true, loc, attn, pl, a, false))) return s;
    // (its gather and accumulate kernels exist for one to three vectors a lane)
    if (!pl.spec || pl.nv > 3)
        return fail(MSDA_ERR_UNSUPPORTED, "on-chip FP32 accumulation needs the specialised kernels");
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    msda::TileArgs t{};
    t.loc = loc;
    t.attn = attn;
    t.grad_out = grad_out;
    t.grad_value = grad_value;
    t.shapes = shapes;
    t.starts = starts;
    t.err = di->err;
    t.counts = reinterpret_cast<unsigned*>(ws + tl.off_counts);
    t.offsets = reinterpret_cast<unsigned*>(ws + tl.off_offsets);
    t.cursor = reinterpret_cast<unsigned*>(ws + tl.off_cursor);
    t.entries = reinterpret_cast<unsigned*>(ws + tl.off_entries);
    t.S = d.S;
    t.M = (int)d.M;
    t.D = (int)d.D;
    t.L = (int)d.L;
    t.K = (int)d.K;
    t.LK = (int)(d.L * d.K);
    t.Q = (int)d.Q;
    t.n_samples = (int)(d.units * d.L * d.K);
    t.div_lk = fast_div((uint32_t)(d.L * d.K));
    t.div_k = fast_div((uint32_t)d.K);
    t.div_qm = fast_div((uint32_t)(d.Q * d.M));
    t.div_m = fast_div((uint32_t)d.M);
    t.lg_tp = tl.lg_tp;
    t.tiles = (int)tl.tiles;
    t.n_tiles = (int)tl.n_tiles;
    t.accumulate = accumulate ? 1 : 0;

    // gather: grad_sampling_locations, grad_attention_weights
    a.value = value;
    a.shapes = shapes;
    a.starts = starts;
    a.loc = loc;
    a.attn = attn;
    a.grad_out = grad_out;
    a.grad_acc = nullptr;
    a.grad_loc = grad_loc;
    a.grad_attn = grad_attn;
    a.err = di->err;
    pl.pdl = false;
    auto launched = [&](const char* what) -> msda_status {
        cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? MSDA_OK : cuda_fail(e, what);
    };
    {
        TraceScope ts(st);
        switch (dt) {
        case MSDA_F16: msda::launch_backward_gather<__half>(a, pl, st); break;
        default: msda::launch_backward_gather<__nv_bfloat16>(a, pl, st); break;
        }
        ts.end(MSDA_KERNEL_BACKWARD, d.units);
        if ((s = launched("backward gather kernel launch"))) return s;
    }
    if ((s = launch_zero(t.counts, tl.n_tiles * 4, di->sms, st))) return s;
    {
        TraceScope ts(st);
        if (dt == MSDA_F16) msda::launch_tile_count<__half>(t, st);
        else msda::launch_tile_count<__nv_bfloat16>(t, st);
        ts.end(MSDA_KERNEL_TILE_COUNT, t.n_samples);
        if ((s = launched("tile count kernel launch"))) return s;
    }
    {
        TraceScope ts(st);
        if (dt == MSDA_F16) msda::launch_tile_scan<__half>(t, st);
        else msda::launch_tile_scan<__nv_bfloat16>(t, st);
        ts.end(MSDA_KERNEL_TILE_SCAN, t.n_tiles);
        if ((s = launched("tile scan kernel launch"))) return s;
    }
    {
        TraceScope ts(st);
        if (dt == MSDA_F16) msda::launch_tile_place<__half>(t, st);
        else msda::launch_tile_place<__nv_bfloat16>(t, st);
        ts.end(MSDA_KERNEL_TILE_PLACE, t.n_samples);
        if ((s = launched("tile place kernel launch"))) return s;
    }
    {
        TraceScope ts(st);
        if (dt == MSDA_F16) msda::launch_tile_accum<__half>(t, pl.nv, st);
        else msda::launch_tile_accum<__nv_bfloat16>(t, pl.nv, st);
        ts.end(MSDA_KERNEL_TILE_ACCUM, t.n_tiles);
        if ((s = launched("tile accumulate kernel launch"))) return s;
    }
    return MSDA_OK;
}

// Backward after argument validation; `fz` non-NULL selects the fused
// operator (sampling_locations / attention_weights then hold offsets /
// logits, their gradients go to grad_sampling_locations / grad_attention_weights).
msda_status backward_core(msda_dtype dt, msda_accum mode, unsigned flags, const Dims& d, const void* value,
                          const int64_t* spatial_shapes, const int64_t* level_start_index,
                          const void* sampling_locations, const void* attention_weights, const void* grad_out,
                          void* grad_value, void* grad_sampling_locations, void* grad_attention_weights,
                          void* workspace, size_t workspace_bytes, cudaStream_t st, const Fused* fz) {
    const int64_t B = d.B, S = d.S, M = d.M, D = d.D, L = d.L, K = d.K, Q = d.Q;
    msda_status s;
    const size_t es = esize(dt);
    const bool work = d.units > 0 && D > 0;
    const bool accumulate = (flags & MSDA_BWD_ACCUMULATE) != 0;
    const bool ws_zeroed = (flags & MSDA_BWD_WORKSPACE_ZEROED) != 0;
    const msda_accum acc = msda_resolve_accum(dt, mode, B, S, M, D, L, K, Q);
    if (acc == MSDA_ACCUM_DETERMINISTIC && work && d.n_value > 0)
        return backward_deterministic(dt, accumulate, d, value, spatial_shapes, level_start_index, sampling_locations,
                                      attention_weights, grad_out, grad_value, grad_sampling_locations,
                                      grad_attention_weights, workspace, workspace_bytes, st, fz);
    const bool use_ws = dt != MSDA_F32 && acc == MSDA_ACCUM_FP32 && work && d.n_value > 0;
    TileLayout tl;
    if (use_ws && tiled_layout(dt, acc, d, fz != nullptr, &tl)) {
        const bool aligned16 = aligned(value, 16) && aligned(grad_out, 16) && aligned(grad_value, 16);
        if (aligned16)
            return backward_tiled(dt, accumulate, d, tl, value, spatial_shapes, level_start_index, sampling_locations,
                                  attention_weights, grad_out, grad_value, grad_sampling_locations,
                                  grad_attention_weights, workspace, workspace_bytes, st);
        // unaligned pointers: the workspace path below, with its B*S*M*D*4 bytes
    }
    if (use_ws) {
        const size_t need = (size_t)d.n_value * 4;
        if (!workspace || workspace_bytes < need)
            return fail(MSDA_ERR_WORKSPACE, "FP32 accumulation needs a %zu-byte workspace (got %zu at %p)", need,
                        workspace_bytes, workspace);
        if (!aligned(workspace, 16)) return fail(MSDA_ERR_WORKSPACE, "workspace is not 16-byte aligned");
    }
    const bool empty_params = d.n_param == 0 || (fz && d.B * d.Q * d.L == 0);
    if (d.n_value == 0 && !work && empty_params) return MSDA_OK;

    DeviceInfo* di = nullptr;
    if ((s = device_info(&di))) return s;
    if (!work) {
        // no output channels or no units: every gradient is zero
        if (!accumulate && (s = launch_zero(grad_value, d.n_value * (int64_t)es, di->sms, st))) return s;
        if ((s = launch_zero(grad_sampling_locations, d.n_param * 2 * (int64_t)es, di->sms, st))) return s;
        if ((s = launch_zero(grad_attention_weights, d.n_param * (int64_t)es, di->sms, st))) return s;
        if (fz && (s = launch_zero(fz->grad_ref, d.B * d.Q * d.L * 2 * (int64_t)es, di->sms, st))) return s;
        return MSDA_OK;
    }

    void* acc_buf = use_ws ? workspace : grad_value;
    const bool vec = (D * (int64_t)es) % 16 == 0 && aligned(value, 16) && aligned(grad_out, 16) &&
                     aligned(acc_buf, 16);
    KernelArgs a{};
    Plan pl{};
    // the plan first: a call it rejects enqueues nothing
    if ((s = make_plan(dt, d, vec, di->sms, true, sampling_locations, attention_weights, pl, a, fz != nullptr, 1,
                       use_ws)))
        return s;

    // grad_value (or the workspace) must start from zero / from grad_value
    if (!use_ws) {
        if (!accumulate && (s = launch_zero(grad_value, d.n_value * (int64_t)es, di->sms, st))) return s;
    } else if (!accumulate) {
        // a workspace that holds zeros on entry (MSDA_BWD_WORKSPACE_ZEROED) needs no clearing pass
        if (!ws_zeroed && (s = launch_zero(workspace, d.n_value * 4, di->sms, st))) return s;
    } else {
        TraceScope ts(st);
        const int grid = grid_for(d.n_value, di->sms);
        if (dt == MSDA_F16)
            msda::launch_widen<__half>(static_cast<const __half*>(grad_value), static_cast<float*>(workspace),
                                       d.n_value, grid, st);
        else
            msda::launch_widen<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(grad_value),
                                              static_cast<float*>(workspace), d.n_value, grid, st);
        ts.end(MSDA_KERNEL_CONVERT, d.n_value);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "widen kernel launch");
    }

    // the zero kernel was the last thing enqueued by this call: the backward
    // may be launched as its programmatic dependent (not while tracing, whose
    // events sit between the two launches)
    const bool zeroed_here = !accumulate && (use_ws ? !ws_zeroed : d.n_value > 0);
    a.value = value;
    a.shapes = spatial_shapes;
    a.starts = level_start_index;
    a.loc = sampling_locations;
    a.attn = attention_weights;
    a.grad_out = grad_out;
    a.grad_acc = acc_buf;
    a.grad_loc = grad_sampling_locations;
    a.grad_attn = grad_attention_weights;
    a.err = di->err;
    if (fz) {
        a.ref = fz->ref;
        a.gref = fz->grad_ref;
    }
    pl.pdl = pl.spec && zeroed_here && !trace_active();
    // One pass per pyramid level when value or the accumulator exceeds the
    // L2: each pass's rows of the batch images in flight (value and
    // grad_value or its workspace) then stay in the L2 between the touches of
    // one corner row by different samples, instead of being fetched again.
    const int passes = level_passes(dt, d, pl, fz != nullptr, use_ws, di->l2_bytes, di->sms) ? (int)d.L : 1;
    if (passes > 1) level_pass_plan(d, pl, a);
    // With one pass per level, the FP32 workspace's rows below the first row
    // of level 2 are final once passes 0 and 1 are done: the passes from
    // level 2 on (L2-bound, DRAM mostly idle) round them with extra blocks,
    // and the rounding pass afterwards handles the remaining rows only.
    constexpr int kFoldLevel = 2;
    constexpr long long kFoldChunk = 1 << 16;   // workspace elements per folding block
    // rounding by the tail kernel (msda_round_rows_kernel): one pass per level,
    // 16-byte aligned grad_value, whole 8-element groups
    const bool tail_ok = passes > 1 && use_ws && pl.spec && fz == nullptr && aligned(grad_value, 16) &&
                         (d.S * d.M * d.D) % 8 == 0;
    // Touch classes (msda_device.cuh, touch_sparse): a count pass first classes
    // the rows of the sparse levels; a row with one contribution is then
    // written directly and the rounding reads the workspace rows with several
    // only.  Needs the classes' bytes after the fp32 sums
    // (msda_backward_workspace_size counts them); a workspace of the sums
    // alone runs without.
    const int tau = tune().tau > 0 ? tune().tau : kTouchTau;
    const size_t map_off = touch_map_offset(d.n_value), map_bytes = touch_map_bytes(d.B, d.S, d.M);
    const bool touch = tail_ok && !accumulate && tune().touch != 0 && 4 * d.Q * d.K <= (int64_t)tau * d.S &&
                       d.B * d.S * d.M < (1ll << 31) && d.n_param < (1ll << 31) && d.D % 8 == 0 &&
                       workspace_bytes >= map_off + map_bytes;
    unsigned* touch_map = touch ? reinterpret_cast<unsigned*>(static_cast<unsigned char*>(workspace) + map_off)
                                : nullptr;
    // Eight lanes a unit for the passes into the FP32 workspace (msda_bwd8_kernel):
    // a corner row's load and its reduction take one L1 request each instead of
    // two.  Measured on GB300, stress backward with the touch classes 4.50 ->
    // 4.35 ms (the passes of levels 2 and 3, bound by those requests, 0.58 ->
    // 0.53 ms alone).  It has no folding blocks, and without the touch classes
    // the four-lane passes with the folded rounding are faster (5.60 against
    // 5.69 ms), so by default it runs with the classes only (c8 forces it).
    pl.c8 = passes > 1 && use_ws && pl.spec && fz == nullptr && !pl.merge &&
            (tune().c8 > 0 || (tune().c8 < 0 && touch));
    if (pl.c8) {
        a.lc = 3;
        a.lp = 0;
        a.tpb = msda::kBlockThreads / 8;
        pl.smem = 0;
        pl.grid = dim3((unsigned)((d.units + a.tpb - 1) / a.tpb));
    }
    // With the rounding folded into the passes from level 2 on, the rows below
    // level 2's first row, final once passes 0 and 1 are done, are rounded by
    // extra blocks of those passes, and the tail kernel rounds the rest.  Not
    // with the touch classes by default: the passes of the coarse levels are
    // bound by their own sampling (long-scoreboard waits on the L2), and the
    // folding blocks, which then read few workspace rows, only take their slots
    // (and msda_bwd8_kernel has no folding blocks).
    const int tf = tune().fold;
    const bool fold = tail_ok && d.L > kFoldLevel && !pl.c8 && (tf > 0 || (tf < 0 && !touch));
    // With the touch classes, the rows below level 2's first row are final once
    // passes 0 and 1 are done: a second stream rounds them while the passes
    // from level 2 on run (those are bound by the L2, the rounding by DRAM), and
    // the tail kernel afterwards rounds the rest.  (The count of levels 1 to 3
    // on that stream beside pass 0 gained nothing: pass 0 slowed by what the
    // count saved.)  Measured on GB300, stress backward: 4.67 -> 4.50 ms (the
    // second stream's rounding at the tail
    // kernel's grid; at one, two or four blocks an SM it takes 7.0, 4.1 and
    // 3.1 ms and the backward 8.9, 6.2 and 5.2 ms; the passes on a
    // highest-priority stream and the rounding in short blocks on a
    // lowest-priority one keep the passes at their own speed, but the rounding
    // then waits for them: 4.52 ms).
    const bool overlap = touch && !fold && d.L > kFoldLevel && tune().overlap != 0;
    if (overlap) {
        if ((s = side_stream(di))) return s;
    }
    std::unique_lock<std::mutex> side_lock(di->side_mu, std::defer_lock);
    if (overlap) side_lock.lock();
    long long fold_chunks = 0;
    if (fold || touch) {
        a.conv_level = kFoldLevel;   // the folded rounding's cut
        // the tail kernel: every row, or the rows from level 2's first row on
        // when the folded rounding or the second stream rounds those below
        a.conv_lo = fold || overlap ? kFoldLevel : -1;
        a.conv_hi = (int)d.L;
        a.conv_rezero = ws_zeroed ? 1 : 0;
        a.conv_out = grad_value;
        a.n_images = (int)d.B;
    }
    if (fold) {
        a.conv_chunk = kFoldChunk;
        a.conv_chunks_per_image = (a.slice + kFoldChunk - 1) / kFoldChunk;
        fold_chunks = d.B * a.conv_chunks_per_image;
    }
    cudaStream_t wst = st;   // the stream of the count, the passes and the tail rounding
    if (touch) {
        a.touch = touch_map;
        a.touch_tau = tau;
        a.touch_out = grad_value;
        a.div_lk = fast_div((uint32_t)(d.L * d.K));
        a.div_d8 = fast_div((uint32_t)(d.D / 8));
        // the first pass reads the classes before its griddepcontrol.wait
        pl.pdl = false;
        if (!ws_zeroed && (s = launch_zero(touch_map, (int64_t)map_bytes, di->sms, st))) return s;
        TraceScope ts(wst);
        const int grid = (int)((d.n_param + msda::kBlockThreads - 1) / msda::kBlockThreads);
        if (dt == MSDA_F16) msda::launch_touch_count<__half>(a, grid, wst);
        else msda::launch_touch_count<__nv_bfloat16>(a, grid, wst);
        ts.end(MSDA_KERNEL_TOUCH, d.n_param);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "touch count kernel launch");
    }
    for (int pass = 0; pass < passes; ++pass) {
        Plan lp = pl;
        a.conv_blocks = 0;
        if (passes > 1) {
            a.s_begin = (int)(pass * d.K);
            a.s_end = (int)((pass + 1) * d.K);
            if (pass > 0) lp.pdl = false;
            if (fold && pass >= kFoldLevel) {
                // this pass's share of the chunks, interleaved with its sampling blocks
                const int hosts = passes - kFoldLevel, h = pass - kFoldLevel;
                const long long c0 = fold_chunks * h / hosts, c1 = fold_chunks * (h + 1) / hosts;
                const long long ns = pl.grid.x, nc = c1 - c0;
                if (nc > 0 && ns + nc < 0x7fffffffLL) {
                    a.conv_blocks = (int)nc;
                    a.conv_first = c0;
                    a.conv_every = (int)((ns + nc) / nc);
                    lp.grid = dim3((unsigned)(ns + nc));
                }
            }
        }
        TraceScope ts(wst);
        switch (dt) {
        case MSDA_F32: msda::launch_backward<float, float>(a, lp, wst); break;
        case MSDA_F16:
            if (use_ws) msda::launch_backward<__half, float>(a, lp, wst);
            else msda::launch_backward<__half, __half>(a, lp, wst);
            break;
        default:
            if (use_ws) msda::launch_backward<__nv_bfloat16, float>(a, lp, wst);
            else msda::launch_backward<__nv_bfloat16, __nv_bfloat16>(a, lp, wst);
            break;
        }
        ts.end(MSDA_KERNEL_BACKWARD, d.units);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "backward kernel launch");
        // fork: the rows below level 2's first row on the second stream, once
        // passes 0 and 1 are done (forking the rows below level 1's first row
        // after pass 0 and the next after pass 1 measured slower: 4.18 against
        // 4.13 ms, level 0's rounding then beside the DRAM-bound pass 1)
        if (overlap && pass == kFoldLevel - 1) {
            KernelArgs ab = a;
            ab.conv_lo = -1;
            ab.conv_hi = kFoldLevel;
            if ((e = cudaEventRecord(di->fork, wst)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(di->side, di->fork, 0)) != cudaSuccess)
                return cuda_fail(e, "fork to the second stream");
            TraceScope tb(di->side);
            const int grid = grid_for(d.n_value / 8 / 16 + 1, di->sms);
            if (dt == MSDA_F16) msda::launch_round_rows<__half>(ab, pl.nv, grid, di->side);
            else msda::launch_round_rows<__nv_bfloat16>(ab, pl.nv, grid, di->side);
            tb.end(MSDA_KERNEL_CONVERT, d.n_value);
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "convert kernel launch");
            if ((e = cudaEventRecord(di->join, di->side)) != cudaSuccess)
                return cuda_fail(e, "join of the second stream");
        }
    }
    if (use_ws && (fold || touch)) {
        // the rows from the first row of level 2 on (with the folded
        // rounding), else every row, in every batch image
        TraceScope ts(wst);
        const int grid = grid_for(d.n_value / 8 / 16 + 1, di->sms);
        if (dt == MSDA_F16) msda::launch_round_rows<__half>(a, pl.nv, grid, wst);
        else msda::launch_round_rows<__nv_bfloat16>(a, pl.nv, grid, wst);
        ts.end(MSDA_KERNEL_CONVERT, d.n_value);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "convert kernel launch");
        if (overlap && (e = cudaStreamWaitEvent(st, di->join, 0)) != cudaSuccess)
            return cuda_fail(e, "join of the second stream");
        // a workspace that came in holding zeros leaves holding zeros
        if (touch && ws_zeroed && (s = launch_zero(touch_map, (int64_t)map_bytes, di->sms, st))) return s;
        if (fz && a.rbuf_off < 0) return launch_ref_grad(dt, d, spatial_shapes, grad_sampling_locations, fz->grad_ref, st);
        return MSDA_OK;
    }
    if (use_ws) {
        TraceScope ts(st);
        const int cvec = aligned(grad_value, 16) ? 1 : 0;
        const int grid = grid_for(d.n_value / 8 + 1, di->sms);
        // with MSDA_BWD_WORKSPACE_ZEROED the pass leaves the workspace holding zeros
        const int rezero = ws_zeroed ? 1 : 0;
        if (dt == MSDA_F16)
            msda::launch_convert<__half>(static_cast<float*>(workspace), static_cast<__half*>(grad_value), d.n_value,
                                         cvec, rezero, grid, st);
        else
            msda::launch_convert<__nv_bfloat16>(static_cast<float*>(workspace),
                                                static_cast<__nv_bfloat16*>(grad_value), d.n_value, cvec, rezero,
                                                grid, st);
        ts.end(MSDA_KERNEL_CONVERT, d.n_value);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "convert kernel launch");
    }
    if (fz && a.rbuf_off < 0) return launch_ref_grad(dt, d, spatial_shapes, grad_sampling_locations, fz->grad_ref, st);
    return MSDA_OK;
}


// Validation shared by the two backward entry points.
msda_status backward_checks(msda_dtype dt, msda_accum mode, unsigned flags, Dims& d, const void* value,
                            const int64_t* spatial_shapes, const int64_t* level_start_index, const void* p_loc,
                            const char* n_loc, const void* p_attn, const char* n_attn, const void* grad_out,
                            void* grad_value, void* g_loc, const char* n_gloc, void* g_attn, const char* n_gattn) {
    msda_status s = check_dims(dt, d);
    if (s != MSDA_OK) return s;
    if (mode != MSDA_ACCUM_AUTO && mode != MSDA_ACCUM_NATIVE && mode != MSDA_ACCUM_FP32 &&
        mode != MSDA_ACCUM_DETERMINISTIC)
        return fail(MSDA_ERR_INVALID_ARG, "unknown accumulator mode %d", (int)mode);
    if (flags & ~(MSDA_BWD_ACCUMULATE | MSDA_BWD_WORKSPACE_ZEROED))
        return fail(MSDA_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    const size_t es = esize(dt);
    const bool work = d.units > 0 && d.D > 0;
    if ((s = check_ptr(grad_value, d.n_value > 0, es, "grad_value"))) return s;
    if ((s = check_ptr(g_loc, d.n_param > 0, es, n_gloc)) || (s = check_ptr(g_attn, d.n_param > 0, es, n_gattn)))
        return s;
    if (work) {
        if ((s = check_ptr(value, d.n_value > 0, es, "value")) ||
            (s = check_ptr(spatial_shapes, true, 8, "spatial_shapes")) ||
            (s = check_ptr(level_start_index, true, 8, "level_start_index")) ||
            (s = check_ptr(p_loc, true, es, n_loc)) || (s = check_ptr(p_attn, true, es, n_attn)) ||
            (s = check_ptr(grad_out, true, es, "grad_out")))
            return s;
    }
    return MSDA_OK;
}

}  // namespace

extern "C" {

msda_status msda_backward(msda_dtype dt, msda_accum mode, unsigned flags, int64_t B, int64_t S, int64_t M, int64_t D,
                          int64_t L, int64_t K, int64_t Q, const void* value, const int64_t* spatial_shapes,
                          const int64_t* level_start_index, const void* sampling_locations,
                          const void* attention_weights, const void* grad_out, void* grad_value,
                          void* grad_sampling_locations, void* grad_attention_weights, void* workspace,
                          size_t workspace_bytes, msda_stream_t stream) {
    g_msg[0] = 0;
    Dims d{B, S, M, D, L, K, Q, 0, 0, 0};
    msda_status s = backward_checks(dt, mode, flags, d, value, spatial_shapes, level_start_index, sampling_locations,
                                    "sampling_locations", attention_weights, "attention_weights", grad_out,
                                    grad_value, grad_sampling_locations, "grad_sampling_locations",
                                    grad_attention_weights, "grad_attention_weights");
    if (s != MSDA_OK) return s;
    return backward_core(dt, mode, flags, d, value, spatial_shapes, level_start_index,
                         sampling_locations, attention_weights, grad_out, grad_value, grad_sampling_locations,
                         grad_attention_weights, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                         nullptr);
}

msda_status msda_backward_fused(msda_dtype dt, msda_accum mode, unsigned flags, int64_t B, int64_t S, int64_t M,
                                int64_t D, int64_t L, int64_t K, int64_t Q, const void* value,
                                const int64_t* spatial_shapes, const int64_t* level_start_index,
                                const void* reference_points, const void* sampling_offsets,
                                const void* attention_logits, const void* grad_out, void* grad_value,
                                void* grad_reference_points, void* grad_sampling_offsets,
                                void* grad_attention_logits, void* workspace, size_t workspace_bytes,
                                msda_stream_t stream) {
    g_msg[0] = 0;
    Dims d{B, S, M, D, L, K, Q, 0, 0, 0};
    msda_status s = backward_checks(dt, mode, flags, d, value, spatial_shapes, level_start_index, sampling_offsets,
                                    "sampling_offsets", attention_logits, "attention_logits", grad_out, grad_value,
                                    grad_sampling_offsets, "grad_sampling_offsets", grad_attention_logits,
                                    "grad_attention_logits");
    if (s != MSDA_OK) return s;
    const size_t es = esize(dt);
    const bool nref = d.B * d.Q * d.L > 0;
    if ((s = check_ptr(grad_reference_points, nref, es, "grad_reference_points")) ||
        (s = check_ptr(reference_points, nref && d.units > 0 && d.D > 0, es, "reference_points")) ||
        (s = check_ptr(spatial_shapes, nref, 8, "spatial_shapes")))
        return s;
    const Fused fz{reference_points, grad_reference_points};
    return backward_core(dt, mode, flags, d, value, spatial_shapes, level_start_index,
                         sampling_offsets, attention_logits, grad_out, grad_value, grad_sampling_offsets,
                         grad_attention_logits, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                         &fz);
}

msda_status msda_device_errors(uint32_t* bits, int clear) {
    g_msg[0] = 0;
    if (!bits) return fail(MSDA_ERR_INVALID_ARG, "bits is NULL");
    DeviceInfo* di = nullptr;
    msda_status s = device_info(&di);
    if (s) return s;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_msda_err, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
    *bits = v;
    if (clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_msda_err, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    }
    return MSDA_OK;
}

msda_status msda_trace_enable(int capacity) {
    g_msg[0] = 0;
    if (capacity < 0) return fail(MSDA_ERR_INVALID_ARG, "negative trace capacity");
    std::lock_guard<std::mutex> lk(g_trace_mu);
    for (cudaEvent_t ev : g_trace.ev) cudaEventDestroy(ev);
    g_trace = Trace();
    if (capacity == 0) return MSDA_OK;
    g_trace.ev.resize(2 * (size_t)capacity);
    for (auto& ev : g_trace.ev) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) {
            for (cudaEvent_t x : g_trace.ev)
                if (x) cudaEventDestroy(x);
            g_trace = Trace();
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    g_trace.kernel.assign(capacity, -1);
    g_trace.work.assign(capacity, 0);
    g_trace.cap = capacity;
    return MSDA_OK;
}

void msda_trace_pause(int paused) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace.paused = paused != 0;
}

int msda_trace_read(msda_trace_record* records, int max_records, int* dropped) {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    const int n = g_trace.n < max_records ? g_trace.n : max_records;
    for (int i = 0; i < n; ++i) {
        float ms = -1.f;
        if (cudaEventSynchronize(g_trace.ev[2 * i + 1]) == cudaSuccess)
            cudaEventElapsedTime(&ms, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]);
        records[i].kernel = g_trace.kernel[i];
        records[i].ms = ms;
        records[i].work = g_trace.work[i];
    }
    if (dropped) *dropped = g_trace.dropped + (g_trace.n - n);
    g_trace.n = 0;
    g_trace.dropped = 0;
    return n;
}

}  // extern "C"
