// msda_static_ws.cu -- msda_backward_static_workspace: the fp32-accumulator
// backward with its scratch buffer in a fixed device array instead of a
// caller-provided workspace.
//
// Who needs it: callers that hand this library only their input and output
// buffers and cannot obtain more device memory at that point -- an inference
// engine plugin whose enqueue hook receives pointers but no allocator, a
// real-time loop that forbids allocation after start-up, or code enqueuing
// work under a memory budget fixed by someone else.  msda_backward with the
// FP32 accumulator needs B*S*M*D*4 bytes of scratch; here that scratch is the
// array below, sized at compile time.
//
// The array is a device global: every GPU on which it is used holds
// MSDA_STATIC_WORKSPACE_BYTES until the process exits.  Its device address
// is looked up once per device (cudaGetSymbolAddress, with that device
// current) by the first call made on that device; make that first call before
// any stream capture.  All calls share the one array, so calls whose work can
// overlap on the GPU (different streams, or several threads) race on it and
// must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "msda_internal.h"

namespace {
constexpr size_t kStaticFloats = MSDA_STATIC_WORKSPACE_BYTES / sizeof(float);
constexpr int kMaxDevices = 64;
}  // namespace

// The scratch array itself (one copy per device).
static __device__ __align__(256) float g_msda_static_workspace[kStaticFloats];

namespace {
std::mutex g_mu;
void* g_addr[kMaxDevices];

// Device address of the array on the current device (looked up once per device).
msda_status static_workspace_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return msda::set_error(MSDA_ERR_CUDA, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_msda_static_workspace);
        if (e != cudaSuccess) return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return MSDA_OK;
}
}  // namespace

extern "C" msda_status msda_backward_static_workspace(
    msda_dtype dt, unsigned flags, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, int64_t K, int64_t Q,
    const void* value, const int64_t* spatial_shapes, const int64_t* level_start_index,
    const void* sampling_locations, const void* attention_weights, const void* grad_out, void* grad_value,
    void* grad_sampling_locations, void* grad_attention_weights, msda_stream_t stream) {
    void* ws = nullptr;
    const bool sizes_ok = B >= 0 && S >= 0 && M >= 0 && D >= 0 && Q >= 0;
    if ((dt == MSDA_F16 || dt == MSDA_BF16) && sizes_ok) {
        int64_t n = 0;
        if (__builtin_mul_overflow(B, S, &n) || __builtin_mul_overflow(n, M, &n) || __builtin_mul_overflow(n, D, &n) ||
            n > (int64_t)kStaticFloats)
            return msda::set_error(MSDA_ERR_WORKSPACE,
                                   "msda_backward_static_workspace: B*S*M*D exceeds the static workspace of "
                                   "MSDA_STATIC_WORKSPACE_BYTES / 4 elements");
        if (n > 0) {
            msda_status s = static_workspace_address(&ws);
            if (s != MSDA_OK) return s;
        }
    }
    // The existing backward clears the workspace (or widens grad_value into it
    // when accumulating) before its kernel, so nothing carries over between calls.
    return msda_backward(dt, MSDA_ACCUM_FP32, flags, B, S, M, D, L, K, Q, value, spatial_shapes, level_start_index,
                         sampling_locations, attention_weights, grad_out, grad_value, grad_sampling_locations,
                         grad_attention_weights, ws, ws ? MSDA_STATIC_WORKSPACE_BYTES : 0, stream);
}
