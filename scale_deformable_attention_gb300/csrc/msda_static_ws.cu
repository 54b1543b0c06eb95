// msda_static_ws.cu -- msda_backward_static_workspace: the fp32-accumulator
// backward with its scratch buffer in a fixed device array instead of a
// caller-provided workspace.
//
// Who needs it: callers that hand this library only their input and output
// buffers and cannot obtain more device memory at that point -- an inference
// engine plugin whose enqueue hook receives pointers but no allocator, a
// real-time loop that forbids allocation after start-up, or code enqueuing
// work under a memory budget fixed by someone else.  msda_backward with the
// FP32 accumulator needs B*S*M*D*4 bytes of scratch for its fp32 sums (plus
// the optional touch classes of their rows); here that scratch is the array
// below, sized at compile time.
//
// The array is a device global of this translation unit's module: it
// occupies MSDA_STATIC_WORKSPACE_BYTES on every device where that module is
// loaded, until the process exits.  With lazy module loading (the CUDA
// default) that is a device on which this entry point has looked the array
// up; with CUDA_MODULE_LOADING=EAGER it is every device the process creates a
// context on, whether or not this entry point is ever called.
//
// The array's device address is looked up with cudaGetSymbolAddress, with the
// caller's device current, on every call made while the stream is not being
// captured (so a context destroyed and recreated, e.g. by cudaDeviceReset,
// never leaves a stale address behind).  While the stream is being captured
// into a CUDA graph the address remembered from the last uncaptured call on
// that device is used, so make one uncaptured call on each device before
// capturing.  All calls share the one array, so calls whose work can overlap
// on the GPU (different streams, or several threads) race on it and must be
// serialised by the caller.
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

// Device address of the array on the current device.
msda_status static_workspace_address(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return msda::set_error(MSDA_ERR_CUDA, "device ordinal out of range");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
    std::lock_guard<std::mutex> lk(g_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_msda_static_workspace);
        if (e != cudaSuccess) return msda::set_error(MSDA_ERR_CUDA, cudaGetErrorString(e));
        g_addr[dev] = p;
    } else if (!g_addr[dev]) {
        return msda::set_error(MSDA_ERR_CUDA,
                               "msda_backward_static_workspace: make one call on this device outside stream "
                               "capture before capturing it");
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
    // The array is cleared by every call that uses it; a caller cannot vouch
    // for its contents, so the flag that says the workspace holds zeros is
    // not for this entry point.
    if (flags & MSDA_BWD_WORKSPACE_ZEROED)
        return msda::set_error(MSDA_ERR_INVALID_ARG,
                               "msda_backward_static_workspace: MSDA_BWD_WORKSPACE_ZEROED does not apply to the "
                               "library's own array");
    // First the call without scratch.  msda_backward checks every argument
    // before it enqueues anything, and asks for a workspace (MSDA_ERR_WORKSPACE)
    // only after they all pass and only when there is something to sample;
    // any other status, OK included, is the call's result as it stands.
    msda_status s = msda_backward(dt, MSDA_ACCUM_FP32, flags, B, S, M, D, L, K, Q, value, spatial_shapes,
                                  level_start_index, sampling_locations, attention_weights, grad_out, grad_value,
                                  grad_sampling_locations, grad_attention_weights, nullptr, 0, stream);
    if (s != MSDA_ERR_WORKSPACE) return s;
    // the fp32 sums must fit; the touch classes are used when they fit too
    const size_t need = msda::fp32_workspace_bytes(dt, B, S, M, D, L, K, Q, false);
    if (need > (size_t)MSDA_STATIC_WORKSPACE_BYTES)
        return msda::set_error(MSDA_ERR_WORKSPACE,
                               "msda_backward_static_workspace: the FP32 accumulator needs more scratch than the "
                               "static workspace holds (B*S*M*D*4 > MSDA_STATIC_WORKSPACE_BYTES)");
    void* ws = nullptr;
    s = static_workspace_address(reinterpret_cast<cudaStream_t>(stream), &ws);
    if (s != MSDA_OK) return s;
    // msda_backward clears the workspace (or widens grad_value into it when
    // accumulating) before its kernel, so nothing carries over between calls.
    return msda_backward(dt, MSDA_ACCUM_FP32, flags, B, S, M, D, L, K, Q, value, spatial_shapes, level_start_index,
                         sampling_locations, attention_weights, grad_out, grad_value, grad_sampling_locations,
                         grad_attention_weights, ws, MSDA_STATIC_WORKSPACE_BYTES, stream);
}
