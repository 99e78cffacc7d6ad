// zero1_grad_norm_static: the gradient-norm call without a caller-provided
// workspace.  The per-tile partial sums go to a fixed array that lives in the
// library's own device memory, so the call needs no allocation at all.
//
// Who needs it: callers that cannot hand the library a scratch buffer or
// cannot afford to get one -- a plain C host program that drives the C ABI
// without any device allocator of its own, a process where a framework's
// caching allocator has already reserved almost all of the GPU's memory so a
// separate cudaMalloc would fail, or a training loop that must not call
// cudaMalloc/cudaFree mid-step because those can synchronise the whole device.
//
// Costs and rules:
//   - The array holds ZERO1_STATIC_NORM_MAX_TILES 8-byte partials (2 MiB).  Every GPU
//     that loads the library keeps it allocated until the process exits.
//   - It covers arenas of up to ZERO1_STATIC_NORM_MAX_NUMEL elements; larger
//     plans are rejected with ZERO1_ETOOBIG before anything is launched.
//   - All calls on a device share the one array.  Nothing in it has to start
//     at zero: every partial the reduction reads is written earlier in the
//     same call, in stream order.  Calls whose kernels overlap on the GPU
//     (other streams, other host threads) race on it and must be serialised
//     by the caller.
//   - The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, which may load the module) with that device
//     current; make that first call before any stream capture.  The address
//     is cached per device together with the unique ID of the CUDA context
//     it was resolved in, and looked up again when the current context is
//     another one (after cudaDeviceReset, or when a driver-API caller has
//     made its own context current), so a stale address is never used.
#include <cuda.h>  // CUcontext and CUresult only: the two driver calls below are
                   // reached through the runtime, so the library does not link libcuda
#include <mutex>

#include "zero1_internal.h"

// Device-side home of the partial sums.  In host code this name is only a
// stand-in for the symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) double g_static_norm_partials[ZERO1_STATIC_NORM_MAX_TILES];

namespace {

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct Resolved {
    bool valid = false;
    unsigned long long context_id = 0;  // the context the address belongs to
    double* address = nullptr;
};

std::mutex g_lock;
Resolved g_resolved[kMaxDevices];
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The two driver entry points, looked up once through the runtime.
cudaError_t driver_entry_points() {
    if (g_ctx_get_current != nullptr && g_ctx_get_id != nullptr) return cudaSuccess;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || f == nullptr) return cudaErrorSymbolNotFound;
    void* g = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &g, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || g == nullptr) return cudaErrorSymbolNotFound;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(g);
    return cudaSuccess;
}

// Unique ID of the calling thread's current context; false when none is current.
bool current_context_id(unsigned long long* id) {
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array in the current device's current context, or
// nullptr with *err set.
double* static_partials(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> guard(g_lock);
    *err = driver_entry_points();
    if (*err != cudaSuccess) return nullptr;
    Resolved& r = g_resolved[dev];
    unsigned long long id = 0;
    if (r.valid && current_context_id(&id) && id == r.context_id) return r.address;
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_static_norm_partials);  // makes the device's context current if none is
    if (*err != cudaSuccess) return nullptr;
    if (!current_context_id(&id)) {
        *err = cudaErrorDeviceUninitialized;  // no context is current after the lookup
        return nullptr;
    }
    r.valid = true;
    r.context_id = id;
    r.address = static_cast<double*>(p);
    return r.address;
}

}  // namespace

extern "C" int zero1_grad_norm_static(const zero1_plan* plan, const float* grad, double extra_sumsq,
                                      zero1_norm_out* d_out, void* stream) {
    if (plan == nullptr || d_out == nullptr) return ZERO1_EINVAL;
    if (plan->arena_numel > ZERO1_STATIC_NORM_MAX_NUMEL) return ZERO1_ETOOBIG;
    const int64_t n_tiles = zero1::norm_tiles(plan->arena_numel);
    if (n_tiles > 0 && grad == nullptr) return ZERO1_EINVAL;
    if ((n_tiles > 0 && (reinterpret_cast<uintptr_t>(grad) & 15u)) || (reinterpret_cast<uintptr_t>(d_out) & 15u))
        return ZERO1_EALIGN;
    if (extra_sumsq != extra_sumsq || extra_sumsq < 0.0) return ZERO1_EINVAL;
    cudaError_t e = cudaSuccess;
    double* partials = static_partials(&e);
    if (partials == nullptr) return zero1::record_cuda_error(e);
    e = zero1::launch_grad_norm(grad, plan->arena_numel, partials, n_tiles, extra_sumsq, d_out,
                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : zero1::record_cuda_error(e);
}
