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
//     current; make that first call before any stream capture.
#include <mutex>

#include "zero1_internal.h"

// Device-side home of the partial sums.  In host code this name is only a
// stand-in for the symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) double g_static_norm_partials[ZERO1_STATIC_NORM_MAX_TILES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_lock;
double* g_partials_addr[kMaxDevices];  // per device, resolved once

// Device address of the array on the current device, or nullptr with *err set.
double* static_partials(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> guard(g_lock);
    if (g_partials_addr[dev] == nullptr) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_static_norm_partials);
        if (*err != cudaSuccess) return nullptr;
        g_partials_addr[dev] = static_cast<double*>(p);
    }
    return g_partials_addr[dev];
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
