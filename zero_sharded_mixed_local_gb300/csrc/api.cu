// C entry points of the compute calls: argument checks, derivation of the
// fp32 step scalars, and the kernel launches.  Nothing here allocates device
// memory or synchronises, except zero1_read_norm.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "zero1_internal.h"

namespace {

// One NVTX range per compute call, so profiler timelines show each entry
// point around its kernels (no cost unless a tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

thread_local char g_cuda_error[256] = "";

int cuda_fail(cudaError_t e) {
    std::snprintf(g_cuda_error, sizeof g_cuda_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return ZERO1_ECUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A gradient divisor is used as fp32: it must be finite and positive after
// that rounding too (1e300 would become inf, 1e-300 zero).
bool divisor_ok(double d) {
    const float f = static_cast<float>(d);
    return std::isfinite(d) && d > 0.0 && std::isfinite(f) && f > 0.0f;
}

// Can kernels on the current device read `p`?  Device and managed memory,
// and pinned or registered host memory (unified addressing), always; plain
// pageable host memory only where the device reads host page tables (ATS on
// Grace-based systems such as GB300).  Returns ZERO1_OK, ZERO1_EINVAL, or
// ZERO1_ECUDA if the query itself fails.
int check_readable(const void* p) {
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) return cuda_fail(e);
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeHost)
        return ZERO1_OK;
    int dev = 0, pageable = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    return pageable ? ZERO1_OK : ZERO1_EINVAL;
}

}  // namespace

namespace zero1 {

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

cudaError_t after_launch(cudaError_t launched) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const cudaError_t last = cudaGetLastError();  // also clears it
    return launched != cudaSuccess ? launched : last;
}

}  // namespace zero1

extern "C" uint64_t zero1_launch_count(void) { return zero1::g_launches.load(std::memory_order_relaxed); }

extern "C" int zero1_accumulate(const zero1_plan* plan, float* grad, const uint16_t* const* micro_bf16,
                                int32_t n_micro, int32_t overwrite_first, void* stream) {
    NvtxRange range("zero1_accumulate");
    if (plan == nullptr || micro_bf16 == nullptr) return ZERO1_EINVAL;
    if (n_micro < 1 || n_micro > ZERO1_MAX_MICRO) return ZERO1_EINVAL;
    if (plan->arena_numel == 0) return ZERO1_OK;  // nothing to do; empty buffers may be NULL
    if (grad == nullptr) return ZERO1_EINVAL;
    zero1::AccumulateParams p{};
    p.grad = grad;
    for (int k = 0; k < n_micro; ++k) {
        if (micro_bf16[k] == nullptr) return ZERO1_EINVAL;
        if (!aligned16(micro_bf16[k])) return ZERO1_EALIGN;
        p.micro[k] = micro_bf16[k];
    }
    if (!aligned16(grad)) return ZERO1_EALIGN;
    for (int k = 0; k < n_micro; ++k) {
        const int rc = check_readable(micro_bf16[k]);
        if (rc != ZERO1_OK) return rc;
    }
    p.n_micro = n_micro;
    p.overwrite_first = overwrite_first ? 1 : 0;
    p.n_vec = plan->arena_numel / ZERO1_ARENA_ALIGN;
    const cudaError_t e = zero1::launch_accumulate(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

extern "C" int zero1_accumulate_norm(const zero1_plan* plan, float* grad, const uint16_t* const* micro_bf16,
                                     int32_t n_micro, int32_t overwrite_first, double grad_divisor,
                                     double extra_sumsq, void* workspace, size_t workspace_bytes,
                                     zero1_norm_out* d_out, void* stream) {
    NvtxRange range("zero1_accumulate_norm");
    if (plan == nullptr || micro_bf16 == nullptr || d_out == nullptr) return ZERO1_EINVAL;
    if (n_micro < 1 || n_micro > ZERO1_MAX_MICRO) return ZERO1_EINVAL;
    if (!divisor_ok(grad_divisor)) return ZERO1_EINVAL;
    if (std::isnan(extra_sumsq) || extra_sumsq < 0.0) return ZERO1_EINVAL;
    if (!aligned16(d_out)) return ZERO1_EALIGN;
    const int64_t n_tiles = zero1::norm_tiles(plan->arena_numel);
    zero1::AccumulateParams p{};
    if (n_tiles > 0) {
        if (grad == nullptr || workspace == nullptr) return ZERO1_EINVAL;
        if (workspace_bytes < static_cast<size_t>(n_tiles) * sizeof(double)) return ZERO1_EINVAL;
        for (int k = 0; k < n_micro; ++k) {
            if (micro_bf16[k] == nullptr) return ZERO1_EINVAL;
            if (!aligned16(micro_bf16[k])) return ZERO1_EALIGN;
            p.micro[k] = micro_bf16[k];
        }
        if (!aligned16(grad) || !aligned16(workspace)) return ZERO1_EALIGN;
        for (int k = 0; k < n_micro; ++k) {
            const int rc = check_readable(micro_bf16[k]);
            if (rc != ZERO1_OK) return rc;
        }
    }
    p.grad = grad;
    p.n_micro = n_micro;
    p.overwrite_first = overwrite_first ? 1 : 0;
    p.n_vec = plan->arena_numel / ZERO1_ARENA_ALIGN;
    p.divisor = static_cast<float>(grad_divisor);
    p.divide = grad_divisor != 1.0 ? 1 : 0;
    const cudaError_t e = zero1::launch_accumulate_norm(p, static_cast<double*>(workspace), n_tiles, extra_sumsq,
                                                        d_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

extern "C" int zero1_grad_norm(const zero1_plan* plan, const float* grad, double extra_sumsq, void* workspace,
                               size_t workspace_bytes, zero1_norm_out* d_out, void* stream) {
    NvtxRange range("zero1_grad_norm");
    if (plan == nullptr || d_out == nullptr) return ZERO1_EINVAL;
    const int64_t n_tiles = zero1::norm_tiles(plan->arena_numel);
    if (n_tiles > 0) {
        if (grad == nullptr || workspace == nullptr) return ZERO1_EINVAL;
        if (workspace_bytes < static_cast<size_t>(n_tiles) * sizeof(double)) return ZERO1_EINVAL;
        if (!aligned16(grad) || !aligned16(workspace)) return ZERO1_EALIGN;
    }
    if (!aligned16(d_out)) return ZERO1_EALIGN;
    if (std::isnan(extra_sumsq) || extra_sumsq < 0.0) return ZERO1_EINVAL;
    const cudaError_t e = zero1::launch_grad_norm(grad, plan->arena_numel, static_cast<double*>(workspace), n_tiles,
                                                  extra_sumsq, d_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

namespace zero1 {

int fill_step_scalars(const zero1_plan* plan, const zero1_hparams* hp, int64_t step_t, zero1_step_scalars* sc) {
    if (plan == nullptr || hp == nullptr || sc == nullptr || step_t < 1) return ZERO1_EINVAL;
    const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
    if (!std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(wd) || !std::isfinite(hp->clip_grad))
        return ZERO1_EINVAL;
    if (!(b1 >= 0.0 && b1 < 1.0) || !(b2 >= 0.0 && b2 < 1.0) || eps < 0.0) return ZERO1_EINVAL;
    // Step scalars in double, each rounded once to fp32.
    const double bc1 = 1.0 - std::pow(b1, static_cast<double>(step_t));
    const double bc2 = 1.0 - std::pow(b2, static_cast<double>(step_t));
    if (!(bc1 > 0.0) || !(bc2 > 0.0)) return ZERO1_EINVAL;
    for (int g = 0; g < ZERO1_MAX_GROUPS; ++g) {
        const double lr_g = lr * plan->lr_scale[g];
        const double wd_g = wd * plan->wd_scale[g];
        sc->stepsize[g] = static_cast<float>(lr_g / bc1);
        sc->dfac[g] = static_cast<float>(1.0 - lr_g * wd_g);
    }
    sc->b1 = static_cast<float>(b1);
    sc->b2 = static_cast<float>(b2);
    sc->omb1 = static_cast<float>(1.0 - b1);
    sc->omb2 = static_cast<float>(1.0 - b2);
    sc->eps = static_cast<float>(eps);
    sc->sqrtbc2 = static_cast<float>(std::sqrt(bc2));
    sc->clip = hp->clip_grad;
    return ZERO1_OK;
}

}  // namespace zero1

namespace {

// The step's buffer checks (shared by zero1_step, zero1_step_dev and zero1_local_step).
int check_step_buffers(const zero1_plan* plan, const float* master, const float* exp_avg, const float* exp_avg_sq,
                       const float* grad, const uint16_t* weight_bf16, const zero1_norm_out* d_norm) {
    if (plan->arena_numel == 0) return ZERO1_OK;  // nothing to do; empty buffers may be NULL
    if (master == nullptr || exp_avg == nullptr || exp_avg_sq == nullptr || grad == nullptr) return ZERO1_EINVAL;
    if (!aligned16(master) || !aligned16(exp_avg) || !aligned16(exp_avg_sq) || !aligned16(grad)) return ZERO1_EALIGN;
    if (weight_bf16 != nullptr && !aligned16(weight_bf16)) return ZERO1_EALIGN;
    if (d_norm != nullptr && !aligned16(d_norm)) return ZERO1_EALIGN;
    return ZERO1_OK;
}

// Checks shared by zero1_step and zero1_step_dev, and the launch.
int launch_checked_step(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq, const float* grad,
                        uint16_t* weight_bf16, const zero1_step_scalars* sc, const zero1_step_scalars* d_scalars,
                        const zero1_norm_out* d_norm, void* stream) {
    const int rc = check_step_buffers(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, d_norm);
    if (rc != ZERO1_OK || plan->arena_numel == 0) return rc;
    zero1::StepParams p{};
    p.master = master;
    p.m = exp_avg;
    p.v = exp_avg_sq;
    p.grad = grad;
    p.w = weight_bf16;
    p.norm = d_norm;
    p.n_vec = plan->arena_numel / ZERO1_ARENA_ALIGN;
    for (int g = 0; g < ZERO1_MAX_GROUPS; ++g) p.group_begin_vec[g] = plan->group_begin[g] / ZERO1_ARENA_ALIGN;
    if (sc != nullptr) p.sc = *sc;
    p.dev_scalars = d_scalars;
    const cudaError_t e = zero1::launch_step(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

}  // namespace

extern "C" int zero1_step(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq,
                          const float* grad, uint16_t* weight_bf16, const zero1_hparams* hp, int64_t step_t,
                          const zero1_norm_out* d_norm, void* stream) {
    NvtxRange range("zero1_step");
    zero1_step_scalars sc{};
    const int rc = zero1::fill_step_scalars(plan, hp, step_t, &sc);
    if (rc != ZERO1_OK) return rc;
    return launch_checked_step(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, &sc, nullptr, d_norm, stream);
}

extern "C" int zero1_micro_norm(const zero1_plan* plan, const uint16_t* micro_bf16, double grad_divisor,
                                double extra_sumsq, void* workspace, size_t workspace_bytes, zero1_norm_out* d_out,
                                void* stream) {
    NvtxRange range("zero1_micro_norm");
    if (plan == nullptr || d_out == nullptr) return ZERO1_EINVAL;
    if (!divisor_ok(grad_divisor)) return ZERO1_EINVAL;
    if (std::isnan(extra_sumsq) || extra_sumsq < 0.0) return ZERO1_EINVAL;
    if (!aligned16(d_out)) return ZERO1_EALIGN;
    const int64_t n_tiles = zero1::norm_tiles(plan->arena_numel);
    if (n_tiles > 0) {
        if (micro_bf16 == nullptr || workspace == nullptr) return ZERO1_EINVAL;
        if (workspace_bytes < static_cast<size_t>(n_tiles) * sizeof(double)) return ZERO1_EINVAL;
        if (!aligned16(micro_bf16) || !aligned16(workspace)) return ZERO1_EALIGN;
        const int rc = check_readable(micro_bf16);
        if (rc != ZERO1_OK) return rc;
    }
    const cudaError_t e = zero1::launch_micro_norm(micro_bf16, plan->arena_numel, static_cast<float>(grad_divisor),
                                                   grad_divisor != 1.0, static_cast<double*>(workspace), n_tiles,
                                                   extra_sumsq, d_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

namespace {

// zero1_step_accumulate's checks (all before any launch) and launch.
int step_accumulate(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq, float* grad,
                    const uint16_t* micro_bf16, double grad_divisor, uint16_t* weight_bf16,
                    const zero1_step_scalars* sc, const zero1_norm_out* d_norm, void* stream) {
    if (!divisor_ok(grad_divisor)) return ZERO1_EINVAL;
    int rc = check_step_buffers(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, d_norm);
    if (rc != ZERO1_OK || plan->arena_numel == 0) return rc;
    if (micro_bf16 == nullptr) return ZERO1_EINVAL;
    if (!aligned16(micro_bf16)) return ZERO1_EALIGN;
    rc = check_readable(micro_bf16);
    if (rc != ZERO1_OK) return rc;
    zero1::StepParams p{};
    p.master = master;
    p.m = exp_avg;
    p.v = exp_avg_sq;
    p.grad = nullptr;
    p.w = weight_bf16;
    p.micro = micro_bf16;
    p.grad_out = grad;
    p.divisor = static_cast<float>(grad_divisor);
    p.divide = grad_divisor != 1.0 ? 1 : 0;
    p.norm = d_norm;
    p.n_vec = plan->arena_numel / ZERO1_ARENA_ALIGN;
    for (int g = 0; g < ZERO1_MAX_GROUPS; ++g) p.group_begin_vec[g] = plan->group_begin[g] / ZERO1_ARENA_ALIGN;
    p.sc = *sc;
    p.dev_scalars = nullptr;
    const cudaError_t e = zero1::launch_step(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

}  // namespace

extern "C" int zero1_step_accumulate(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq,
                                     float* grad, const uint16_t* micro_bf16, double grad_divisor,
                                     uint16_t* weight_bf16, const zero1_hparams* hp, int64_t step_t,
                                     const zero1_norm_out* d_norm, void* stream) {
    NvtxRange range("zero1_step_accumulate");
    zero1_step_scalars sc{};
    const int rc = zero1::fill_step_scalars(plan, hp, step_t, &sc);
    if (rc != ZERO1_OK) return rc;
    return step_accumulate(plan, master, exp_avg, exp_avg_sq, grad, micro_bf16, grad_divisor, weight_bf16, &sc,
                           d_norm, stream);
}

extern "C" int zero1_local_step(const zero1_plan* plan, float* grad, const uint16_t* const* micro_bf16,
                                int32_t n_micro, double grad_divisor, double extra_sumsq, void* workspace,
                                size_t workspace_bytes, zero1_norm_out* d_norm, float* master, float* exp_avg,
                                float* exp_avg_sq, uint16_t* weight_bf16, const zero1_hparams* hp, int64_t step_t,
                                void* stream) {
    NvtxRange range("zero1_local_step");
    if (plan == nullptr || d_norm == nullptr) return ZERO1_EINVAL;
    // Every argument of both passes is checked before the first launch, so a rejected call
    // leaves every buffer as it was.
    zero1_step_scalars sc{};
    int rc = zero1::fill_step_scalars(plan, hp, step_t, &sc);
    if (rc != ZERO1_OK) return rc;
    rc = check_step_buffers(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, d_norm);
    if (rc != ZERO1_OK) return rc;
    if (n_micro == 1 && micro_bf16 != nullptr && plan->arena_numel > 0) {
        // one micro-batch: the norm from the micro-batch alone, then the step that writes the gradient
        if (micro_bf16[0] == nullptr) return ZERO1_EINVAL;
        if (!aligned16(micro_bf16[0])) return ZERO1_EALIGN;
        if (!divisor_ok(grad_divisor)) return ZERO1_EINVAL;
        rc = check_readable(micro_bf16[0]);
        if (rc != ZERO1_OK) return rc;
        rc = zero1_micro_norm(plan, micro_bf16[0], grad_divisor, extra_sumsq, workspace, workspace_bytes, d_norm,
                              stream);
        if (rc != ZERO1_OK) return rc;
        return step_accumulate(plan, master, exp_avg, exp_avg_sq, grad, micro_bf16[0], grad_divisor, weight_bf16, &sc,
                               d_norm, stream);
    }
    rc = zero1_accumulate_norm(plan, grad, micro_bf16, n_micro, 1, grad_divisor, extra_sumsq, workspace,
                               workspace_bytes, d_norm, stream);
    if (rc != ZERO1_OK) return rc;
    return launch_checked_step(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, &sc, nullptr, d_norm, stream);
}

extern "C" int zero1_step_scalars_fill(const zero1_plan* plan, const zero1_hparams* hp, int64_t step_t,
                                       zero1_step_scalars* out) {
    return zero1::fill_step_scalars(plan, hp, step_t, out);
}

extern "C" int zero1_step_dev(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq,
                              const float* grad, uint16_t* weight_bf16, const zero1_step_scalars* d_scalars,
                              const zero1_norm_out* d_norm, void* stream) {
    NvtxRange range("zero1_step_dev");
    if (plan == nullptr || d_scalars == nullptr) return ZERO1_EINVAL;
    if (!aligned16(d_scalars)) return ZERO1_EALIGN;
    return launch_checked_step(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, nullptr, d_scalars, d_norm,
                               stream);
}

extern "C" int zero1_layout_table_upload(const zero1_plan* plan, void* d_table, size_t table_bytes, void* stream) {
    if (plan == nullptr) return ZERO1_EINVAL;
    const size_t need = plan->layout_chunks.size() * sizeof(LayoutChunk);
    if (need == 0) return ZERO1_OK;
    if (d_table == nullptr || table_bytes < need) return ZERO1_EINVAL;
    if (!aligned16(d_table)) return ZERO1_EALIGN;
    // A pageable source: the call returns once the bytes are staged, so the
    // plan may be destroyed right after it.
    const cudaError_t e = cudaMemcpyAsync(d_table, plan->layout_chunks.data(), need, cudaMemcpyHostToDevice,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

namespace {

int layout_copy(const zero1_plan* plan, const void* d_table, const void* src, void* dst, int32_t elem_bytes,
                bool to_arena, void* stream) {
    if (plan == nullptr) return ZERO1_EINVAL;
    if (elem_bytes != 2 && elem_bytes != 4) return ZERO1_EINVAL;
    const int64_t n_chunks = static_cast<int64_t>(plan->layout_chunks.size());
    if (n_chunks == 0) return ZERO1_OK;
    if (d_table == nullptr || src == nullptr || dst == nullptr) return ZERO1_EINVAL;
    const void* arena = to_arena ? dst : src;
    const void* full = to_arena ? src : dst;
    if (!aligned16(d_table) || !aligned16(arena)) return ZERO1_EALIGN;
    if (reinterpret_cast<uintptr_t>(full) % static_cast<uintptr_t>(elem_bytes)) return ZERO1_EALIGN;
    const cudaError_t e = zero1::launch_layout_copy(static_cast<const LayoutChunk*>(d_table), n_chunks, src, dst,
                                                    elem_bytes, to_arena, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

}  // namespace

extern "C" int zero1_shard_gather(const zero1_plan* plan, const void* d_table, const void* full, void* arena,
                                  int32_t elem_bytes, void* stream) {
    NvtxRange range("zero1_shard_gather");
    return layout_copy(plan, d_table, full, arena, elem_bytes, true, stream);
}

extern "C" int zero1_shard_scatter(const zero1_plan* plan, const void* d_table, const void* arena, void* full,
                                   int32_t elem_bytes, void* stream) {
    NvtxRange range("zero1_shard_scatter");
    return layout_copy(plan, d_table, arena, full, elem_bytes, false, stream);
}

extern "C" int zero1_read_norm(const zero1_norm_out* d_norm, void* stream, zero1_norm_out* host_out) {
    if (d_norm == nullptr || host_out == nullptr) return ZERO1_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_out, d_norm, sizeof(zero1_norm_out), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

extern "C" const char* zero1_strerror(int code) {
    switch (code) {
        case ZERO1_OK: return "ok";
        case ZERO1_EINVAL: return "invalid argument";
        case ZERO1_EALIGN: return "buffer not 16-byte aligned";
        case ZERO1_ECUDA: return "CUDA error";
        case ZERO1_ENONFINITE: return "gradient norm is not finite; step skipped";
        case ZERO1_ENOMEM: return "out of host memory";
        case ZERO1_ETOOBIG: return "arena larger than the static norm scratch allows (ZERO1_STATIC_NORM_MAX_NUMEL)";
        default: return "unknown status";
    }
}

extern "C" const char* zero1_last_cuda_error(void) { return g_cuda_error; }

/* ---- tensor lists --------------------------------------------------------- */

extern "C" int zero1_list_table_upload(const zero1_plan* plan, void* d_table, size_t table_bytes, void* stream) {
    if (plan == nullptr) return ZERO1_EINVAL;
    const size_t need = plan->list_chunks.size() * sizeof(ListChunk);
    if (need == 0) return ZERO1_OK;
    if (d_table == nullptr || table_bytes < need) return ZERO1_EINVAL;
    if (!aligned16(d_table)) return ZERO1_EALIGN;
    const cudaError_t e = cudaMemcpyAsync(d_table, plan->list_chunks.data(), need, cudaMemcpyHostToDevice,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

extern "C" int zero1_list_ptrs_upload(const zero1_plan* plan, const void* const* host_ptrs, int32_t n_lists,
                                      int32_t elem_bytes, void* d_lists, size_t lists_bytes, void* stream) {
    if (plan == nullptr || n_lists < 1 || n_lists > ZERO1_MAX_MICRO) return ZERO1_EINVAL;
    if (elem_bytes != 2 && elem_bytes != 4) return ZERO1_EINVAL;
    const size_t count = static_cast<size_t>(n_lists) * static_cast<size_t>(plan->n_tensors);
    if (count == 0) return ZERO1_OK;
    if (host_ptrs == nullptr || d_lists == nullptr) return ZERO1_EINVAL;
    if (lists_bytes < count * sizeof(void*)) return ZERO1_EINVAL;
    if (!aligned16(d_lists)) return ZERO1_EALIGN;
    for (int32_t k = 0; k < n_lists; ++k) {
        for (int32_t i = 0; i < plan->n_tensors; ++i) {
            const void* p = host_ptrs[static_cast<size_t>(k) * plan->n_tensors + i];
            if (plan->shard_numel[i] == 0) continue;  // never dereferenced
            if (p == nullptr) return ZERO1_EINVAL;
            if (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(elem_bytes)) return ZERO1_EALIGN;
        }
    }
    // Copied from library-owned pageable memory: the call returns once the
    // bytes are staged, whatever kind of memory the caller's array is.
    std::vector<const void*> staged;
    try {
        staged.assign(host_ptrs, host_ptrs + count);
    } catch (const std::bad_alloc&) {
        return ZERO1_ENOMEM;
    }
    const cudaError_t e = cudaMemcpyAsync(d_lists, staged.data(), count * sizeof(void*), cudaMemcpyHostToDevice,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

namespace {

// Checks shared by the tensor-list gradient passes.
int list_grad_checked(const zero1_plan* plan, const void* d_table, float* const* d_grad,
                      const uint16_t* const* d_micro, int32_t n_micro, int32_t overwrite_first, double grad_divisor,
                      zero1::ListGradMode mode, double extra_sumsq, void* workspace, size_t workspace_bytes,
                      zero1_norm_out* d_out, void* stream) {
    if (plan == nullptr) return ZERO1_EINVAL;
    const bool reads_micro = mode != zero1::ListGradMode::kNorm;
    const bool norm = mode != zero1::ListGradMode::kAccumulate;
    if (reads_micro && (n_micro < 1 || n_micro > ZERO1_MAX_MICRO)) return ZERO1_EINVAL;
    if (norm) {
        if (d_out == nullptr) return ZERO1_EINVAL;
        if (!aligned16(d_out)) return ZERO1_EALIGN;
        if (std::isnan(extra_sumsq) || extra_sumsq < 0.0) return ZERO1_EINVAL;
    }
    if (!divisor_ok(grad_divisor)) return ZERO1_EINVAL;
    const int64_t n_chunks = static_cast<int64_t>(plan->list_chunks.size());
    const bool uses_grad = mode != zero1::ListGradMode::kMicroNorm;
    if (n_chunks > 0) {
        if (d_table == nullptr || (uses_grad && d_grad == nullptr) || (reads_micro && d_micro == nullptr))
            return ZERO1_EINVAL;
        if (!aligned16(d_table) || (uses_grad && !aligned16(d_grad)) || (reads_micro && !aligned16(d_micro)))
            return ZERO1_EALIGN;
        if (norm) {
            if (workspace == nullptr) return ZERO1_EINVAL;
            if (workspace_bytes < static_cast<size_t>(n_chunks) * sizeof(double)) return ZERO1_EINVAL;
            if (!aligned16(workspace)) return ZERO1_EALIGN;
        }
    } else if (!norm) {
        return ZERO1_OK;  // nothing to do
    }
    zero1::ListParams p{};
    p.table = static_cast<const ListChunk*>(d_table);
    p.grad = d_grad;
    p.micro = d_micro;
    p.n_tensors = plan->n_tensors;
    p.n_micro = reads_micro ? n_micro : 0;
    p.overwrite_first = overwrite_first ? 1 : 0;
    p.divisor = static_cast<float>(grad_divisor);
    p.divide = grad_divisor != 1.0 ? 1 : 0;
    const cudaError_t e = zero1::launch_list_grad(p, mode, n_chunks, static_cast<double*>(workspace), extra_sumsq,
                                                  d_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

}  // namespace

extern "C" int zero1_list_accumulate(const zero1_plan* plan, const void* d_table, float* const* d_grad,
                                     const uint16_t* const* d_micro, int32_t n_micro, int32_t overwrite_first,
                                     void* stream) {
    NvtxRange range("zero1_list_accumulate");
    return list_grad_checked(plan, d_table, d_grad, d_micro, n_micro, overwrite_first, 1.0,
                             zero1::ListGradMode::kAccumulate, 0.0, nullptr, 0, nullptr, stream);
}

extern "C" int zero1_list_accumulate_norm(const zero1_plan* plan, const void* d_table, float* const* d_grad,
                                          const uint16_t* const* d_micro, int32_t n_micro, int32_t overwrite_first,
                                          double grad_divisor, double extra_sumsq, void* workspace,
                                          size_t workspace_bytes, zero1_norm_out* d_out, void* stream) {
    NvtxRange range("zero1_list_accumulate_norm");
    return list_grad_checked(plan, d_table, d_grad, d_micro, n_micro, overwrite_first, grad_divisor,
                             zero1::ListGradMode::kAccumulateNorm, extra_sumsq, workspace, workspace_bytes, d_out,
                             stream);
}

extern "C" int zero1_list_micro_norm(const zero1_plan* plan, const void* d_table, const uint16_t* const* d_micro,
                                     double grad_divisor, double extra_sumsq, void* workspace, size_t workspace_bytes,
                                     zero1_norm_out* d_out, void* stream) {
    NvtxRange range("zero1_list_micro_norm");
    return list_grad_checked(plan, d_table, nullptr, d_micro, 1, 1, grad_divisor, zero1::ListGradMode::kMicroNorm,
                             extra_sumsq, workspace, workspace_bytes, d_out, stream);
}

extern "C" int zero1_list_grad_norm(const zero1_plan* plan, const void* d_table, const float* const* d_grad,
                                    double extra_sumsq, void* workspace, size_t workspace_bytes,
                                    zero1_norm_out* d_out, void* stream) {
    NvtxRange range("zero1_list_grad_norm");
    // The norm pass only reads through the gradient list.
    return list_grad_checked(plan, d_table, const_cast<float* const*>(d_grad), nullptr, 0, 0, 1.0,
                             zero1::ListGradMode::kNorm, extra_sumsq, workspace, workspace_bytes, d_out, stream);
}

namespace {

// Checks shared by zero1_list_step, zero1_list_step_dev and zero1_list_step_accumulate (d_micro:
// the one-micro-batch form, which writes the gradient list), and the launch.
int list_step_checked(const zero1_plan* plan, const void* d_table, float* const* d_master, float* const* d_exp_avg,
                      float* const* d_exp_avg_sq, const float* const* d_grad, uint16_t* const* d_weight_bf16,
                      const zero1_step_scalars* sc, const zero1_step_scalars* d_scalars,
                      const zero1_norm_out* d_norm, void* stream, const uint16_t* const* d_micro = nullptr,
                      double grad_divisor = 1.0) {
    if (!divisor_ok(grad_divisor)) return ZERO1_EINVAL;
    const int64_t n_chunks = static_cast<int64_t>(plan->list_chunks.size());
    if (n_chunks == 0) return ZERO1_OK;  // nothing to do; empty lists may be NULL
    if (d_table == nullptr || d_master == nullptr || d_exp_avg == nullptr || d_exp_avg_sq == nullptr ||
        d_grad == nullptr)
        return ZERO1_EINVAL;
    if (d_micro != nullptr && !aligned16(d_micro)) return ZERO1_EALIGN;
    if (!aligned16(d_table) || !aligned16(d_master) || !aligned16(d_exp_avg) || !aligned16(d_exp_avg_sq) ||
        !aligned16(d_grad))
        return ZERO1_EALIGN;
    if (d_weight_bf16 != nullptr && !aligned16(d_weight_bf16)) return ZERO1_EALIGN;
    if (d_norm != nullptr && !aligned16(d_norm)) return ZERO1_EALIGN;
    zero1::ListParams p{};
    p.table = static_cast<const ListChunk*>(d_table);
    p.grad = const_cast<float* const*>(d_grad);
    p.master = d_master;
    p.m = d_exp_avg;
    p.v = d_exp_avg_sq;
    p.w = d_weight_bf16;
    p.norm = d_norm;
    p.n_tensors = plan->n_tensors;
    if (sc != nullptr) p.sc = *sc;
    p.dev_scalars = d_scalars;
    if (d_micro != nullptr) {
        p.micro = d_micro;
        p.n_micro = 1;
        p.micro_step = 1;
        p.divisor = static_cast<float>(grad_divisor);
        p.divide = grad_divisor != 1.0 ? 1 : 0;
    }
    const cudaError_t e = zero1::launch_list_step(p, n_chunks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZERO1_OK : cuda_fail(e);
}

}  // namespace

extern "C" int zero1_list_step(const zero1_plan* plan, const void* d_table, float* const* d_master,
                               float* const* d_exp_avg, float* const* d_exp_avg_sq, const float* const* d_grad,
                               uint16_t* const* d_weight_bf16, const zero1_hparams* hp, int64_t step_t,
                               const zero1_norm_out* d_norm, void* stream) {
    NvtxRange range("zero1_list_step");
    zero1_step_scalars sc{};
    const int rc = zero1::fill_step_scalars(plan, hp, step_t, &sc);
    if (rc != ZERO1_OK) return rc;
    return list_step_checked(plan, d_table, d_master, d_exp_avg, d_exp_avg_sq, d_grad, d_weight_bf16, &sc, nullptr,
                             d_norm, stream);
}

extern "C" int zero1_list_step_accumulate(const zero1_plan* plan, const void* d_table, float* const* d_master,
                                          float* const* d_exp_avg, float* const* d_exp_avg_sq, float* const* d_grad,
                                          const uint16_t* const* d_micro, double grad_divisor,
                                          uint16_t* const* d_weight_bf16, const zero1_hparams* hp, int64_t step_t,
                                          const zero1_norm_out* d_norm, void* stream) {
    NvtxRange range("zero1_list_step_accumulate");
    zero1_step_scalars sc{};
    const int rc = zero1::fill_step_scalars(plan, hp, step_t, &sc);
    if (rc != ZERO1_OK) return rc;
    if (d_micro == nullptr && !plan->list_chunks.empty()) return ZERO1_EINVAL;
    return list_step_checked(plan, d_table, d_master, d_exp_avg, d_exp_avg_sq, d_grad, d_weight_bf16, &sc, nullptr,
                             d_norm, stream, d_micro, grad_divisor);
}

extern "C" int zero1_list_step_dev(const zero1_plan* plan, const void* d_table, float* const* d_master,
                                   float* const* d_exp_avg, float* const* d_exp_avg_sq, const float* const* d_grad,
                                   uint16_t* const* d_weight_bf16, const zero1_step_scalars* d_scalars,
                                   const zero1_norm_out* d_norm, void* stream) {
    NvtxRange range("zero1_list_step_dev");
    if (plan == nullptr || d_scalars == nullptr) return ZERO1_EINVAL;
    if (!aligned16(d_scalars)) return ZERO1_EALIGN;
    return list_step_checked(plan, d_table, d_master, d_exp_avg, d_exp_avg_sq, d_grad, d_weight_bf16, nullptr,
                             d_scalars, d_norm, stream);
}
