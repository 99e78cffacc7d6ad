// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "zero1.h"

// One contiguous run of a shard, as the model-layout <-> arena copies see it.
struct LayoutChunk {
    int64_t model_offset;  // first element in the model layout
    int64_t arena_offset;  // first element in the arena
    int32_t len;           // elements, 1 .. kLayoutChunk
    int32_t reserved;
};
static_assert(sizeof(LayoutChunk) == 24, "LayoutChunk is 24 bytes");

// One run of one tensor's shard, as the tensor-list kernels see it: block b
// of a launch handles run b.
struct ListChunk {
    int64_t offset;   // first element inside the tensor's shard buffer (a multiple of kNormTile)
    int32_t tensor;   // index into the pointer lists
    uint16_t len;     // elements, 1 .. kNormTile
    uint8_t group;    // the tensor's parameter group
    uint8_t reserved;
};
static_assert(sizeof(ListChunk) == 16, "ListChunk is 16 bytes");

struct zero1_plan {
    int32_t n_tensors = 0;
    int32_t dp_size = 1;
    int32_t dp_rank = 0;
    std::vector<int64_t> numel;
    std::vector<int64_t> shard_start;
    std::vector<int64_t> shard_numel;
    std::vector<int64_t> arena_offset;
    std::vector<uint8_t> group;
    int64_t total_numel = 0;
    int64_t local_numel = 0;
    int64_t arena_numel = 0;
    int64_t group_begin[ZERO1_MAX_GROUPS] = {};
    int64_t group_end[ZERO1_MAX_GROUPS] = {};
    double lr_scale[ZERO1_MAX_GROUPS] = {};
    double wd_scale[ZERO1_MAX_GROUPS] = {};
    std::vector<LayoutChunk> layout_chunks;  // the shard's runs, cut at kLayoutChunk elements
    std::vector<ListChunk> list_chunks;      // the same runs per tensor, cut at kNormTile elements
};

namespace zero1 {

// Elements per partial sum of the gradient norm; also fixes the reduction order.
constexpr int64_t kNormTile = 16384;
static_assert(ZERO1_STATIC_NORM_MAX_NUMEL == ZERO1_STATIC_NORM_MAX_TILES * kNormTile, "static norm limit");

inline int64_t norm_tiles(int64_t arena_numel) { return (arena_numel + kNormTile - 1) / kNormTile; }

// Most elements one layout-copy block moves.
constexpr int64_t kLayoutChunk = 16384;

// Launch parameters, passed by value (kernel parameter space).
struct AccumulateParams {
    float* grad;
    const uint16_t* micro[ZERO1_MAX_MICRO];
    int32_t n_micro;
    int32_t overwrite_first;
    int64_t n_vec;      // arena_numel / 8
    float divisor;      // accumulate_norm: divide the sum by this after the last addition
    int32_t divide;     // 0: plain sum (divisor unused)
};

struct StepParams {
    float* master;
    float* m;
    float* v;
    const float* grad;
    uint16_t* w;
    // The step that accumulates its one micro-batch (micro != null): the gradient is
    // float(micro) / divisor (divide: 0 keeps the plain values), written to grad_out.
    const uint16_t* micro;
    float* grad_out;
    float divisor;
    int32_t divide;
    const zero1_norm_out* norm;  // may be null: no clipping
    int64_t n_vec;               // arena_numel / 8
    int64_t group_begin_vec[ZERO1_MAX_GROUPS];  // first 8-element vector of each group
    zero1_step_scalars sc;                      // the step's scalars, at launch
    const zero1_step_scalars* dev_scalars;      // or read from device memory when the kernel runs
};
static_assert(sizeof(zero1_step_scalars) == 96, "zero1_step_scalars is 96 bytes");

// The fp32 step scalars for (plan, hp, t); ZERO1_OK or ZERO1_EINVAL.
int fill_step_scalars(const zero1_plan* plan, const zero1_hparams* hp, int64_t step_t, zero1_step_scalars* sc);

cudaError_t launch_accumulate(const AccumulateParams& p, cudaStream_t stream);
cudaError_t launch_grad_norm(const float* grad, int64_t n, double* partials, int64_t n_tiles,
                             double extra_sumsq, zero1_norm_out* out, cudaStream_t stream);
cudaError_t launch_accumulate_norm(const AccumulateParams& p, double* partials, int64_t n_tiles, double extra_sumsq,
                                   zero1_norm_out* out, cudaStream_t stream);
// The norm record of float(micro) / divisor (divide: 0 keeps the plain values) without writing it.
cudaError_t launch_micro_norm(const uint16_t* micro, int64_t n, float divisor, bool divide, double* partials,
                              int64_t n_tiles, double extra_sumsq, zero1_norm_out* out, cudaStream_t stream);
cudaError_t launch_step(const StepParams& p, cudaStream_t stream);

cudaError_t launch_layout_copy(const LayoutChunk* table, int64_t n_chunks, const void* src, void* dst,
                               int elem_bytes, bool to_arena, cudaStream_t stream);

// Tensor-list launches: every quantity is a device array of n_tensors
// pointers, one buffer per tensor shard.
struct ListParams {
    const ListChunk* table;
    float* const* grad;
    const uint16_t* const* micro;  // n_micro lists of n_tensors pointers, back to back
    float* const* master;
    float* const* m;
    float* const* v;
    uint16_t* const* w;            // may be null: no bf16 copy
    const zero1_norm_out* norm;    // may be null: no clipping
    int32_t n_tensors;
    int32_t n_micro;
    int32_t overwrite_first;
    int32_t divide;                // 0: plain sum (divisor unused)
    float divisor;
    int32_t micro_step;            // the step reads micro list 0 and writes grad (one micro-batch)
    zero1_step_scalars sc;                   // the step's scalars, at launch
    const zero1_step_scalars* dev_scalars;   // or read from device memory when the kernel runs
};

// What list_grad passes do with the gradient runs.
// kMicroNorm: the partials of one micro-batch's gradient without writing it (zero1_micro_norm).
enum class ListGradMode { kAccumulate, kAccumulateNorm, kNorm, kMicroNorm };

cudaError_t launch_list_grad(const ListParams& p, ListGradMode mode, int64_t n_chunks, double* partials,
                             double extra_sumsq, zero1_norm_out* out, cudaStream_t stream);
cudaError_t launch_list_step(const ListParams& p, int64_t n_chunks, cudaStream_t stream);

// Record a CUDA error for zero1_last_cuda_error() and return ZERO1_ECUDA.
int record_cuda_error(cudaError_t e);

// Called once for every kernel launch with the launch call's own result:
// counts it for zero1_launch_count() and returns the launch's error (that
// result, else cudaGetLastError()).
cudaError_t after_launch(cudaError_t launched = cudaSuccess);

// Work items one full-grid launch may cover (2^31 - 1 blocks of `threads`).
constexpr int64_t kMaxGridVectors(int threads) { return static_cast<int64_t>(0x7fffffff) * threads; }

}  // namespace zero1
