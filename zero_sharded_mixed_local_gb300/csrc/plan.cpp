// Shard plan and arena layout (host only, no CUDA calls).
//
// "ZeRO-1 风格的 Distributed Optimizer", section 6.3: nanotron cuts every
// parameter on its own rather than flattening them into one blob; a tensor's
// total numel is split evenly over the dp_size ranks and each rank keeps fp32
// master, m and v for its own part.  The remainder goes to the lowest ranks,
// one element each (the page leaves this open).
#include <algorithm>
#include <cmath>
#include <new>

#include "zero1_internal.h"

namespace {

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" int zero1_plan_create(const int64_t* numels, const uint8_t* no_decay, int32_t n_tensors,
                                 int32_t dp_size, int32_t dp_rank, zero1_plan** out) {
    if (n_tensors > 0 && no_decay != nullptr) {
        for (int32_t i = 0; i < n_tensors; ++i) {
            if (no_decay[i] > 1) {
                if (out) *out = nullptr;
                return ZERO1_EINVAL;
            }
        }
    }
    return zero1_plan_create_grouped(numels, no_decay, n_tensors, nullptr, nullptr, dp_size, dp_rank, out);
}

extern "C" int zero1_plan_create_grouped(const int64_t* numels, const uint8_t* group, int32_t n_tensors,
                                         const double* lr_scale, const double* wd_scale, int32_t dp_size,
                                         int32_t dp_rank, zero1_plan** out) {
    if (out == nullptr) return ZERO1_EINVAL;
    *out = nullptr;
    if (n_tensors < 0 || dp_size < 1 || dp_rank < 0 || dp_rank >= dp_size) return ZERO1_EINVAL;
    if (n_tensors > 0 && (numels == nullptr || group == nullptr)) return ZERO1_EINVAL;
    int64_t total = 0;  // bounded so that no offset, padded or not, can overflow
    for (int32_t i = 0; i < n_tensors; ++i) {
        if (numels[i] < 0 || numels[i] > ZERO1_MAX_TOTAL_NUMEL - total || group[i] >= ZERO1_MAX_GROUPS)
            return ZERO1_EINVAL;
        total += numels[i];
    }
    for (int g = 0; g < ZERO1_MAX_GROUPS; ++g) {
        if (lr_scale && !(std::isfinite(lr_scale[g]) && lr_scale[g] >= 0.0)) return ZERO1_EINVAL;
        if (wd_scale && !(std::isfinite(wd_scale[g]) && wd_scale[g] >= 0.0)) return ZERO1_EINVAL;
    }

    zero1_plan* p = new (std::nothrow) zero1_plan;
    if (p == nullptr) return ZERO1_ENOMEM;
    try {
        const size_t n = static_cast<size_t>(n_tensors);
        p->numel.assign(numels, numels + n);
        p->group.assign(group, group + n);
        p->shard_start.resize(n);
        p->shard_numel.resize(n);
        p->arena_offset.resize(n);
    } catch (const std::bad_alloc&) {
        delete p;
        return ZERO1_ENOMEM;
    }
    p->n_tensors = n_tensors;
    p->dp_size = dp_size;
    p->dp_rank = dp_rank;
    for (int g = 0; g < ZERO1_MAX_GROUPS; ++g) {
        p->lr_scale[g] = lr_scale ? lr_scale[g] : 1.0;
        p->wd_scale[g] = wd_scale ? wd_scale[g] : (g == 1 ? 0.0 : 1.0);
    }

    const int64_t dp = dp_size, r = dp_rank;
    for (int32_t i = 0; i < n_tensors; ++i) {
        const int64_t n = p->numel[i];
        const int64_t base = n / dp;
        const int64_t rem = n % dp;
        p->shard_numel[i] = base + (r < rem ? 1 : 0);
        p->shard_start[i] = base * r + std::min(r, rem);
        p->total_numel += n;
        p->local_numel += p->shard_numel[i];
    }

    // Group-contiguous arena: group 0's shards, then group 1's, ..., each
    // group in model order.  One set of step scalars per contiguous range
    // lets the step kernel stream the arena flat, with no per-tensor table.
    int64_t off = 0;
    for (int g = 0; g < ZERO1_MAX_GROUPS; ++g) {
        p->group_begin[g] = off;
        for (int32_t i = 0; i < n_tensors; ++i) {
            if (p->group[i] != g) continue;
            p->arena_offset[i] = off;
            off += round_up(p->shard_numel[i], ZERO1_ARENA_ALIGN);
        }
        p->group_end[g] = off;
    }
    p->arena_numel = off;

    // Runs of the shard for the model-layout <-> arena copies.
    try {
        int64_t model_offset = 0;
        for (int32_t i = 0; i < n_tensors; ++i) {
            for (int64_t k = 0; k < p->shard_numel[i]; k += zero1::kLayoutChunk) {
                const int64_t len = std::min<int64_t>(zero1::kLayoutChunk, p->shard_numel[i] - k);
                p->layout_chunks.push_back(
                    {model_offset + p->shard_start[i] + k, p->arena_offset[i] + k, static_cast<int32_t>(len), 0});
            }
            model_offset += p->numel[i];
        }
        // Runs of each tensor's own shard buffer, for the tensor-list calls.
        for (int32_t i = 0; i < n_tensors; ++i) {
            for (int64_t k = 0; k < p->shard_numel[i]; k += zero1::kNormTile) {
                const int64_t len = std::min<int64_t>(zero1::kNormTile, p->shard_numel[i] - k);
                p->list_chunks.push_back({k, i, static_cast<uint16_t>(len), p->group[i], 0});
            }
        }
    } catch (const std::bad_alloc&) {
        delete p;
        return ZERO1_ENOMEM;
    }
    *out = p;
    return ZERO1_OK;
}

extern "C" void zero1_plan_destroy(zero1_plan* plan) { delete plan; }

extern "C" int32_t zero1_plan_num_tensors(const zero1_plan* plan) { return plan ? plan->n_tensors : -1; }
extern "C" int64_t zero1_plan_total_numel(const zero1_plan* plan) { return plan ? plan->total_numel : -1; }
extern "C" int64_t zero1_plan_local_numel(const zero1_plan* plan) { return plan ? plan->local_numel : -1; }
extern "C" int64_t zero1_plan_arena_numel(const zero1_plan* plan) { return plan ? plan->arena_numel : -1; }

extern "C" int zero1_plan_tensor(const zero1_plan* plan, int32_t i, int64_t* shard_start,
                                 int64_t* shard_numel, int64_t* arena_offset) {
    if (plan == nullptr || i < 0 || i >= plan->n_tensors) return ZERO1_EINVAL;
    if (shard_start) *shard_start = plan->shard_start[i];
    if (shard_numel) *shard_numel = plan->shard_numel[i];
    if (arena_offset) *arena_offset = plan->arena_offset[i];
    return ZERO1_OK;
}

extern "C" int zero1_plan_group_range(const zero1_plan* plan, int32_t g, int64_t* begin, int64_t* end) {
    if (plan == nullptr || g < 0 || g >= ZERO1_MAX_GROUPS) return ZERO1_EINVAL;
    if (begin) *begin = plan->group_begin[g];
    if (end) *end = plan->group_end[g];
    return ZERO1_OK;
}

extern "C" int zero1_plan_group_scales(const zero1_plan* plan, int32_t g, double* lr_scale, double* wd_scale) {
    if (plan == nullptr || g < 0 || g >= ZERO1_MAX_GROUPS) return ZERO1_EINVAL;
    if (lr_scale) *lr_scale = plan->lr_scale[g];
    if (wd_scale) *wd_scale = plan->wd_scale[g];
    return ZERO1_OK;
}

// ZeRO-1 keeps the whole bf16 weights and gradient buffer on each rank and
// shards the 12 bytes of fp32 optimizer state ("Distributed Training",
// section 0; "ZeRO-1 风格的 Distributed Optimizer", sections 6.1 and 6.3).
extern "C" int zero1_plan_bytes(const zero1_plan* plan, int32_t grad_bytes, int64_t out[4]) {
    if (plan == nullptr || out == nullptr || (grad_bytes != 2 && grad_bytes != 4)) return ZERO1_EINVAL;
    const int64_t weights = 2 * plan->total_numel;
    const int64_t grads = static_cast<int64_t>(grad_bytes) * plan->total_numel;
    const int64_t optim = 12 * plan->local_numel;
    out[0] = weights;
    out[1] = grads;
    out[2] = optim;
    out[3] = weights + grads + optim;
    return ZERO1_OK;
}

extern "C" size_t zero1_workspace_bytes(const zero1_plan* plan) {
    if (plan == nullptr) return 0;
    return static_cast<size_t>(zero1::norm_tiles(plan->arena_numel)) * sizeof(double);
}

extern "C" size_t zero1_layout_table_bytes(const zero1_plan* plan) {
    if (plan == nullptr) return 0;
    return plan->layout_chunks.size() * sizeof(LayoutChunk);
}

extern "C" size_t zero1_list_table_bytes(const zero1_plan* plan) {
    if (plan == nullptr) return 0;
    return plan->list_chunks.size() * sizeof(ListChunk);
}

extern "C" size_t zero1_list_workspace_bytes(const zero1_plan* plan) {
    if (plan == nullptr) return 0;
    return plan->list_chunks.size() * sizeof(double);
}
