// Copies between the model layout and a rank's arena: the data movement on
// either side of the local step ("ZeRO-1 风格的 Distributed Optimizer",
// section 6.3: after backward the gradients are reduce-scattered to the rank
// that owns each shard, and after the step the updated bf16 weights are
// all-gathered).
//
// Model layout: every parameter whole, concatenated in model order, no
// padding; tensor i occupies [model_offset_i, model_offset_i + numel_i).
// Rank r's shard of tensor i is the contiguous run [model_offset_i +
// shard_start_i, + shard_numel_i), which sits at arena[arena_offset_i ...].
// Every run is cut into chunks of at most 16384 elements; one block copies
// one chunk, so the grid covers the whole shard whatever the tensor sizes.
// The chunk table lives in a caller-provided device buffer (the library
// allocates no device memory).  Memory-bound: elem_bytes read + elem_bytes
// written per element.  Model-side offsets are arbitrary in general, so a
// chunk whose two ends are both 16-byte aligned (every chunk of a model whose
// tensor sizes are multiples of 8, i.e. every real one) moves 16-byte
// vectors plus an element-wise tail; any other chunk moves element by
// element (coalesced across the warp).  Element-wise bf16 copies measured
// 5.8 TB/s on a 1.0B-element shard: two bytes per instruction bound them.
#include "launch.cuh"
#include "zero1_internal.h"

namespace zero1 {
namespace {

constexpr int kLayoutThreads = 256;

template <typename T, bool kToArena>
__global__ void __launch_bounds__(kLayoutThreads)
    layout_copy_kernel(const LayoutChunk* __restrict__ table, const T* __restrict__ src, T* __restrict__ dst,
                       int64_t first_chunk) {
    pdl_enter();
    const LayoutChunk ch = table[first_chunk + blockIdx.x];
    const T* s = src + (kToArena ? ch.model_offset : ch.arena_offset);
    T* d = dst + (kToArena ? ch.arena_offset : ch.model_offset);
    int done = 0;
    if (((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d)) & 15u) == 0) {
        constexpr int kPerVec = 16 / sizeof(T);
        const int nv = ch.len / kPerVec;
        const uint4* s4 = reinterpret_cast<const uint4*>(s);
        uint4* d4 = reinterpret_cast<uint4*>(d);
        // eight vectors' loads before their stores: a full bf16 chunk is one round of load latency
        constexpr int kBatch = 8;
        for (int j0 = threadIdx.x; j0 < nv; j0 += kBatch * kLayoutThreads) {
            uint4 r[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int j = j0 + q * kLayoutThreads;
                if (j < nv) r[q] = s4[j];
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int j = j0 + q * kLayoutThreads;
                if (j < nv) d4[j] = r[q];
            }
        }
        done = nv * kPerVec;
    }
    for (int j = done + threadIdx.x; j < ch.len; j += kLayoutThreads) d[j] = s[j];
}

template <typename T, bool kToArena>
cudaError_t launch_typed(const LayoutChunk* table, int64_t n_chunks, const void* src, void* dst, cudaStream_t stream) {
    for (int64_t first = 0; first < n_chunks; first += 0x7fffffff) {
        const int64_t nb = n_chunks - first < 0x7fffffff ? n_chunks - first : 0x7fffffff;
        const cudaError_t e = launch(layout_copy_kernel<T, kToArena>, static_cast<unsigned>(nb), kLayoutThreads, stream,
                                     table, static_cast<const T*>(src), static_cast<T*>(dst), first);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_layout_copy(const LayoutChunk* table, int64_t n_chunks, const void* src, void* dst,
                               int elem_bytes, bool to_arena, cudaStream_t stream) {
    if (n_chunks == 0) return cudaSuccess;
    if (elem_bytes == 2)
        return to_arena ? launch_typed<uint16_t, true>(table, n_chunks, src, dst, stream)
                        : launch_typed<uint16_t, false>(table, n_chunks, src, dst, stream);
    return to_arena ? launch_typed<uint32_t, true>(table, n_chunks, src, dst, stream)
                    : launch_typed<uint32_t, false>(table, n_chunks, src, dst, stream);
}

}  // namespace zero1
