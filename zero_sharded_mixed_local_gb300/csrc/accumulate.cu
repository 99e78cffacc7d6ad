// Gradient accumulation into the fp32 grad arena.
//
// "ZeRO-1 风格的 Distributed Optimizer", section 6.7 (micro-batch gradients
// are summed into .grad before the data-parallel reduction and the step) and
// the Nanotron config's accumulate_grad_in_fp32.  grad = bf16(micro[0]) when
// overwriting, then grad += bf16(micro[k]) in k order; bf16 -> fp32 is exact,
// each addition rounds once.
//
// Memory-bound: per element 2 bytes read per micro-batch plus 4 written (and 4
// read when not overwriting).  Flat over the arena, one 8-element vector per
// thread and a grid that covers the whole arena: one 16-byte load per
// micro-batch, two 16-byte fp32 accesses.
//
// Where the gradient arena is 32-byte aligned (every torch allocation is),
// the passes that write the gradient without reading it first store each
// thread's eight fp32 values with one 256-bit access instead of two 128-bit
// ones, so each warp instruction writes whole 32-byte sectors.  The write-
// heavy one-micro-batch pass (2 bytes read, 4 written) measured 0.885 ->
// 0.865 ms on the 1.0B-element shard; passes that read the gradient too
// measured no difference.  Each thread keeps its elements, so the sums and
// the norm's summation order, and therefore every bit, are the same either
// way.
//
// accumulate_norm_kernel fuses the last micro-batch's pass with the gradient
// norm (and, when asked, with the division of the reduced gradient by the
// world size that FSDP2 runs as its own kernel, "TorchTitan 生产级预训练方案",
// appendix B.1: one IEEE division per element after the last addition): each
// block owns one 16384-element norm tile, writes the accumulated gradient and
// adds its squares into float pairs with exactly the mapping and
// order of sumsq_tiles_kernel, so the norm record is bit-identical to
// zero1_grad_norm's while the gradient is never read back (4 bytes per element
// saved).
#include "elementwise.cuh"
#include "launch.cuh"
#include "pair_sum.cuh"
#include "store8.cuh"

namespace zero1 {
namespace {

constexpr int kAccThreads = 256;

template <bool kWideStore>
__global__ void __launch_bounds__(kAccThreads)
    accumulate_kernel(const __grid_constant__ AccumulateParams P, int64_t first_vec) {
    pdl_enter();
    const int64_t i = first_vec + static_cast<int64_t>(blockIdx.x) * kAccThreads + threadIdx.x;
    if (i >= P.n_vec) return;
    float4* g4 = reinterpret_cast<float4*>(P.grad) + 2 * i;
    float acc[8];
    int k = 0;
    if (P.overwrite_first) {
        widen8(reinterpret_cast<const uint4*>(P.micro[0])[i], acc);
        k = 1;
    } else {
        const float4 a = g4[0], b = g4[1];
        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
        acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    }
    for (; k < P.n_micro; ++k) {
        float f[8];
        widen8(reinterpret_cast<const uint4*>(P.micro[k])[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], f[j]);
    }
    if (kWideStore) {
        store8_f32(P.grad + 8 * i, make_float4(acc[0], acc[1], acc[2], acc[3]), make_float4(acc[4], acc[5], acc[6], acc[7]));
    } else {
        g4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        g4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// One vector's accumulation, in the same operation order as accumulate_kernel.
__device__ __forceinline__ void accumulate_vec(const AccumulateParams& P, int64_t i, float (&acc)[8]) {
    int k = 0;
    if (P.overwrite_first) {
        widen8(reinterpret_cast<const uint4*>(P.micro[0])[i], acc);
        k = 1;
    } else {
        const float4* g4 = reinterpret_cast<const float4*>(P.grad) + 2 * i;
        const float4 a = g4[0], b = g4[1];
        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
        acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    }
    for (; k < P.n_micro; ++k) {
        float f[8];
        widen8(reinterpret_cast<const uint4*>(P.micro[k])[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], f[j]);
    }
}

// kOneOverwrite: the common call (one micro-batch, first of the step).  A
// thread's eight 16-byte loads go out in two batches of four, and registers
// are capped at 48 so that 5 blocks stay resident per SM without spilling.
// Measured on the 1.0B-element shard: 0.906 ms, against 0.945 ms for all
// eight loads at once (same cap), 1.010 ms uncapped (58 registers, 4
// blocks) and 1.01 ms at 6 blocks.  With the 256-bit gradient stores
// (kWideStore) 4 blocks per SM measured best: 0.865 ms, against 0.870 ms at
// 5.  The general instantiation (adds into grad, or several micro-batches)
// is not capped.  All add the same squares in the same order.
template <bool kOneOverwrite, bool kWideStore>
__global__ void __launch_bounds__(kTileThreads, kOneOverwrite ? (kWideStore ? 4 : 5) : 1)
    accumulate_norm_kernel(const __grid_constant__ AccumulateParams P, float2* __restrict__ partials, int64_t first_tile) {
    pdl_enter();
    __shared__ float2 s_warp[kTileThreads / 32];
    const int64_t tile = first_tile + blockIdx.x;
    const int64_t v0 = tile * kVecsPerTile;
    const int64_t nv = P.n_vec - v0 < kVecsPerTile ? P.n_vec - v0 : kVecsPerTile;
    SquarePairs sq;
    if (kOneOverwrite) {
        // two batches of four 16-byte loads: fewer live registers than eight at once
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint4 raw[kVecsPerThread / 2];
#pragma unroll
            for (int q = 0; q < kVecsPerThread / 2; ++q) {
                const int v = threadIdx.x + (half * (kVecsPerThread / 2) + q) * kTileThreads;
                raw[q] = v < nv ? reinterpret_cast<const uint4*>(P.micro[0])[v0 + v] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < kVecsPerThread / 2; ++q) {
                const int v = threadIdx.x + (half * (kVecsPerThread / 2) + q) * kTileThreads;
                float acc[8];
                widen8(raw[q], acc);
                if (P.divide) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = __fdiv_rn(acc[j], P.divisor);
                }
                const float4 a = make_float4(acc[0], acc[1], acc[2], acc[3]);
                const float4 b = make_float4(acc[4], acc[5], acc[6], acc[7]);
                if (v < nv) {
                    if (kWideStore) {
                        store8_f32(P.grad + 8 * (v0 + v), a, b);
                    } else {
                        float4* g4 = reinterpret_cast<float4*>(P.grad) + 2 * (v0 + v);
                        g4[0] = a;
                        g4[1] = b;
                    }
                }
                sq.add_vec(a, b);
            }
        }
    } else {
#pragma unroll 2
        for (int r = 0; r < kVecsPerThread; ++r) {
            const int v = threadIdx.x + r * kTileThreads;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (v < nv) {
                accumulate_vec(P, v0 + v, acc);
                if (P.divide) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = __fdiv_rn(acc[j], P.divisor);
                }
                float4* g4 = reinterpret_cast<float4*>(P.grad) + 2 * (v0 + v);
                g4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                g4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
            sq.add_vec(make_float4(acc[0], acc[1], acc[2], acc[3]), make_float4(acc[4], acc[5], acc[6], acc[7]));
        }
    }
    sq.fold();
    block_pair_sum<kTileThreads>(sq.s[0], sq.c[0], s_warp);
    if (threadIdx.x == 0) partials[tile] = make_float2(sq.s[0], sq.c[0]);
}

// One micro-batch added to the gradient already there (the last of K > 1
// calls, the general kernel's most common use): all eight of a thread's
// vectors, gradient and micro-batch, are loaded before the additions (110
// registers, 2 blocks per SM).  Measured on the 1.0B-element shard with the
// final reduction: 1.411 ms (7.12 TB/s at 10 bytes per element), against
// 1.434 ms through the general kernel; bit-identical gradient and partials.
// The division by the world size is a template parameter, as in the K-way
// kernel below.
template <bool kDivide>
__global__ void __launch_bounds__(kTileThreads, 2)
    accumulate_norm_add1_kernel(const __grid_constant__ AccumulateParams P, float2* __restrict__ partials,
                                int64_t first_tile) {
    pdl_enter();
    __shared__ float2 s_warp[kTileThreads / 32];
    const uint4* __restrict__ micro = reinterpret_cast<const uint4*>(P.micro[0]);
    float4* __restrict__ grad = reinterpret_cast<float4*>(P.grad);
    const int64_t tile = first_tile + blockIdx.x;
    const int64_t v0 = tile * kVecsPerTile;
    const int64_t nv = P.n_vec - v0 < kVecsPerTile ? P.n_vec - v0 : kVecsPerTile;
    uint4 raw[kVecsPerThread];
    float4 ga[kVecsPerThread], gb[kVecsPerThread];
#pragma unroll
    for (int r = 0; r < kVecsPerThread; ++r) {
        const int v = threadIdx.x + r * kTileThreads;
        if (v < nv) {
            raw[r] = micro[v0 + v];
            ga[r] = grad[2 * (v0 + v)];
            gb[r] = grad[2 * (v0 + v) + 1];
        } else {
            raw[r] = make_uint4(0u, 0u, 0u, 0u);
            ga[r] = gb[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    SquarePairs sq;
#pragma unroll
    for (int r = 0; r < kVecsPerThread; ++r) {
        const int v = threadIdx.x + r * kTileThreads;
        float f[8];
        widen8(raw[r], f);
        float4 a = make_float4(__fadd_rn(ga[r].x, f[0]), __fadd_rn(ga[r].y, f[1]), __fadd_rn(ga[r].z, f[2]),
                               __fadd_rn(ga[r].w, f[3]));
        float4 b = make_float4(__fadd_rn(gb[r].x, f[4]), __fadd_rn(gb[r].y, f[5]), __fadd_rn(gb[r].z, f[6]),
                               __fadd_rn(gb[r].w, f[7]));
        if (kDivide) {
            const float d = P.divisor;
            a = make_float4(__fdiv_rn(a.x, d), __fdiv_rn(a.y, d), __fdiv_rn(a.z, d), __fdiv_rn(a.w, d));
            b = make_float4(__fdiv_rn(b.x, d), __fdiv_rn(b.y, d), __fdiv_rn(b.z, d), __fdiv_rn(b.w, d));
        }
        if (v < nv) {
            grad[2 * (v0 + v)] = a;
            grad[2 * (v0 + v) + 1] = b;
        }
        sq.add_vec(a, b);  // padding and the tail add zeros, as in the kernels above
    }
    sq.fold();
    block_pair_sum<kTileThreads>(sq.s[0], sq.c[0], s_warp);
    if (threadIdx.x == 0) partials[tile] = make_float2(sq.s[0], sq.c[0]);
}

// K micro-batches already resident (2 <= K <= 8), grad overwritten: one pass
// reads the K bf16 arenas and writes the fp32 sum, grad = ((m0 + m1) + m2) +
// ..., the additions of K separate calls in the same order, and adds the
// squares with the tile mapping above.  All K 16-byte loads of a vector go out
// before its additions (K is a template parameter, so nothing waits on a
// runtime-bounded loop); two vectors at a time for K <= 4.  The minimum of one
// block per SM in the launch bounds matters: without it ptxas held the kernel
// to 40 registers, too few to keep K loads in flight (K = 8 on the 213.9M-
// element shard: 0.70 ms at 40 registers, 0.594 ms = 7.2 TB/s at 76).  The
// division by the world size is a template parameter, so the plain sum
// carries no division code.
template <int K, bool kDivide>
__global__ void __launch_bounds__(kTileThreads, 1)
    accumulate_norm_kway_kernel(const __grid_constant__ AccumulateParams P, float2* __restrict__ partials,
                                int64_t first_tile) {
    pdl_enter();
    constexpr int kUnroll = K <= 4 ? 2 : 1;
    __shared__ float2 s_warp[kTileThreads / 32];
    const int64_t tile = first_tile + blockIdx.x;
    const int64_t v0 = tile * kVecsPerTile;
    const int64_t nv = P.n_vec - v0 < kVecsPerTile ? P.n_vec - v0 : kVecsPerTile;
    SquarePairs sq;
#pragma unroll kUnroll
    for (int r = 0; r < kVecsPerThread; ++r) {
        const int v = threadIdx.x + r * kTileThreads;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (v < nv) {
            uint4 raw[K];
#pragma unroll
            for (int k = 0; k < K; ++k) raw[k] = reinterpret_cast<const uint4*>(P.micro[k])[v0 + v];
            widen8(raw[0], acc);
#pragma unroll
            for (int k = 1; k < K; ++k) {
                float f[8];
                widen8(raw[k], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], f[j]);
            }
            if (kDivide) {
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = __fdiv_rn(acc[j], P.divisor);
            }
            float4* g4 = reinterpret_cast<float4*>(P.grad) + 2 * (v0 + v);
            g4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            g4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        sq.add_vec(make_float4(acc[0], acc[1], acc[2], acc[3]), make_float4(acc[4], acc[5], acc[6], acc[7]));
    }
    sq.fold();
    block_pair_sum<kTileThreads>(sq.s[0], sq.c[0], s_warp);
    if (threadIdx.x == 0) partials[tile] = make_float2(sq.s[0], sq.c[0]);
}

template <int K>
cudaError_t launch_kway(const AccumulateParams& p, unsigned nb, float2* pairs, int64_t first, cudaStream_t stream) {
    if (p.divide) return launch(accumulate_norm_kway_kernel<K, true>, nb, kTileThreads, stream, p, pairs, first);
    return launch(accumulate_norm_kway_kernel<K, false>, nb, kTileThreads, stream, p, pairs, first);
}

}  // namespace

cudaError_t launch_accumulate_norm(const AccumulateParams& p, double* partials, int64_t n_tiles, double extra_sumsq,
                                   zero1_norm_out* out, cudaStream_t stream) {
    float2* pairs = reinterpret_cast<float2*>(partials);
    for (int64_t first = 0; first < n_tiles; first += 0x7fffffff) {
        const int64_t nb = n_tiles - first < 0x7fffffff ? n_tiles - first : 0x7fffffff;
        const unsigned g = static_cast<unsigned>(nb);
        const int kway = p.overwrite_first ? p.n_micro : (p.n_micro == 1 ? -1 : 0);
        cudaError_t e;
        switch (kway) {
            case -1:
                e = p.divide ? launch(accumulate_norm_add1_kernel<true>, g, kTileThreads, stream, p, pairs, first)
                             : launch(accumulate_norm_add1_kernel<false>, g, kTileThreads, stream, p, pairs, first);
                break;
            case 1:
                e = wide_store_aligned(p.grad)
                        ? launch(accumulate_norm_kernel<true, true>, g, kTileThreads, stream, p, pairs, first)
                        : launch(accumulate_norm_kernel<true, false>, g, kTileThreads, stream, p, pairs, first);
                break;
            case 2: e = launch_kway<2>(p, g, pairs, first, stream); break;
            case 3: e = launch_kway<3>(p, g, pairs, first, stream); break;
            case 4: e = launch_kway<4>(p, g, pairs, first, stream); break;
            case 5: e = launch_kway<5>(p, g, pairs, first, stream); break;
            case 6: e = launch_kway<6>(p, g, pairs, first, stream); break;
            case 7: e = launch_kway<7>(p, g, pairs, first, stream); break;
            case 8: e = launch_kway<8>(p, g, pairs, first, stream); break;
            default: e = launch(accumulate_norm_kernel<false, false>, g, kTileThreads, stream, p, pairs, first);
        }
        if (e != cudaSuccess) return e;
    }
    return launch_norm_final(pairs, n_tiles, extra_sumsq, out, stream);
}

cudaError_t launch_accumulate(const AccumulateParams& p, cudaStream_t stream) {
    for (int64_t first = 0; first < p.n_vec; first += kMaxGridVectors(kAccThreads)) {
        const int64_t n = p.n_vec - first < kMaxGridVectors(kAccThreads) ? p.n_vec - first : kMaxGridVectors(kAccThreads);
        const unsigned grid = static_cast<unsigned>((n + kAccThreads - 1) / kAccThreads);
        const cudaError_t e = wide_store_aligned(p.grad)
                                  ? launch(accumulate_kernel<true>, grid, kAccThreads, stream, p, first)
                                  : launch(accumulate_kernel<false>, grid, kAccThreads, stream, p, first);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace zero1
