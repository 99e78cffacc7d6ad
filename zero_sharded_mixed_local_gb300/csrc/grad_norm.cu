// Deterministic sum of squares of the fp32 grad arena, for the global L2 norm
// behind clip_grad ("ZeRO-1 风格的 Distributed Optimizer", section 6.6).
//
// The clip coefficient is rounded once to fp32 from the norm, so the sum must
// be accurate far beyond fp32: a plain fp32 running sum of these squares (of
// bf16-derived values, whose low bits are structured) drifts low by ~1e-7
// relative, enough to flip the coefficient's last bit.  Each thread therefore
// keeps an error-free fp32 pair: the exact rounding error of every square
// (an FMA) and of every addition (TwoSum) go into a compensation term, which
// keeps the thread's sum within a few double ulps of exact; all later sums
// are double.  ~10 fp32 operations per element, hidden under the loads.
//
// Two kernels:
//   sumsq_tiles   one partial per 16384-element tile.  Each of 256 threads
//                 sums the squares of its (at most 64) elements in four
//                 compensated fp32 pairs, then the block adds the 256 values
//                 in double through a fixed warp-shuffle tree.  A tile is
//                 always reduced by one block with the same thread mapping,
//                 so the partials do not depend on the grid size.
//   sumsq_final   one block adds the partials in double in a fixed order,
//                 adds the other ranks' share and writes {sumsq, norm, status}.
// Memory-bound: 4 bytes read per element.
#include "zero1_internal.h"

namespace zero1 {
namespace {

constexpr int kTileThreads = 256;
constexpr int kFinalThreads = 1024;
static_assert(kNormTile % (4 * kTileThreads) == 0, "tile must be a whole number of float4 rows");

// s + c += g*g without losing any rounding error of the square or the addition.
__device__ __forceinline__ void add_square(float& s, float& c, float g) {
    const float p = __fmul_rn(g, g);
    const float pe = __fmaf_rn(g, g, -p);  // g*g - p, exactly
    const float t = __fadd_rn(s, p);
    const float bp = __fsub_rn(t, s);
    const float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));  // s + p - t, exactly
    s = t;
    c = __fadd_rn(c, __fadd_rn(e, pe));
}

__device__ __forceinline__ double warp_sum(double x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xffffffffu, x, off);
    return x;
}

// Sum of `x` over the block in a fixed order; the result is valid in thread 0.
template <int kThreads>
__device__ __forceinline__ double block_sum(double x, double* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_sum(x);
    if (lane == 0) s_warp[warp] = x;
    __syncthreads();
    double t = 0.0;
    if (warp == 0) {
        t = lane < kThreads / 32 ? s_warp[lane] : 0.0;
        t = warp_sum(t);
    }
    __syncthreads();  // s_warp may be reused right after
    return t;
}

__global__ void __launch_bounds__(kTileThreads)
    sumsq_tiles_kernel(const float* __restrict__ grad, int64_t n, double* __restrict__ partials, int64_t n_tiles) {
    __shared__ double s_warp[kTileThreads / 32];
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t base = tile * kNormTile;
        const int64_t len = min(kNormTile, n - base);  // a multiple of 8
        const float4* g4 = reinterpret_cast<const float4*>(grad + base);
        const int n4 = static_cast<int>(len / 4);
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll 4
        for (int j = threadIdx.x; j < n4; j += kTileThreads) {
            const float4 g = g4[j];
            add_square(s0, c0, g.x);
            add_square(s1, c1, g.y);
            add_square(s2, c2, g.z);
            add_square(s3, c3, g.w);
        }
        const double mine = ((static_cast<double>(s0) + static_cast<double>(s1)) +
                             (static_cast<double>(s2) + static_cast<double>(s3))) +
                            ((static_cast<double>(c0) + static_cast<double>(c1)) +
                             (static_cast<double>(c2) + static_cast<double>(c3)));
        const double s = block_sum<kTileThreads>(mine, s_warp);
        if (threadIdx.x == 0) partials[tile] = s;
    }
}

__global__ void __launch_bounds__(kFinalThreads)
    sumsq_final_kernel(const double* __restrict__ partials, int64_t n_tiles, double extra, zero1_norm_out* out) {
    __shared__ double s_warp[kFinalThreads / 32];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < n_tiles; i += kFinalThreads) s += partials[i];
    s = block_sum<kFinalThreads>(s, s_warp);
    if (threadIdx.x == 0) {
        const double total = s + extra;
        out->sumsq = total;
        out->norm = sqrt(total);
        out->status = isfinite(total) ? ZERO1_OK : ZERO1_ENONFINITE;
        out->n_partials = static_cast<int32_t>(n_tiles);
    }
}

}  // namespace

cudaError_t launch_grad_norm(const float* grad, int64_t n, double* partials, int64_t n_tiles, double extra_sumsq,
                             zero1_norm_out* out, cudaStream_t stream) {
    if (n_tiles > 0) {
        const int64_t grid =
            streaming_grid(reinterpret_cast<const void*>(&sumsq_tiles_kernel), kTileThreads, n_tiles * kTileThreads);
        sumsq_tiles_kernel<<<static_cast<unsigned>(grid), kTileThreads, 0, stream>>>(grad, n, partials, n_tiles);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    sumsq_final_kernel<<<1, kFinalThreads, 0, stream>>>(partials, n_tiles, extra_sumsq, out);
    return cudaGetLastError();
}

}  // namespace zero1
