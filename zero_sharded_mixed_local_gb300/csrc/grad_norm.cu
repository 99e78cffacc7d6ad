// Deterministic sum of squares of the fp32 grad arena, for the global L2 norm
// behind clip_grad ("ZeRO-1 风格的 Distributed Optimizer", section 6.6).
//
// The clip coefficient is rounded once to fp32 from the norm, so the sum must
// be accurate far beyond fp32: a plain fp32 running sum of these squares (of
// bf16-derived values, whose low bits are structured) drifts low by ~1e-7
// relative, enough to flip the coefficient's last bit.  Every sum here is
// therefore an unevaluated pair of floats (hi + lo): the exact rounding error
// of each square (an FMA) and of each addition of high parts (TwoSum) goes
// into the low part.  That keeps the result within ~1e-13 relative of the
// exact sum while staying on the fp32 pipes; GB300's FP64 rate is a small
// fraction of its fp32 rate, and double arithmetic in the block reductions
// measured as the bound of this kernel.  Only the final total is double.
//
// Two kernels:
//   sumsq_tiles   one block per 16384-element tile (the grid covers the
//                 arena).  Each of 256 threads sums the squares of its 64
//                 elements in four float pairs, then the block adds the pairs
//                 through a fixed warp-shuffle tree and stores the tile's
//                 pair.  The reduction order is fixed by the tile, not by the
//                 launch.
//   sumsq_final   one block adds the tile pairs in a fixed order, converts to
//                 double, adds the other ranks' share and writes
//                 {sumsq, norm, status}.
// Memory-bound: 4 bytes read per element.
#include "zero1_internal.h"

namespace zero1 {
namespace {

constexpr int kTileThreads = 256;
constexpr int kFinalThreads = 1024;
static_assert(kNormTile % (4 * kTileThreads) == 0, "tile must be a whole number of float4 rows");

// s + e = a + b exactly (Knuth's TwoSum, six rounded operations).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (s, c) += g*g: the square's rounding error and the addition's go into c.
__device__ __forceinline__ void add_square(float& s, float& c, float g) {
    const float p = __fmul_rn(g, g);
    const float pe = __fmaf_rn(g, g, -p);  // g*g - p, exactly
    float t, e;
    two_sum(s, p, t, e);
    s = t;
    c = __fadd_rn(c, __fadd_rn(e, pe));
}

// (s, c) += (t, d)
__device__ __forceinline__ void add_pair(float& s, float& c, float t, float d) {
    float h, e;
    two_sum(s, t, h, e);
    s = h;
    c = __fadd_rn(c, __fadd_rn(d, e));
}

__device__ __forceinline__ void warp_sum(float& s, float& c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float t = __shfl_down_sync(0xffffffffu, s, off);
        const float d = __shfl_down_sync(0xffffffffu, c, off);
        add_pair(s, c, t, d);
    }
}

// Sum of the threads' pairs over the block in a fixed order; valid in thread 0.
template <int kThreads>
__device__ __forceinline__ void block_sum(float& s, float& c, float2* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_sum(s, c);
    if (lane == 0) s_warp[warp] = make_float2(s, c);
    __syncthreads();
    if (warp == 0) {
        const float2 x = lane < kThreads / 32 ? s_warp[lane] : make_float2(0.f, 0.f);
        s = x.x;
        c = x.y;
        warp_sum(s, c);
    }
}

__global__ void __launch_bounds__(kTileThreads)
    sumsq_tiles_kernel(const float* __restrict__ grad, int64_t n, float2* __restrict__ partials, int64_t first_tile) {
    __shared__ float2 s_warp[kTileThreads / 32];
    const int64_t tile = first_tile + blockIdx.x;
    const int64_t base = tile * kNormTile;
    const int64_t len = min(kNormTile, n - base);  // a positive multiple of 8
    const float4* g4 = reinterpret_cast<const float4*>(grad + base);
    const int n4 = static_cast<int>(len / 4);
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
    if (n4 == kNormTile / 4) {
        // full tile: all sixteen 16-byte loads in flight before any arithmetic
        float4 x[kNormTile / 4 / kTileThreads];
#pragma unroll
        for (int r = 0; r < kNormTile / 4 / kTileThreads; ++r) x[r] = g4[threadIdx.x + r * kTileThreads];
#pragma unroll
        for (int r = 0; r < kNormTile / 4 / kTileThreads; ++r) {
            add_square(s0, c0, x[r].x);
            add_square(s1, c1, x[r].y);
            add_square(s2, c2, x[r].z);
            add_square(s3, c3, x[r].w);
        }
    } else {
        for (int j = threadIdx.x; j < n4; j += kTileThreads) {
            const float4 x = g4[j];
            add_square(s0, c0, x.x);
            add_square(s1, c1, x.y);
            add_square(s2, c2, x.z);
            add_square(s3, c3, x.w);
        }
    }
    add_pair(s0, c0, s1, c1);
    add_pair(s2, c2, s3, c3);
    add_pair(s0, c0, s2, c2);
    block_sum<kTileThreads>(s0, c0, s_warp);
    if (threadIdx.x == 0) partials[tile] = make_float2(s0, c0);
}

__global__ void __launch_bounds__(kFinalThreads)
    sumsq_final_kernel(const float2* __restrict__ partials, int64_t n_tiles, double extra, zero1_norm_out* out) {
    __shared__ float2 s_warp[kFinalThreads / 32];
    float s = 0.f, c = 0.f;
    for (int64_t i = threadIdx.x; i < n_tiles; i += kFinalThreads) {
        const float2 x = partials[i];
        add_pair(s, c, x.x, x.y);
    }
    block_sum<kFinalThreads>(s, c, s_warp);
    if (threadIdx.x == 0) {
        const double total = (static_cast<double>(s) + static_cast<double>(c)) + extra;
        out->sumsq = total;
        out->norm = sqrt(total);
        out->status = isfinite(total) ? ZERO1_OK : ZERO1_ENONFINITE;
        out->n_partials = static_cast<int32_t>(n_tiles);
    }
}

}  // namespace

cudaError_t launch_grad_norm(const float* grad, int64_t n, double* partials, int64_t n_tiles, double extra_sumsq,
                             zero1_norm_out* out, cudaStream_t stream) {
    // The workspace holds one 8-byte (hi, lo) float pair per tile.
    float2* pairs = reinterpret_cast<float2*>(partials);
    for (int64_t first = 0; first < n_tiles; first += 0x7fffffff) {
        const int64_t nb = n_tiles - first < 0x7fffffff ? n_tiles - first : 0x7fffffff;
        sumsq_tiles_kernel<<<static_cast<unsigned>(nb), kTileThreads, 0, stream>>>(grad, n, pairs, first);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    sumsq_final_kernel<<<1, kFinalThreads, 0, stream>>>(pairs, n_tiles, extra_sumsq, out);
    return cudaGetLastError();
}

}  // namespace zero1
