// Deterministic sum of squares of the fp32 grad arena, for the global L2 norm
// behind clip_grad ("ZeRO-1 风格的 Distributed Optimizer", section 6.6).
//
// The clip coefficient is rounded once to fp32 from the norm, so the sum must
// be accurate far beyond fp32: a plain fp32 running sum of these squares (of
// bf16-derived values, whose low bits are structured) drifts low by ~1e-7
// relative, enough to flip the coefficient's last bit.  Every sum here is
// therefore an unevaluated pair of floats (pair_sum.cuh), within ~1e-13
// relative of the exact sum, on the fp32 pipes; double arithmetic in the
// block reductions measured as this kernel's bound on GB300.  Only the final
// total is double.
//
// Two kernels:
//   sumsq_tiles   one block per 16384-element tile (the grid covers the
//                 arena).  Each of 256 threads loads its eight 8-element
//                 vectors (all sixteen 16-byte loads in flight), adds their
//                 squares into four float pairs, and the block adds the pairs
//                 through a fixed warp-shuffle tree.  The tile mapping is the
//                 one the fused accumulate-and-norm kernel uses, so both give
//                 identical partials.
//   sumsq_final   one block adds the tile pairs in a fixed order, converts to
//                 double, adds the other ranks' share and writes
//                 {sumsq, norm, status}.
// Memory-bound: 4 bytes read per element.
#include "elementwise.cuh"
#include "launch.cuh"
#include "pair_sum.cuh"

namespace zero1 {
namespace {

constexpr int kFinalThreads = 1024;

__global__ void __launch_bounds__(kTileThreads)
    sumsq_tiles_kernel(const float* __restrict__ grad, int64_t n_vec, float2* __restrict__ partials, int64_t first_tile) {
    pdl_enter();
    __shared__ float2 s_warp[kTileThreads / 32];
    const int64_t tile = first_tile + blockIdx.x;
    const int64_t v0 = tile * kVecsPerTile;
    const int64_t nv = n_vec - v0 < kVecsPerTile ? n_vec - v0 : kVecsPerTile;  // vectors in this tile
    const float4* g4 = reinterpret_cast<const float4*>(grad) + 2 * v0;
    float4 a[kVecsPerThread], b[kVecsPerThread];
#pragma unroll
    for (int r = 0; r < kVecsPerThread; ++r) {
        const int v = threadIdx.x + r * kTileThreads;
        if (v < nv) {
            a[r] = g4[2 * v];
            b[r] = g4[2 * v + 1];
        } else {
            a[r] = b[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    SquarePairs sq;
#pragma unroll
    for (int r = 0; r < kVecsPerThread; ++r) sq.add_vec(a[r], b[r]);
    sq.fold();
    block_pair_sum<kTileThreads>(sq.s[0], sq.c[0], s_warp);
    if (threadIdx.x == 0) partials[tile] = make_float2(sq.s[0], sq.c[0]);
}

// The partials of the gradient one micro-batch gives, float(micro) / divisor, without writing it:
// the same values squared in the same order as accumulate_norm_kernel's one-micro-batch overwrite
// pass (each thread's vectors r = 0..7 of the tile), so the partials are bit for bit that pass's.
// Reads 2 bytes per element.  Bound by the fp32 pipe rather than DRAM (the compensated squares cost
// about ten operations per element), so without a divisor a thread whose 64 values all square
// exactly (bf16_squares_exact: integer checks on the raw bits) adds them without the residual term.
// Five blocks per SM without the divisor (48 registers, a few spilled): 0.3256 ms on the 1.0B-element
// shard against 0.3309 at four.
template <bool kDivide>
__global__ void __launch_bounds__(kTileThreads, kDivide ? 4 : 5)
    micro_sumsq_tiles_kernel(const uint16_t* __restrict__ micro, int64_t n_vec, float divisor,
                             float2* __restrict__ partials, int64_t first_tile) {
    pdl_enter();
    __shared__ float2 s_warp[kTileThreads / 32];
    const int64_t tile = first_tile + blockIdx.x;
    const int64_t v0 = tile * kVecsPerTile;
    const int64_t nv = n_vec - v0 < kVecsPerTile ? n_vec - v0 : kVecsPerTile;
    const uint4* m4 = reinterpret_cast<const uint4*>(micro) + v0;
    uint4 raw[kVecsPerThread];
#pragma unroll
    for (int r = 0; r < kVecsPerThread; ++r) {
        const int v = threadIdx.x + r * kTileThreads;
        raw[r] = v < nv ? m4[v] : make_uint4(0u, 0u, 0u, 0u);
    }
    SquarePairs sq;
    if (!kDivide && bf16_squares_exact(raw)) {
        // every square exact: no residual to add (the same bits; 0.368 -> 0.330 ms on 1.0B elements)
#pragma unroll
        for (int r = 0; r < kVecsPerThread; ++r) {
            float f[8];
            widen8(raw[r], f);
            sq.add_vec_exact(make_float4(f[0], f[1], f[2], f[3]), make_float4(f[4], f[5], f[6], f[7]));
        }
    } else {
#pragma unroll
        for (int r = 0; r < kVecsPerThread; ++r) {
            float f[8];
            widen8(raw[r], f);
            if (kDivide) {
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = __fdiv_rn(f[j], divisor);
            }
            sq.add_vec(make_float4(f[0], f[1], f[2], f[3]), make_float4(f[4], f[5], f[6], f[7]));
        }
    }
    sq.fold();
    block_pair_sum<kTileThreads>(sq.s[0], sq.c[0], s_warp);
    if (threadIdx.x == 0) partials[tile] = make_float2(sq.s[0], sq.c[0]);
}

__global__ void __launch_bounds__(kFinalThreads)
    sumsq_final_kernel(const float2* __restrict__ partials, int64_t n_tiles, double extra, zero1_norm_out* out) {
    pdl_enter();
    __shared__ float2 s_warp[kFinalThreads / 32];
    // thread t adds tiles t, t + kFinalThreads, ... in that order; the loads of kAhead of them go out
    // before their additions (the same order, so the same bits, without a load's latency per tile)
    constexpr int kAhead = 8;
    float s = 0.f, c = 0.f;
    int64_t i = threadIdx.x;
    for (; i + (kAhead - 1) * static_cast<int64_t>(kFinalThreads) < n_tiles; i += kAhead * kFinalThreads) {
        float2 x[kAhead];
#pragma unroll
        for (int q = 0; q < kAhead; ++q) x[q] = partials[i + q * kFinalThreads];
#pragma unroll
        for (int q = 0; q < kAhead; ++q) add_pair(s, c, x[q].x, x[q].y);
    }
    for (; i < n_tiles; i += kFinalThreads) {
        const float2 x = partials[i];
        add_pair(s, c, x.x, x.y);
    }
    block_pair_sum<kFinalThreads>(s, c, s_warp);
    if (threadIdx.x == 0) {
        const double total = (static_cast<double>(s) + static_cast<double>(c)) + extra;
        out->sumsq = total;
        out->norm = sqrt(total);
        out->status = isfinite(total) ? ZERO1_OK : ZERO1_ENONFINITE;
        out->n_partials = static_cast<int32_t>(n_tiles);
    }
}

}  // namespace

cudaError_t launch_norm_final(const float2* partials, int64_t n_tiles, double extra_sumsq, zero1_norm_out* out,
                              cudaStream_t stream) {
    return launch(sumsq_final_kernel, 1, kFinalThreads, stream, partials, n_tiles, extra_sumsq, out);
}

cudaError_t launch_micro_norm(const uint16_t* micro, int64_t n, float divisor, bool divide, double* partials,
                              int64_t n_tiles, double extra_sumsq, zero1_norm_out* out, cudaStream_t stream) {
    float2* pairs = reinterpret_cast<float2*>(partials);
    for (int64_t first = 0; first < n_tiles; first += 0x7fffffff) {
        const int64_t nb = n_tiles - first < 0x7fffffff ? n_tiles - first : 0x7fffffff;
        const unsigned g = static_cast<unsigned>(nb);
        const cudaError_t e =
            divide ? launch(micro_sumsq_tiles_kernel<true>, g, kTileThreads, stream, micro, n / 8, divisor, pairs, first)
                   : launch(micro_sumsq_tiles_kernel<false>, g, kTileThreads, stream, micro, n / 8, divisor, pairs, first);
        if (e != cudaSuccess) return e;
    }
    return launch_norm_final(pairs, n_tiles, extra_sumsq, out, stream);
}

cudaError_t launch_grad_norm(const float* grad, int64_t n, double* partials, int64_t n_tiles, double extra_sumsq,
                             zero1_norm_out* out, cudaStream_t stream) {
    // The workspace holds one 8-byte (hi, lo) float pair per tile.
    float2* pairs = reinterpret_cast<float2*>(partials);
    for (int64_t first = 0; first < n_tiles; first += 0x7fffffff) {
        const int64_t nb = n_tiles - first < 0x7fffffff ? n_tiles - first : 0x7fffffff;
        const cudaError_t e = launch(sumsq_tiles_kernel, static_cast<unsigned>(nb), kTileThreads, stream, grad,
                                     n / 8, pairs, first);
        if (e != cudaSuccess) return e;
    }
    return launch_norm_final(pairs, n_tiles, extra_sumsq, out, stream);
}

}  // namespace zero1
