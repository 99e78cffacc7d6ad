// Sums of squares kept as unevaluated float pairs (hi + lo), shared by the
// norm kernels.  The rounding error of every square (an FMA) and of every
// addition of high parts (TwoSum) goes into the low part, so a pair stays
// within ~1e-13 relative of the exact sum while all arithmetic runs on the
// fp32 pipes (GB300's FP64 rate is a small fraction of its fp32 rate).
//
// Tile mapping (fixes the summation order, hence bit-identical results in
// every kernel that uses it): a tile is kNormTile = 16384 elements, i.e.
// 2048 vectors of 8; thread t of a 256-thread block owns vectors t, t + 256,
// ..., t + 7*256 and adds each vector's elements 0..7 into its four pairs in
// the order (0,1,2,3,4,5,6,7) -> pairs (0,1,2,3,0,1,2,3).
#pragma once

#include "zero1_internal.h"

namespace zero1 {

constexpr int kTileThreads = 256;
constexpr int kVecsPerTile = static_cast<int>(kNormTile / 8);          // 2048
constexpr int kVecsPerThread = kVecsPerTile / kTileThreads;            // 8
static_assert(kVecsPerThread * kTileThreads * 8 == kNormTile, "tile mapping");

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

// Two fp32 lanes in one 64-bit register, for Blackwell's packed fp32x2 instructions (sm_100 and
// later).  Each lane is rounded exactly as the scalar instruction rounds it (round to nearest, no
// flush to zero), so packed code gives the bits of the scalar code it replaces.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// add_square on two pairs at once (lanes: g0 into the low pair, g1 into the high one), with each
// lane's operations those of add_square in the same order.  The exact residual of each square
// stays a scalar FMA, whose negated addend costs nothing.
__device__ __forceinline__ void add_square2(uint64_t& s, uint64_t& c, float g0, float g1) {
    const uint64_t g = pack2(g0, g1);
    const uint64_t p = mul2(g, g);
    float p0, p1;
    unpack2(p, p0, p1);
    const uint64_t pe = pack2(__fmaf_rn(g0, g0, -p0), __fmaf_rn(g1, g1, -p1));  // g*g - p, exactly
    const uint64_t t = add2(s, p);  // two_sum(s, p)
    const uint64_t bp = sub2(t, s);
    const uint64_t e = add2(sub2(s, sub2(t, bp)), sub2(p, bp));
    s = t;
    c = add2(c, add2(e, pe));
}

// add_square2 for squares known to be exact, whose FMA residual is +0: c + (e + 0) is c + e bit for
// bit, because e is never -0 (a rounded sum is -0 only when both addends are, and neither the running
// sum s, which starts at +0, nor a square is ever -0).
__device__ __forceinline__ void add_exact_square2(uint64_t& s, uint64_t& c, float g0, float g1) {
    const uint64_t g = pack2(g0, g1);
    const uint64_t p = mul2(g, g);
    const uint64_t t = add2(s, p);  // two_sum(s, p)
    const uint64_t bp = sub2(t, s);
    const uint64_t e = add2(sub2(s, sub2(t, bp)), sub2(p, bp));
    s = t;
    c = add2(c, e);
}

// Exact squares of bf16 values.  A bf16 value with exponent field E (1..254) is M * 2^(E - 134) with
// M < 2^8, so its square M^2 * 2^(2E - 268) has at most 16 significant bits: it is an fp32 value
// exactly when 2E - 268 >= -149 (no bits below the smallest subnormal) and it is below 2^128, i.e.
// for E in 60..190.  In the magnitude bits of the bf16 (E << 7 | mantissa) that is the range below.
// Zero also squares exactly (+0).  Bf16 subnormals, tiny or huge values, infinities and NaN fall
// outside it and take add_square2.
constexpr uint32_t kExactSquareMin = 0x1E00u;  // E = 60, mantissa 0
constexpr uint32_t kExactSquareMax = 0x5F7Fu;  // E = 190, mantissa 0x7F

// 16-bit SIMD on the two halves of a word (sm_90 and later).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t add_u16x2(uint32_t a, uint32_t b) {  // per half, modulo 2^16
    uint32_t r;
    asm("add.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// True when every bf16 value in the vectors (eight per uint4) squares exactly in fp32: the largest
// magnitude is at most kExactSquareMax and the smallest non-zero one at least kExactSquareMin.  Each
// half's magnitude minus one (modulo 2^16) sends zeros to 0xFFFF, out of the way of the minimum.
template <int kN>
__device__ __forceinline__ bool bf16_squares_exact(const uint4 (&raw)[kN]) {
    uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll
    for (int r = 0; r < kN; ++r) {
        const uint32_t w[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t a = w[k] & 0x7FFF7FFFu;
            mx = max_u16x2(mx, a);
            mn = min_u16x2(mn, add_u16x2(a, 0xFFFFFFFFu));
        }
    }
    const uint32_t hi = max(mx & 0xFFFFu, mx >> 16), lo = min(mn & 0xFFFFu, mn >> 16);
    return hi <= kExactSquareMax && lo >= kExactSquareMin - 1u;
}

// A thread's four running pairs over its vectors.  While adding they are kept packed, pairs (0, 1)
// and (2, 3) in two registers each, so every instruction serves two pairs (measured 5% faster on the
// norm of a bf16 micro-batch, which was then bound by instruction issue rather than DRAM); fold()
// unpacks them into s[] and c[].
struct SquarePairs {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    uint64_t s01 = 0, s23 = 0, c01 = 0, c23 = 0;  // +0.0f in both lanes

    // The vector's elements 0..7 into pairs 0, 1, 2, 3, 0, 1, 2, 3.
    __device__ __forceinline__ void add_vec(const float4& a, const float4& b) {
        add_square2(s01, c01, a.x, a.y);
        add_square2(s23, c23, a.z, a.w);
        add_square2(s01, c01, b.x, b.y);
        add_square2(s23, c23, b.z, b.w);
    }

    // add_vec for a vector whose squares are exact (bf16_squares_exact): the same bits, two fp32
    // operations fewer per element.
    __device__ __forceinline__ void add_vec_exact(const float4& a, const float4& b) {
        add_exact_square2(s01, c01, a.x, a.y);
        add_exact_square2(s23, c23, a.z, a.w);
        add_exact_square2(s01, c01, b.x, b.y);
        add_exact_square2(s23, c23, b.z, b.w);
    }

    // Fold the four pairs into (s[0], c[0]) in a fixed order.
    __device__ __forceinline__ void fold() {
        unpack2(s01, s[0], s[1]);
        unpack2(c01, c[0], c[1]);
        unpack2(s23, s[2], s[3]);
        unpack2(c23, c[2], c[3]);
        add_pair(s[0], c[0], s[1], c[1]);
        add_pair(s[2], c[2], s[3], c[3]);
        add_pair(s[0], c[0], s[2], c[2]);
    }
};

__device__ __forceinline__ void warp_pair_sum(float& s, float& c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float t = __shfl_down_sync(0xffffffffu, s, off);
        const float d = __shfl_down_sync(0xffffffffu, c, off);
        add_pair(s, c, t, d);
    }
}

// Sum of the threads' pairs over the block in a fixed order; valid in thread 0.
template <int kThreads>
__device__ __forceinline__ void block_pair_sum(float& s, float& c, float2* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_pair_sum(s, c);
    if (lane == 0) s_warp[warp] = make_float2(s, c);
    __syncthreads();
    if (warp == 0) {
        const float2 x = lane < kThreads / 32 ? s_warp[lane] : make_float2(0.f, 0.f);
        s = x.x;
        c = x.y;
        warp_pair_sum(s, c);
    }
}

// Second kernel of every norm: adds the per-tile pairs in a fixed order,
// converts to double, adds the other ranks' share and writes the record.
cudaError_t launch_norm_final(const float2* partials, int64_t n_tiles, double extra_sumsq, zero1_norm_out* out,
                              cudaStream_t stream);

}  // namespace zero1
