// Per-element arithmetic shared by the arena kernels and the tensor-list
// kernels, so both paths round every operation identically.
//
// AdamW ("ZeRO-1 风格的 Distributed Optimizer", section 6.6: adam_w with
// beta1 0.9, beta2 0.95, eps 1e-8 and decoupled weight decay), decay on p
// first, bias-corrected moments, eps outside the square root, each fp32
// operation rounded once:
//     g = grad*coef;  p = p*dfac;  m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g)
//     d = sqrt(v)/sqrtbc2 + eps;  p = p - stepsize*(m/d)
// The rounding-explicit intrinsics (__fmul_rn, __fadd_rn, __fdiv_rn,
// __fsqrt_rn) are never contracted into FMAs, which keeps the order exact.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "zero1.h"

namespace zero1 {

struct StepConsts {
    float b1, b2, omb1, omb2, eps, sqrtbc2;
};

__device__ __forceinline__ void adamw_elem(float& p, float& m, float& v, float grad, float coef, float dfac,
                                           float stepsize, const StepConsts& c) {
    const float g = __fmul_rn(grad, coef);
    p = __fmul_rn(p, dfac);
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
    const float d = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), c.sqrtbc2), c.eps);
    p = __fsub_rn(p, __fmul_rn(stepsize, __fdiv_rn(m, d)));
}

// bf16 -> fp32 is exact: the 16 bits become the high half of the float.
__device__ __forceinline__ float bf16_bits_to_float(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Eight bf16 values (one 16-byte vector) widened to fp32, in memory order.
__device__ __forceinline__ void widen8(const uint4& b, float (&f)[8]) {
    f[0] = bf16_lo(b.x);
    f[1] = bf16_hi(b.x);
    f[2] = bf16_lo(b.y);
    f[3] = bf16_hi(b.y);
    f[4] = bf16_lo(b.z);
    f[5] = bf16_hi(b.z);
    f[6] = bf16_lo(b.w);
    f[7] = bf16_hi(b.w);
}

// fp32 -> bf16 rounded to nearest even, as raw bits.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t bf16_rne_bits(float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<const uint16_t*>(&h);
}

// The clip coefficient from a device-resident norm record ("ZeRO-1 风格的
// Distributed Optimizer", section 6.6, clip_grad): coef = clip/(norm + 1e-6)
// when that is below 1 and clip > 0, else 1, with norm = sqrt(sumsq) in
// double.  The norm is re-derived from sumsq so that a caller may sum that
// one field across ranks in place between the norm and the step.  skip = 1
// (write nothing) when the record's status is bad or sumsq is not finite.
__device__ __forceinline__ void clip_from_norm(const zero1_norm_out* norm, double clip, float& coef, int& skip) {
    coef = 1.0f;
    skip = 0;
    if (norm != nullptr) {
        const double sumsq = norm->sumsq;
        if (norm->status != ZERO1_OK || !isfinite(sumsq)) {
            skip = 1;
        } else if (clip > 0.0) {
            const double q = clip / (sqrt(sumsq) + 1e-6);
            if (q < 1.0) coef = static_cast<float>(q);
        }
    }
}

}  // namespace zero1
