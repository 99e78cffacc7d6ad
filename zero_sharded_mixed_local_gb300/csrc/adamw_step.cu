// Fused clip + AdamW + bf16 copy over the local shard arena (one pass).
//
// "ZeRO-1 风格的 Distributed Optimizer", sections 6.2-6.3: each rank steps only
// its own fp32 master / m / v shard and then ships the updated bf16 weights;
// section 6.6 gives adam_w with beta1 0.9, beta2 0.95, eps 1e-8 and decoupled
// weight decay.  Per element (decay on p first, bias-corrected moments, eps
// outside the square root; every fp32 operation rounded once):
//     g = grad*coef;  p = p*dfac;  m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g)
//     d = sqrt(v)/sqrtbc2 + eps;  p = p - stepsize*(m/d);  w = bf16_rne(p)
//
// Memory-bound: 16 bytes read (grad, master, m, v) and 14 written (master, m,
// v, bf16) per element, ~20 fp32 operations.  The arena is streamed flat with
// 16-byte vector accesses, 8 elements per thread per iteration, from a grid
// sized to fill every SM once (grid-stride).  The weight-decay group of a
// vector is found by comparing its index with the group boundaries (groups
// are contiguous in the arena), so no per-tensor table is read.  The
// rounding-explicit intrinsics (__fmul_rn, __fadd_rn, __fdiv_rn, __fsqrt_rn)
// are never contracted into FMAs, which keeps the operation order exact.
#include <cuda_bf16.h>

#include "zero1_internal.h"

namespace zero1 {
namespace {

constexpr int kStepThreads = 256;

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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <bool kWriteBf16>
__global__ void __launch_bounds__(kStepThreads) adamw_step_kernel(const __grid_constant__ StepParams P) {
    __shared__ float s_coef;
    __shared__ int s_skip;
    if (threadIdx.x == 0) {
        // Clip coefficient from the device-resident norm: no host round trip.
        float coef = 1.0f;
        int skip = 0;
        if (P.norm != nullptr) {
            // The norm is re-derived from sumsq, so a caller may sum that one
            // field across ranks in place between the norm and the step.
            const double sumsq = P.norm->sumsq;
            if (P.norm->status != ZERO1_OK || !isfinite(sumsq)) {
                skip = 1;
            } else if (P.clip > 0.0) {
                const double q = P.clip / (sqrt(sumsq) + 1e-6);
                if (q < 1.0) coef = static_cast<float>(q);
            }
        }
        s_coef = coef;
        s_skip = skip;
    }
    __syncthreads();
    if (s_skip) return;  // non-finite gradient norm: leave every buffer as it is

    const float coef = s_coef;
    const StepConsts c{P.b1, P.b2, P.omb1, P.omb2, P.eps, P.sqrtbc2};
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStepThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kStepThreads + threadIdx.x; i < P.n_vec; i += stride) {
        float dfac = P.dfac[0];
        float stepsize = P.stepsize[0];
#pragma unroll
        for (int k = 1; k < ZERO1_NUM_GROUPS; ++k) {
            if (i >= P.group_begin_vec[k]) {
                dfac = P.dfac[k];
                stepsize = P.stepsize[k];
            }
        }
        const float4* g4 = reinterpret_cast<const float4*>(P.grad) + 2 * i;
        float4* p4 = reinterpret_cast<float4*>(P.master) + 2 * i;
        float4* m4 = reinterpret_cast<float4*>(P.m) + 2 * i;
        float4* v4 = reinterpret_cast<float4*>(P.v) + 2 * i;
        // Issue all eight 16-byte loads before any arithmetic.
        const float4 ga = g4[0], gb = g4[1];
        float4 pa = p4[0], pb = p4[1];
        float4 ma = m4[0], mb = m4[1];
        float4 va = v4[0], vb = v4[1];

        adamw_elem(pa.x, ma.x, va.x, ga.x, coef, dfac, stepsize, c);
        adamw_elem(pa.y, ma.y, va.y, ga.y, coef, dfac, stepsize, c);
        adamw_elem(pa.z, ma.z, va.z, ga.z, coef, dfac, stepsize, c);
        adamw_elem(pa.w, ma.w, va.w, ga.w, coef, dfac, stepsize, c);
        adamw_elem(pb.x, mb.x, vb.x, gb.x, coef, dfac, stepsize, c);
        adamw_elem(pb.y, mb.y, vb.y, gb.y, coef, dfac, stepsize, c);
        adamw_elem(pb.z, mb.z, vb.z, gb.z, coef, dfac, stepsize, c);
        adamw_elem(pb.w, mb.w, vb.w, gb.w, coef, dfac, stepsize, c);

        p4[0] = pa;
        p4[1] = pb;
        m4[0] = ma;
        m4[1] = mb;
        v4[0] = va;
        v4[1] = vb;
        if (kWriteBf16) {
            uint4 w;
            w.x = pack_bf16x2(pa.x, pa.y);
            w.y = pack_bf16x2(pa.z, pa.w);
            w.z = pack_bf16x2(pb.x, pb.y);
            w.w = pack_bf16x2(pb.z, pb.w);
            reinterpret_cast<uint4*>(P.w)[i] = w;
        }
    }
}

}  // namespace

cudaError_t launch_step(const StepParams& p, cudaStream_t stream) {
    if (p.n_vec == 0) return cudaSuccess;
    const bool bf16 = p.w != nullptr;
    const void* fn = bf16 ? reinterpret_cast<const void*>(&adamw_step_kernel<true>)
                          : reinterpret_cast<const void*>(&adamw_step_kernel<false>);
    const int64_t grid = streaming_grid(fn, kStepThreads, p.n_vec);
    if (bf16)
        adamw_step_kernel<true><<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(p);
    else
        adamw_step_kernel<false><<<static_cast<unsigned>(grid), kStepThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace zero1
