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
// v, bf16) per element, ~20 fp32 operations.  One thread owns one 8-element
// vector and the grid covers the whole arena (one wave after another, no
// grid-stride loop): on GB300 this keeps DRAM busier than a persistent grid,
// which measured ~20% slower because too few loads were in flight per SM.
// Each thread issues its eight 16-byte loads before thread 0 derives the clip
// coefficient from the device-resident norm, so that prologue hides under the
// load latency.  The weight-decay group of a vector is found by comparing its
// index with the group boundaries (groups are contiguous in the arena), so no
// per-tensor table is read.  The rounding-explicit intrinsics (__fmul_rn,
// __fadd_rn, __fdiv_rn, __fsqrt_rn) are never contracted into FMAs, which
// keeps the operation order exact (elementwise.cuh).
//
// The one-micro-batch form (kFromMicro): with a single micro-batch the gradient
// is float(micro) / divisor, exactly what the accumulate pass would write, so
// the step reads the 2-byte micro-batch instead of the 4-byte gradient and
// writes the gradient itself (a 256-bit store where it is 32-byte aligned).
// Its norm comes first from a pass that only reads the micro-batch
// (micro_sumsq_tiles_kernel).  Per element the two passes move 2 + 32 bytes
// instead of 6 + 30, with the same values: the gradient, the norm record and
// every state element are bit for bit those of zero1_accumulate_norm +
// zero1_step.  A skipped step (non-finite norm) still writes the gradient.
#include "elementwise.cuh"
#include "l2_policy.cuh"
#include "launch.cuh"
#include "store8.cuh"
#include "zero1_internal.h"

namespace zero1 {
namespace {

constexpr int kStepThreads = 256;

// kDevScalars: the scalars come from P.dev_scalars (read by thread 0 into
// shared memory after the loads are issued) rather than from P.sc.
// kFromMicro: the one-micro-batch form above; kWideGrad: its gradient store
// is one 256-bit access.
template <bool kWriteBf16, bool kDevScalars, bool kFromMicro, bool kWideGrad>
__global__ void __launch_bounds__(kStepThreads) adamw_step_kernel(const __grid_constant__ StepParams P, int64_t first_vec) {
    pdl_enter();
    __shared__ float s_coef;
    __shared__ int s_skip;
    __shared__ zero1_step_scalars s_sc;
    const int64_t i = first_vec + static_cast<int64_t>(blockIdx.x) * kStepThreads + threadIdx.x;
    const bool live = i < P.n_vec;

    // Loads first: they do not depend on the clip coefficient.
    float4 ga, gb, pa, pb, ma, mb, va, vb;
    uint4 raw;
    if (live) {
        const float4* p4 = reinterpret_cast<const float4*>(P.master) + 2 * i;
        const float4* m4 = reinterpret_cast<const float4*>(P.m) + 2 * i;
        const float4* v4 = reinterpret_cast<const float4*>(P.v) + 2 * i;
        if (kFromMicro) {
            raw = reinterpret_cast<const uint4*>(P.micro)[i];
        } else {
            const float4* g4 = reinterpret_cast<const float4*>(P.grad) + 2 * i;
            ga = g4[0];
            gb = g4[1];
        }
        pa = p4[0];
        pb = p4[1];
        ma = m4[0];
        mb = m4[1];
        va = v4[0];
        vb = v4[1];
    }
    if (threadIdx.x == 0) {
        double clip = P.sc.clip;
        if (kDevScalars) {
            s_sc = *P.dev_scalars;
            clip = s_sc.clip;
        }
        // Clip coefficient from the device-resident norm: no host round trip
        // (the rule of clip_from_norm, written out here because the call form
        // costs the device-scalar variant four registers, 62 -> 66).
        float coef = 1.0f;
        int skip = 0;
        if (P.norm != nullptr) {
            const double sumsq = P.norm->sumsq;
            if (P.norm->status != ZERO1_OK || !isfinite(sumsq)) {
                skip = 1;
            } else if (clip > 0.0) {
                const double q = clip / (sqrt(sumsq) + 1e-6);
                if (q < 1.0) coef = static_cast<float>(q);
            }
        }
        s_coef = coef;
        s_skip = skip;
    }
    __syncthreads();
    if (kFromMicro) {
        if (!live) return;
        float f[8];
        widen8(raw, f);
        if (P.divide) {
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __fdiv_rn(f[j], P.divisor);
        }
        ga = make_float4(f[0], f[1], f[2], f[3]);
        gb = make_float4(f[4], f[5], f[6], f[7]);
        const uint64_t pol = l2_evict_last();
        if (kWideGrad) {
            store_f32x8(P.grad_out + 8 * i, ga, gb, pol);
        } else {
            float4* g4 = reinterpret_cast<float4*>(P.grad_out) + 2 * i;
            store_f32x4(g4, ga, pol);
            store_f32x4(g4 + 1, gb, pol);
        }
        if (s_skip) return;  // the gradient is written; master, m, v and the bf16 copy stay as they are
    } else if (s_skip || !live) {
        return;  // a non-finite gradient norm leaves every buffer as it is
    }

    const float coef = s_coef;
    const zero1_step_scalars& S = kDevScalars ? s_sc : P.sc;
    const StepConsts c{S.b1, S.b2, S.omb1, S.omb2, S.eps, S.sqrtbc2};
    float dfac = S.dfac[0];
    float stepsize = S.stepsize[0];
#pragma unroll
    for (int k = 1; k < ZERO1_MAX_GROUPS; ++k) {
        if (i >= P.group_begin_vec[k]) {
            dfac = S.dfac[k];
            stepsize = S.stepsize[k];
        }
    }
    adamw_elem(pa.x, ma.x, va.x, ga.x, coef, dfac, stepsize, c);
    adamw_elem(pa.y, ma.y, va.y, ga.y, coef, dfac, stepsize, c);
    adamw_elem(pa.z, ma.z, va.z, ga.z, coef, dfac, stepsize, c);
    adamw_elem(pa.w, ma.w, va.w, ga.w, coef, dfac, stepsize, c);
    adamw_elem(pb.x, mb.x, vb.x, gb.x, coef, dfac, stepsize, c);
    adamw_elem(pb.y, mb.y, vb.y, gb.y, coef, dfac, stepsize, c);
    adamw_elem(pb.z, mb.z, vb.z, gb.z, coef, dfac, stepsize, c);
    adamw_elem(pb.w, mb.w, vb.w, gb.w, coef, dfac, stepsize, c);

    float4* p4 = reinterpret_cast<float4*>(P.master) + 2 * i;
    float4* m4 = reinterpret_cast<float4*>(P.m) + 2 * i;
    float4* v4 = reinterpret_cast<float4*>(P.v) + 2 * i;
    // every result with the evict_last L2 priority (l2_policy.cuh)
    const uint64_t pol = l2_evict_last();
    store_f32x4(p4, pa, pol);
    store_f32x4(p4 + 1, pb, pol);
    store_f32x4(m4, ma, pol);
    store_f32x4(m4 + 1, mb, pol);
    store_f32x4(v4, va, pol);
    store_f32x4(v4 + 1, vb, pol);
    if (kWriteBf16) {
        uint4 w;
        w.x = pack_bf16x2(pa.x, pa.y);
        w.y = pack_bf16x2(pa.z, pa.w);
        w.z = pack_bf16x2(pb.x, pb.y);
        w.w = pack_bf16x2(pb.z, pb.w);
        store_u32x4(reinterpret_cast<uint4*>(P.w) + i, w, pol);
    }
}

}  // namespace

cudaError_t launch_step(const StepParams& p, cudaStream_t stream) {
    // One thread per 8-element vector; grids beyond the launch limit are split.
    for (int64_t first = 0; first < p.n_vec; first += kMaxGridVectors(kStepThreads)) {
        const int64_t n = p.n_vec - first < kMaxGridVectors(kStepThreads) ? p.n_vec - first : kMaxGridVectors(kStepThreads);
        const unsigned grid = static_cast<unsigned>((n + kStepThreads - 1) / kStepThreads);
        cudaError_t e;
        if (p.micro != nullptr) {
            const bool wide = wide_store_aligned(p.grad_out);
            if (p.w != nullptr)
                e = wide ? launch(adamw_step_kernel<true, false, true, true>, grid, kStepThreads, stream, p, first)
                         : launch(adamw_step_kernel<true, false, true, false>, grid, kStepThreads, stream, p, first);
            else
                e = wide ? launch(adamw_step_kernel<false, false, true, true>, grid, kStepThreads, stream, p, first)
                         : launch(adamw_step_kernel<false, false, true, false>, grid, kStepThreads, stream, p, first);
        } else if (p.dev_scalars != nullptr) {
            e = p.w != nullptr ? launch(adamw_step_kernel<true, true, false, false>, grid, kStepThreads, stream, p, first)
                               : launch(adamw_step_kernel<false, true, false, false>, grid, kStepThreads, stream, p, first);
        } else {
            e = p.w != nullptr ? launch(adamw_step_kernel<true, false, false, false>, grid, kStepThreads, stream, p, first)
                               : launch(adamw_step_kernel<false, false, false, false>, grid, kStepThreads, stream, p, first);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace zero1
