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
#include "zero1_internal.h"

namespace zero1 {
namespace {

constexpr int kAccThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

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

__global__ void __launch_bounds__(kAccThreads)
    accumulate_kernel(const __grid_constant__ AccumulateParams P, int64_t first_vec) {
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
    g4[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    g4[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

}  // namespace

cudaError_t launch_accumulate(const AccumulateParams& p, cudaStream_t stream) {
    for (int64_t first = 0; first < p.n_vec; first += kMaxGridVectors(kAccThreads)) {
        const int64_t n = p.n_vec - first < kMaxGridVectors(kAccThreads) ? p.n_vec - first : kMaxGridVectors(kAccThreads);
        accumulate_kernel<<<static_cast<unsigned>((n + kAccThreads - 1) / kAccThreads), kAccThreads, 0, stream>>>(p, first);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace zero1
