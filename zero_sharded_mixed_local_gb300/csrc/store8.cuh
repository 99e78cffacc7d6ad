// 256-bit global stores (sm_100 and later): eight consecutive fp32 values in
// one access, so each warp instruction writes whole 32-byte sectors.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace zero1 {

// The address must be 32-byte aligned; callers choose this form only after
// checking that (wide_store_aligned).
__device__ __forceinline__ void store8_f32(float* p, const float4& a, const float4& b) {
    asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(a.x), "f"(a.y), "f"(a.z),
                 "f"(a.w), "f"(b.x), "f"(b.y), "f"(b.z), "f"(b.w)
                 : "memory");
}

// True when a buffer may take store8_f32 at every 8-element vector.
inline bool wide_store_aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

}  // namespace zero1
