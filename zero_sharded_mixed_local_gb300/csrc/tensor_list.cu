// The local-shard step over a LIST of tensors: every parameter's shard of
// grad, master, m, v and the bf16 copy is its own buffer, as a framework
// holds it when each parameter keeps its own optimizer state ("ZeRO-1 风格的
// Distributed Optimizer", section 6.3: each parameter is cut on its own, and
// each rank keeps the fp32 master weights and Adam moments of its slice of
// every parameter).
//
// Multi-tensor apply: a chunk table (ListChunk, built with the plan) cuts
// every tensor's shard into runs of at most kNormTile = 16384 elements.  A
// block finds its run in the table and its buffers' addresses in the caller's
// device pointer lists (broadcast loads that L1 serves to the whole block),
// then streams the run with the arena kernels' arithmetic (elementwise.cuh),
// so results are bit-identical to the arena calls for the same inputs; the
// work per launch does not depend on how many tensors there are or how large
// they are.
//
// In the gradient passes one block owns one run and thread t the 8-element
// vectors t, t + 256, ..., t + 7*256 (the arena norm tile mapping), so the norm
// partial of a run is formed in a fixed order and the total is deterministic.
// The step has no reduction and splits each run over four blocks.  Vectors
// move as 16-byte loads and stores when every buffer of the run starts on a
// 16-byte boundary (runs start at multiples of 16384 elements, so this is a
// property of the tensor); a run of a buffer that does not, and the last
// partial vector of a shard, fall back to element-wise accesses with the same
// arithmetic.
//
// Bandwidth depends on where the buffers start: a run whose buffers are not
// 128-byte aligned touches one cache line more per warp access and shares its
// edge lines with the neighbouring tensor's runs (on the 20,000-tensor list,
// shards packed at 32-byte offsets stepped 6% slower than the same shards in
// separate 512-byte-aligned allocations).
#include "elementwise.cuh"
#include "launch.cuh"
#include "l2_policy.cuh"
#include "pair_sum.cuh"

namespace zero1 {
namespace {

// Eight consecutive elements from x (n of them valid, the rest read as 0).
__device__ __forceinline__ void load8(const float* x, int n, bool vec, float (&f)[8]) {
    if (vec) {
        const float4 a = reinterpret_cast<const float4*>(x)[0];
        const float4 b = reinterpret_cast<const float4*>(x)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = j < n ? x[j] : 0.f;
    }
}

__device__ __forceinline__ void store8(float* x, int n, bool vec, const float (&f)[8]) {
    if (vec) {
        reinterpret_cast<float4*>(x)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(x)[1] = make_float4(f[4], f[5], f[6], f[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < n) x[j] = f[j];
    }
}

// store8, and the bf16 rounding of eight values, with the evict_last L2 priority on the vector
// path (the step's results; l2_policy.cuh).
__device__ __forceinline__ void store8_last(float* x, int n, bool vec, const float (&f)[8], uint64_t pol) {
    if (vec) {
        store_f32x4(reinterpret_cast<float4*>(x), make_float4(f[0], f[1], f[2], f[3]), pol);
        store_f32x4(reinterpret_cast<float4*>(x) + 1, make_float4(f[4], f[5], f[6], f[7]), pol);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < n) x[j] = f[j];
    }
}

__device__ __forceinline__ void load8_bf16(const uint16_t* x, int n, bool vec, float (&f)[8]) {
    if (vec) {
        widen8(*reinterpret_cast<const uint4*>(x), f);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = j < n ? bf16_bits_to_float(x[j]) : 0.f;
    }
}

__device__ __forceinline__ void store8_bf16_last(uint16_t* x, int n, bool vec, const float (&f)[8], uint64_t pol) {
    if (vec) {
        uint4 w;
        w.x = pack_bf16x2(f[0], f[1]);
        w.y = pack_bf16x2(f[2], f[3]);
        w.z = pack_bf16x2(f[4], f[5]);
        w.w = pack_bf16x2(f[6], f[7]);
        store_u32x4(reinterpret_cast<uint4*>(x), w, pol);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < n) x[j] = bf16_rne_bits(f[j]);
    }
}

__device__ __forceinline__ bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// A run descriptor this launch can use: a table built for another plan (more
// tensors, or corrupted) is skipped rather than read through.
__device__ __forceinline__ bool run_in_range(const ListChunk& ch, int32_t n_tensors) {
    return ch.tensor >= 0 && ch.tensor < n_tensors && ch.len >= 1 && ch.len <= kNormTile &&
           ch.group < ZERO1_MAX_GROUPS && ch.offset >= 0;
}

// Gradient passes over the runs: accumulate (as zero1_accumulate), accumulate
// and take the norm partials (as zero1_accumulate_norm), the partials alone
// (as zero1_grad_norm), or the partials of one micro-batch's gradient without
// writing it (as zero1_micro_norm; kK = 1).  One block per run, thread t owning vectors t + 256r
// (r = 0..7, the norm's fixed order).  Every thread reads the run descriptor
// and its buffers' addresses itself (broadcast loads through L1), so nothing
// waits on a barrier before the data loads go out.  A run whose list entry is
// NULL is skipped (the upload call rejects such lists).
//
// kK = 0 handles any micro-batch count and either overwrite mode, through the
// element-wise-capable loop (or, for one micro-batch or the norm alone, a full
// aligned run's loads two vectors ahead).  kK = 1..8 is the overwriting pass
// over exactly kK micro-batches: their addresses stay in registers and a full
// aligned run issues all kK loads of a vector (of two vectors, for kK <= 4)
// before the additions, which run in micro-batch order as in kK separate calls.
//
// kK = 1 (grad = the one micro-batch): 6 blocks per SM (registers capped at 40,
// a few spilled).  The micro-batch norm form holds all eight vectors: 5 blocks
// per SM (48 registers, a few spilled; 0.354 ms on the 1.0B-element shard,
// against 0.375 at 4 blocks and 0.366 at 6).  Measured on the 1.0B-element shard, fused pass: 0.911 ms,
// against 0.978 ms for batches of four at 5 blocks, 1.001 ms uncapped and
// 0.985 ms for a shared-memory prologue behind a barrier.
template <ListGradMode kMode, int kK>
__global__ void __launch_bounds__(kTileThreads,
                                  kMode == ListGradMode::kMicroNorm ? 5 : (kK == 1 ? 6 : 4))
    list_grad_kernel(const __grid_constant__ ListParams P, float2* __restrict__ partials, int64_t first_chunk) {
    pdl_enter();
    constexpr bool kReadsMicro = kMode != ListGradMode::kNorm;
    constexpr bool kSumsSquares = kMode != ListGradMode::kAccumulate;
    constexpr bool kUsesGrad = kMode != ListGradMode::kMicroNorm;
    constexpr bool kWritesGrad = kMode == ListGradMode::kAccumulate || kMode == ListGradMode::kAccumulateNorm;
    constexpr int kBatch = 2;
    constexpr int kSlots = kK > 0 ? kK : 1;
    __shared__ float2 s_warp[kTileThreads / 32];
    const int64_t c = first_chunk + blockIdx.x;
    const ListChunk ch = P.table[c];
    if (!run_in_range(ch, P.n_tensors)) {  // the same for every thread of the block
        if (kSumsSquares && threadIdx.x == 0) partials[c] = make_float2(0.f, 0.f);
        return;
    }
    float* grad = kUsesGrad ? P.grad[ch.tensor] : nullptr;
    bool missing = kUsesGrad && grad == nullptr, unaligned = false;
    const uint16_t* micro0 = nullptr;
    const uint16_t* mp[kSlots];
    if (kReadsMicro) {
        if (kK > 0) {
#pragma unroll
            for (int k = 0; k < kSlots; ++k) {
                const uint16_t* mk = P.micro[static_cast<int64_t>(k) * P.n_tensors + ch.tensor];
                missing |= mk == nullptr;
                mp[k] = mk != nullptr ? mk + ch.offset : nullptr;
                unaligned |= misaligned16(mp[k]);
            }
            micro0 = mp[0];
        } else {
            for (int k = 0; k < P.n_micro; ++k) {
                const uint16_t* mk = P.micro[static_cast<int64_t>(k) * P.n_tensors + ch.tensor];
                missing |= mk == nullptr;
                if (mk != nullptr) unaligned |= misaligned16(mk + ch.offset);
                if (k == 0 && mk != nullptr) micro0 = mk + ch.offset;
            }
        }
    }
    if (missing) {  // the same for every thread of the block
        if (kSumsSquares && threadIdx.x == 0) partials[c] = make_float2(0.f, 0.f);
        return;
    }
    if (kUsesGrad) {
        grad += ch.offset;
        unaligned |= misaligned16(grad);
    }
    const int len = ch.len;
    const bool overwrite = kK > 0 || (kReadsMicro && P.overwrite_first);
    const bool divide = (kMode == ListGradMode::kAccumulateNorm || kMode == ListGradMode::kMicroNorm) && P.divide;
    const bool full = !unaligned && len == kNormTile;

    SquarePairs sq;
    if (kK >= 2 && full) {
        constexpr int kUnroll = kK <= 4 ? 2 : 1;
#pragma unroll kUnroll
        for (int r = 0; r < kVecsPerThread; ++r) {
            const int v = threadIdx.x + r * kTileThreads;
            uint4 raw[kSlots];
#pragma unroll
            for (int k = 0; k < kSlots; ++k) raw[k] = reinterpret_cast<const uint4*>(mp[k])[v];
            float acc[8];
            widen8(raw[0], acc);
#pragma unroll
            for (int k = 1; k < kSlots; ++k) {
                float f[8];
                widen8(raw[k], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], f[j]);
            }
            if (divide) {
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = __fdiv_rn(acc[j], P.divisor);
            }
            if (kWritesGrad) {
                reinterpret_cast<float4*>(grad)[2 * v] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                reinterpret_cast<float4*>(grad)[2 * v + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            }
            if (kSumsSquares)
                sq.add_vec(make_float4(acc[0], acc[1], acc[2], acc[3]), make_float4(acc[4], acc[5], acc[6], acc[7]));
        }
    } else if (kMode == ListGradMode::kMicroNorm && full && !divide) {
        // as the arena micro-batch norm: all eight vectors loaded, then the squares, without the
        // residual term where all of the thread's squares are exact (the same bits)
        uint4 raw[kVecsPerThread];
#pragma unroll
        for (int r = 0; r < kVecsPerThread; ++r)
            raw[r] = reinterpret_cast<const uint4*>(micro0)[threadIdx.x + r * kTileThreads];
        const bool exact = bf16_squares_exact(raw);
#pragma unroll
        for (int r = 0; r < kVecsPerThread; ++r) {
            float f[8];
            widen8(raw[r], f);
            if (exact)
                sq.add_vec_exact(make_float4(f[0], f[1], f[2], f[3]), make_float4(f[4], f[5], f[6], f[7]));
            else
                sq.add_vec(make_float4(f[0], f[1], f[2], f[3]), make_float4(f[4], f[5], f[6], f[7]));
        }
    } else if (kK <= 1 && full && (kMode == ListGradMode::kNorm || P.n_micro == 1)) {
#pragma unroll
        for (int h = 0; h < kVecsPerThread / kBatch; ++h) {
            uint4 raw[kBatch];
            float4 ga[kBatch], gb[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int v = threadIdx.x + (h * kBatch + q) * kTileThreads;
                if (kReadsMicro) raw[q] = reinterpret_cast<const uint4*>(micro0)[v];
                if (!kReadsMicro || !overwrite) {
                    ga[q] = reinterpret_cast<const float4*>(grad)[2 * v];
                    gb[q] = reinterpret_cast<const float4*>(grad)[2 * v + 1];
                }
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int v = threadIdx.x + (h * kBatch + q) * kTileThreads;
                float acc[8];
                if (kReadsMicro) {
                    float f[8];
                    widen8(raw[q], f);
                    if (overwrite) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[j] = f[j];
                    } else {
                        const float g[8] = {ga[q].x, ga[q].y, ga[q].z, ga[q].w, gb[q].x, gb[q].y, gb[q].z, gb[q].w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(g[j], f[j]);
                    }
                    if (divide) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[j] = __fdiv_rn(acc[j], P.divisor);
                    }
                    if (kWritesGrad) {
                        reinterpret_cast<float4*>(grad)[2 * v] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                        reinterpret_cast<float4*>(grad)[2 * v + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
                    }
                    if (kSumsSquares)
                        sq.add_vec(make_float4(acc[0], acc[1], acc[2], acc[3]),
                                   make_float4(acc[4], acc[5], acc[6], acc[7]));
                } else {
                    sq.add_vec(ga[q], gb[q]);
                }
            }
        }
    } else {
#pragma unroll 1
        for (int r = 0; r < kVecsPerThread; ++r) {
            const int e = 8 * (static_cast<int>(threadIdx.x) + r * kTileThreads);
            if (e >= len) break;  // this thread's later vectors lie beyond the run too
            const int n = len - e < 8 ? len - e : 8;
            const bool vec = !unaligned && n == 8;
            float acc[8];
            if (kMode == ListGradMode::kNorm) {
                load8(grad + e, n, vec, acc);
            } else {
                int k = 0;
                if (overwrite) {
                    load8_bf16(micro0 + e, n, vec, acc);
                    k = 1;
                } else {
                    load8(grad + e, n, vec, acc);
                }
                for (; k < P.n_micro; ++k) {
                    const uint16_t* mk = P.micro[static_cast<int64_t>(k) * P.n_tensors + ch.tensor] + ch.offset;
                    float f[8];
                    load8_bf16(mk + e, n, vec, f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], f[j]);
                }
                if (divide) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = __fdiv_rn(acc[j], P.divisor);
                }
                if (kWritesGrad) store8(grad + e, n, vec, acc);
            }
            if (kSumsSquares)
                sq.add_vec(make_float4(acc[0], acc[1], acc[2], acc[3]), make_float4(acc[4], acc[5], acc[6], acc[7]));
        }
    }
    if (kSumsSquares) {
        sq.fold();
        block_pair_sum<kTileThreads>(sq.s[0], sq.c[0], s_warp);
        if (threadIdx.x == 0) partials[c] = make_float2(sq.s[0], sq.c[0]);
    }
}

// Fused clip + AdamW + bf16 copy over the runs (kDevScalars: the step's
// scalars are read from device memory by thread 0, next to the clip, as the
// arena kernel does for CUDA-graph replay).  Each run is split into
// kStepSubBlocks blocks of 4096 elements (no reduction here, so any mapping
// works): thread t of sub-block s owns vectors 512s + t and 512s + t + 256.
// Every thread reads the run descriptor and the five addresses itself and
// issues its first vector's loads before the block's one barrier, behind which
// thread 0 derives the clip coefficient.  Registers are capped at 64 (4 blocks
// per SM).  Measured per step on the 1.0B-element shard (separately allocated
// tensors): 4.28 ms, against 4.38 ms for one block per run with the addresses
// staged in shared memory behind a barrier; on the 20,000-tensor list 11.70 ms
// against 11.99 ms.
constexpr int kStepSubBlocks = 4;
constexpr int kStepVecsPerThread = kVecsPerThread / kStepSubBlocks;  // 2

// kFromMicro: the one-micro-batch form (zero1_step_accumulate): the gradient of each element is
// float(micro) / divisor, read from micro list 0 and written to the gradient list, also when the
// step is skipped; the arithmetic after that is the same.
template <bool kWriteBf16, bool kDevScalars, bool kFromMicro>
__global__ void __launch_bounds__(kTileThreads, 4) list_step_kernel(const __grid_constant__ ListParams P, int64_t first_block) {
    pdl_enter();
    __shared__ float s_coef;
    __shared__ int s_skip;
    __shared__ zero1_step_scalars s_sc;
    const int64_t b = first_block + blockIdx.x;
    const ListChunk ch = P.table[b / kStepSubBlocks];
    if (!run_in_range(ch, P.n_tensors)) return;  // the same for every thread of the block
    const int sub = static_cast<int>(b % kStepSubBlocks);
    float* master = P.master[ch.tensor];
    float* m = P.m[ch.tensor];
    float* v = P.v[ch.tensor];
    float* grad = P.grad[ch.tensor];
    const uint16_t* micro = kFromMicro ? P.micro[ch.tensor] : nullptr;
    uint16_t* w = kWriteBf16 ? P.w[ch.tensor] : nullptr;
    if (master == nullptr || m == nullptr || v == nullptr || grad == nullptr || (kWriteBf16 && w == nullptr) ||
        (kFromMicro && micro == nullptr))
        return;  // the same for every thread of the block
    master += ch.offset;
    m += ch.offset;
    v += ch.offset;
    grad += ch.offset;
    if (kFromMicro) micro += ch.offset;
    if (kWriteBf16) w += ch.offset;
    const bool aligned = !(misaligned16(master) || misaligned16(m) || misaligned16(v) || misaligned16(grad) ||
                           (kWriteBf16 && misaligned16(w)) || (kFromMicro && misaligned16(micro)));
    // a 32-byte-aligned gradient takes one 256-bit store per vector (whole sectors per warp instruction)
    const bool wide_grad = kFromMicro && aligned && (reinterpret_cast<uintptr_t>(grad) & 31u) == 0;
    const int len = ch.len;
    const int v0 = sub * kStepVecsPerThread * kTileThreads + static_cast<int>(threadIdx.x);

    // the first vector's loads, ahead of the barrier
    const int e0 = 8 * v0;
    const int n0 = len - e0 < 8 ? len - e0 : 8;
    float g[8], p[8], mm[8], vv[8];
    if (e0 < len) {
        const bool vec = aligned && n0 == 8;
        if (kFromMicro)
            load8_bf16(micro + e0, n0, vec, g);
        else
            load8(grad + e0, n0, vec, g);
        load8(master + e0, n0, vec, p);
        load8(m + e0, n0, vec, mm);
        load8(v + e0, n0, vec, vv);
    }
    if (threadIdx.x == 0) {
        double clip = P.sc.clip;
        if (kDevScalars) {
            s_sc = *P.dev_scalars;
            clip = s_sc.clip;
        }
        float coef;
        int skip;
        clip_from_norm(P.norm, clip, coef, skip);
        s_coef = coef;
        s_skip = skip;
    }
    __syncthreads();
    if (e0 >= len || (!kFromMicro && s_skip)) return;  // a non-finite norm leaves every buffer as it is

    const float coef = s_coef;
    const zero1_step_scalars& S = kDevScalars ? s_sc : P.sc;
    const StepConsts sc{S.b1, S.b2, S.omb1, S.omb2, S.eps, S.sqrtbc2};
    const float dfac = S.dfac[ch.group];
    const float stepsize = S.stepsize[ch.group];
    const uint64_t pol = l2_evict_last();  // every result with the evict_last L2 priority
#pragma unroll 1
    for (int r = 0; r < kStepVecsPerThread; ++r) {
        const int e = 8 * (v0 + r * kTileThreads);
        if (e >= len) break;
        const int n = len - e < 8 ? len - e : 8;
        const bool vec = aligned && n == 8;
        if (r > 0) {
            if (kFromMicro)
                load8_bf16(micro + e, n, vec, g);
            else
                load8(grad + e, n, vec, g);
            load8(master + e, n, vec, p);
            load8(m + e, n, vec, mm);
            load8(v + e, n, vec, vv);
        }
        if (kFromMicro) {
            if (P.divide) {
#pragma unroll
                for (int j = 0; j < 8; ++j) g[j] = __fdiv_rn(g[j], P.divisor);
            }
            // the gradient, whether or not the step applies
            if (wide_grad && n == 8)
                store_f32x8(grad + e, make_float4(g[0], g[1], g[2], g[3]), make_float4(g[4], g[5], g[6], g[7]),
                            pol);
            else
                store8_last(grad + e, n, vec, g, pol);
            if (s_skip) continue;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) adamw_elem(p[j], mm[j], vv[j], g[j], coef, dfac, stepsize, sc);
        store8_last(master + e, n, vec, p, pol);
        store8_last(m + e, n, vec, mm, pol);
        store8_last(v + e, n, vec, vv, pol);
        if (kWriteBf16) store8_bf16_last(w + e, n, vec, p, pol);
    }
}

}  // namespace

namespace {

template <ListGradMode kMode, int kK>
cudaError_t launch_k(const ListParams& p, unsigned nb, float2* pairs, int64_t first, cudaStream_t stream) {
    return launch(list_grad_kernel<kMode, kK>, nb, kTileThreads, stream, p, pairs, first);
}

template <ListGradMode kMode>
cudaError_t launch_grad_mode(const ListParams& p, unsigned nb, float2* pairs, int64_t first, cudaStream_t stream) {
    if constexpr (kMode == ListGradMode::kNorm) {
        return launch_k<kMode, 0>(p, nb, pairs, first, stream);
    } else if constexpr (kMode == ListGradMode::kMicroNorm) {
        return launch_k<kMode, 1>(p, nb, pairs, first, stream);
    } else {
        // the micro-batch count, when the pass overwrites the gradient with their sum
        switch (p.overwrite_first ? p.n_micro : 0) {
            case 1: return launch_k<kMode, 1>(p, nb, pairs, first, stream);
            case 2: return launch_k<kMode, 2>(p, nb, pairs, first, stream);
            case 3: return launch_k<kMode, 3>(p, nb, pairs, first, stream);
            case 4: return launch_k<kMode, 4>(p, nb, pairs, first, stream);
            case 5: return launch_k<kMode, 5>(p, nb, pairs, first, stream);
            case 6: return launch_k<kMode, 6>(p, nb, pairs, first, stream);
            case 7: return launch_k<kMode, 7>(p, nb, pairs, first, stream);
            case 8: return launch_k<kMode, 8>(p, nb, pairs, first, stream);
            default: return launch_k<kMode, 0>(p, nb, pairs, first, stream);
        }
    }
}

}  // namespace

cudaError_t launch_list_grad(const ListParams& p, ListGradMode mode, int64_t n_chunks, double* partials,
                             double extra_sumsq, zero1_norm_out* out, cudaStream_t stream) {
    // The workspace holds one 8-byte (hi, lo) float pair per run.
    float2* pairs = reinterpret_cast<float2*>(partials);
    for (int64_t first = 0; first < n_chunks; first += 0x7fffffff) {
        const unsigned nb = static_cast<unsigned>(n_chunks - first < 0x7fffffff ? n_chunks - first : 0x7fffffff);
        cudaError_t e = cudaSuccess;
        switch (mode) {
            case ListGradMode::kAccumulate:
                e = launch_grad_mode<ListGradMode::kAccumulate>(p, nb, pairs, first, stream);
                break;
            case ListGradMode::kAccumulateNorm:
                e = launch_grad_mode<ListGradMode::kAccumulateNorm>(p, nb, pairs, first, stream);
                break;
            case ListGradMode::kNorm:
                e = launch_grad_mode<ListGradMode::kNorm>(p, nb, pairs, first, stream);
                break;
            case ListGradMode::kMicroNorm:
                e = launch_grad_mode<ListGradMode::kMicroNorm>(p, nb, pairs, first, stream);
                break;
        }
        if (e != cudaSuccess) return e;
    }
    if (mode == ListGradMode::kAccumulate) return cudaSuccess;
    return launch_norm_final(pairs, n_chunks, extra_sumsq, out, stream);
}

cudaError_t launch_list_step(const ListParams& p, int64_t n_chunks, cudaStream_t stream) {
    const int64_t n_blocks = n_chunks * kStepSubBlocks;
    for (int64_t first = 0; first < n_blocks; first += 0x7fffffff) {
        const unsigned nb = static_cast<unsigned>(n_blocks - first < 0x7fffffff ? n_blocks - first : 0x7fffffff);
        cudaError_t e;
        if (p.micro_step)
            e = p.w != nullptr ? launch(list_step_kernel<true, false, true>, nb, kTileThreads, stream, p, first)
                               : launch(list_step_kernel<false, false, true>, nb, kTileThreads, stream, p, first);
        else if (p.dev_scalars != nullptr)
            e = p.w != nullptr ? launch(list_step_kernel<true, true, false>, nb, kTileThreads, stream, p, first)
                               : launch(list_step_kernel<false, true, false>, nb, kTileThreads, stream, p, first);
        else
            e = p.w != nullptr ? launch(list_step_kernel<true, false, false>, nb, kTileThreads, stream, p, first)
                               : launch(list_step_kernel<false, false, false>, nb, kTileThreads, stream, p, first);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace zero1
