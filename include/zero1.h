/*
 * zero1.h -- C ABI of the ZeRO-1 local-shard optimizer step for GB300 (sm_103a).
 *
 * One data-parallel rank's step under ZeRO-1 mixed precision, as the pages
 * describe it ("ZeRO-1 风格的 Distributed Optimizer", sections 6.2-6.3 and
 * 6.7; "Nanotron Guide: Minimalist 3D-Parallelism LLM Training", "Memory &
 * Optimization", item 1; "Distributed Training", sections 0, 2 and 3):
 *
 *   1. zero1_accumulate  add K bf16 micro-batch gradients into an fp32 grad buffer
 *   2. zero1_grad_norm   global L2 norm of the accumulated gradient (for clip_grad)
 *   3. zero1_step        AdamW on the fp32 master / m / v shard, clip applied on
 *                        the fly, and the bf16 weight copy the all-gather ships
 *
 * preceded once by zero1_plan_create, which cuts every parameter tensor by
 * numel into dp_size contiguous shards and lays the local shards out in one
 * flat "arena" per quantity.
 *
 * The same step in other shapes (the arena ones give the results of the
 * three calls bit for bit; the list ones take the norm's partials per run of
 * a shard, so their sum of squares can differ from the arena's in its last
 * bits):
 *   zero1_accumulate_norm        the last micro-batch's pass and the norm together
 *   zero1_micro_norm,            one micro-batch: the norm from it, then the
 *   zero1_step_accumulate        step that writes the fp32 gradient it uses
 *   zero1_local_step             the whole step in one call
 *   zero1_list_*                 the calls over one buffer per tensor shard
 *   zero1_step_dev, zero1_list_step_dev
 *                                the step's scalars read from device memory
 *                                (CUDA-graph replay)
 *   zero1_grad_norm_static       the norm without a caller workspace
 * and around it zero1_shard_gather / zero1_shard_scatter, the model layout <->
 * arena copies on either side of the data-parallel exchanges.
 *
 * Conventions (all entry points):
 *   - Plain pointers and sizes only.  Device pointers are CUDA global-memory
 *     addresses on the current device; host pointers are ordinary memory.
 *   - The caller allocates and owns every device buffer (grad, master, m, v,
 *     bf16 copy, micro-batch gradients, norm workspace, norm output).  The
 *     library allocates no device memory and keeps no pointer after a call
 *     returns.  A plan owns only host memory.
 *   - Every device buffer must start on a 16-byte boundary (ZERO1_EALIGN).
 *   - Compute calls are asynchronous on the given stream (a cudaStream_t
 *     passed as void*; NULL is the legacy default stream).  They launch
 *     kernels and return; nothing synchronises except zero1_read_norm.
 *   - Return value: ZERO1_OK (0) or a negative ZERO1_E* code.  Argument errors
 *     are detected before any launch and leave every buffer untouched.  No
 *     call aborts the process, traps or waits on the GPU.
 *   - Thread safety: a plan is read-only after creation and may be shared by
 *     threads; buffers may not be shared by concurrent calls.
 */
#ifndef ZERO1_H
#define ZERO1_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define ZERO1_OK 0
#define ZERO1_EINVAL (-1)     /* null pointer, bad size, rank >= dp_size, t < 1, ... */
#define ZERO1_EALIGN (-2)     /* a buffer is not 16-byte aligned */
#define ZERO1_ECUDA (-3)      /* a CUDA call or launch failed; see zero1_last_cuda_error() */
#define ZERO1_ENONFINITE (-4) /* device status: the gradient norm is inf or NaN */
#define ZERO1_ENOMEM (-5)     /* host allocation failed while building a plan */
#define ZERO1_ETOOBIG (-6)    /* the arena exceeds zero1_grad_norm_static's fixed scratch */

/* Each shard starts on a multiple of this many elements inside an arena, so
 * that 16-byte vector loads of bf16 (8 elements) never straddle tensors. */
#define ZERO1_ARENA_ALIGN 8
/* The numels of one plan add up to at most this many elements (2^56). */
#define ZERO1_MAX_TOTAL_NUMEL (((int64_t)1) << 56)
/* Tensors are grouped (at most ZERO1_MAX_GROUPS groups); each group has its
 * own learning-rate and weight-decay multipliers.  zero1_plan_create's
 * no_decay flags make group 0 (decayed) and group 1 (excluded). */
#define ZERO1_MAX_GROUPS 8
/* Most micro-batch gradients one zero1_accumulate call accepts. */
#define ZERO1_MAX_MICRO 16

typedef struct zero1_plan zero1_plan; /* opaque, host memory only */

/* AdamW hyper-parameters ("ZeRO-1 风格的 Distributed Optimizer", section 6.6:
 * adam_beta1 0.9, adam_beta2 0.95, adam_eps 1e-8, weight_decay 0.1,
 * clip_grad 1.0).  Doubles, so decimal settings arrive unrounded; the library
 * derives the fp32 step scalars once per call.  clip_grad <= 0 disables
 * clipping. */
typedef struct zero1_hparams {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    double clip_grad;
} zero1_hparams;

/* Result of zero1_grad_norm.  Lives in DEVICE memory (24 bytes; 16-byte
 * alignment is required as for every buffer).  zero1_step reads `sumsq` and
 * `status` and derives the norm itself, so with several data-parallel ranks
 * the caller may all-reduce (sum) the `sumsq` double in place between
 * zero1_grad_norm and zero1_step: that one scalar is the only exchange the
 * step needs, and a non-finite sum on any rank makes every rank skip. */
typedef struct zero1_norm_out {
    double sumsq;     /* local sum of squares + extra_sumsq */
    double norm;      /* sqrt(sumsq) */
    int32_t status;   /* ZERO1_OK, or ZERO1_ENONFINITE if sumsq is inf/NaN */
    int32_t n_partials; /* number of per-tile partial sums that were reduced */
} zero1_norm_out;

/* ---- plan (host only; no CUDA call) ------------------------------------- */

/* Build the shard plan of rank dp_rank out of dp_size.
 * "ZeRO-1 风格的 Distributed Optimizer", section 6.3: each parameter is cut on
 * its own, its total numel split evenly over the dp_size ranks (not one
 * flattened blob).  Remainder rule (not stated on the page): shards are
 * contiguous in rank order and the first (numel mod dp_size) ranks get one
 * extra element, so a tensor with fewer than dp_size elements leaves some
 * ranks with an empty shard.
 *   numels[n_tensors]   total elements of each parameter tensor (>= 0), in
 *                       model order
 *   no_decay[n_tensors] 1 = excluded from weight decay (norm weights), else 0
 *   out                 receives the plan; free it with zero1_plan_destroy
 * Arena layout: the decayed tensors' shards first, then the excluded ones,
 * each group in model order; every shard starts on a multiple of
 * ZERO1_ARENA_ALIGN elements.  Arena buffers hold zero1_plan_arena_numel()
 * elements; the padding elements between shards must be zero when the
 * buffers are created and the library keeps them zero.
 * Errors: ZERO1_EINVAL (n_tensors < 0, dp_size < 1, dp_rank outside
 * [0, dp_size), a negative numel, numels adding up to more than
 * ZERO1_MAX_TOTAL_NUMEL, a no_decay value other than 0/1, a null pointer
 * with n_tensors > 0, out == NULL), ZERO1_ENOMEM. */
int zero1_plan_create(const int64_t* numels, const uint8_t* no_decay, int32_t n_tensors,
                      int32_t dp_size, int32_t dp_rank, zero1_plan** out);

/* zero1_plan_create with parameter groups ("Nanotron Guide", "3. Spectral
 * muTransfer": learning rates scaled per layer class, eta_hidden = eta_0 /
 * d_model; torch-style param groups with their own lr and weight decay).
 *   group[n_tensors]            group of each tensor, 0 .. ZERO1_MAX_GROUPS-1
 *   lr_scale[ZERO1_MAX_GROUPS]  per-group multiplier of hparams.lr, or NULL
 *                               for all 1
 *   wd_scale[ZERO1_MAX_GROUPS]  per-group multiplier of hparams.weight_decay,
 *                               or NULL for 1 everywhere except group 1 (0)
 * Group g then steps with lr_g = lr*lr_scale[g] and wd_g = weight_decay *
 * wd_scale[g] (decay factor 1 - lr_g*wd_g).  The arena holds the groups in
 * increasing group order, each in model order.  Scales must be finite and
 * >= 0.  zero1_plan_create(numels, no_decay, ...) is this call with
 * group = no_decay and both scale arrays NULL.
 * Errors: as zero1_plan_create, plus ZERO1_EINVAL for a group id out of range
 * or a bad scale. */
int zero1_plan_create_grouped(const int64_t* numels, const uint8_t* group, int32_t n_tensors,
                              const double* lr_scale, const double* wd_scale, int32_t dp_size,
                              int32_t dp_rank, zero1_plan** out);

/* Multipliers of group g (either output may be NULL). */
int zero1_plan_group_scales(const zero1_plan* plan, int32_t g, double* lr_scale, double* wd_scale);

/* Free a plan (NULL is ignored). */
void zero1_plan_destroy(zero1_plan* plan);

/* Plan queries; on a NULL plan they return -1. */
int32_t zero1_plan_num_tensors(const zero1_plan* plan);
int64_t zero1_plan_total_numel(const zero1_plan* plan); /* sum of numels, all ranks */
int64_t zero1_plan_local_numel(const zero1_plan* plan); /* sum of this rank's shards */
int64_t zero1_plan_arena_numel(const zero1_plan* plan); /* padded arena length */

/* Tensor i's shard: elements [shard_start, shard_start + shard_numel) of the
 * flattened tensor, stored at arena[arena_offset ...].  Any output pointer
 * may be NULL.  ZERO1_EINVAL if plan is NULL or i is out of range. */
int zero1_plan_tensor(const zero1_plan* plan, int32_t i, int64_t* shard_start,
                      int64_t* shard_numel, int64_t* arena_offset);

/* Arena element range [begin, end) of group g (0 .. ZERO1_MAX_GROUPS-1;
 * empty for a group with no tensors). */
int zero1_plan_group_range(const zero1_plan* plan, int32_t g, int64_t* begin, int64_t* end);

/* Bytes one rank holds under ZeRO-1 mixed precision ("Distributed Training",
 * section 0: 2 + 2 + 12 = 16 bytes per parameter; "ZeRO-1 风格的 Distributed
 * Optimizer", sections 6.1 and 6.3: only the 12 bytes of fp32 master, m and v
 * are sharded, the bf16 weights and gradients stay whole).
 *   grad_bytes  2 (bf16 gradient, the 16-byte count) or 4 (fp32 gradient,
 *               the 18-byte itemisation of the Nanotron guide)
 *   out[4]      {bf16 weights, gradients, optimizer state of the local shard,
 *               total}, in bytes */
int zero1_plan_bytes(const zero1_plan* plan, int32_t grad_bytes, int64_t out[4]);

/* Device workspace zero1_grad_norm needs (8 bytes, one float pair, per
 * 16384-element tile of the arena); 0 for an empty arena. */
size_t zero1_workspace_bytes(const zero1_plan* plan);

/* ---- compute (asynchronous on `stream`) ---------------------------------- */

/* Gradient accumulation ("ZeRO-1 风格的 Distributed Optimizer", section 6.7:
 * micro-batch gradients are added into .grad before the data-parallel
 * reduction and the optimizer step; "Distributed Training", section 2; the
 * Nanotron config's accumulate_grad_in_fp32).  Element-wise over the arena:
 *     grad = bf16->fp32(micro[0])            if overwrite_first
 *     grad = grad + bf16->fp32(micro[k])     for the other k, in order
 * every addition a single fp32 rounding; a plain sum (no 1/K).
 *   grad          device fp32 arena (arena_numel), read and written
 *   micro_bf16    HOST array of n_micro pointers to bf16 arenas (raw bits as
 *                 uint16), read only.  Each may be device memory, or host
 *                 memory the device can read: pinned/registered memory
 *                 always, ordinary pageable memory where the device reads
 *                 host page tables (Grace-based GB300 nodes).  Host arenas
 *                 are read by the kernel itself over the CPU-GPU link, with
 *                 no staging copy.
 *   n_micro       1 .. ZERO1_MAX_MICRO
 * Errors: ZERO1_EINVAL (including a host pointer this device cannot read),
 * ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_accumulate(const zero1_plan* plan, float* grad, const uint16_t* const* micro_bf16,
                     int32_t n_micro, int32_t overwrite_first, void* stream);

/* Global gradient L2 norm for clipping ("ZeRO-1 风格的 Distributed
 * Optimizer", section 6.6, clip_grad).  sumsq = sum over the arena of grad^2
 * (padding adds 0) + extra_sumsq, where extra_sumsq is the other ranks' share
 * of the global sum (0 when this rank is alone); norm = sqrt(sumsq), in
 * double.  Every partial sum is an unevaluated pair of floats (hi + lo) that
 * carries the exact rounding error of each square and of each addition, so
 * the total is within ~1e-13 relative of the exact sum of squares; the
 * reduction order is fixed by 16384-element tiles, so the result is
 * deterministic and independent of launch shape.
 *   grad        device fp32 arena, read only
 *   workspace   device scratch of zero1_workspace_bytes(plan) bytes
 *               (may be NULL when that is 0); contents are overwritten
 *   d_out       device zero1_norm_out, written (status ZERO1_ENONFINITE if
 *               the sum is inf or NaN)
 * Errors: ZERO1_EINVAL (workspace_bytes too small, ...), ZERO1_EALIGN,
 * ZERO1_ECUDA. */
int zero1_grad_norm(const zero1_plan* plan, const float* grad, double extra_sumsq,
                    void* workspace, size_t workspace_bytes, zero1_norm_out* d_out, void* stream);

/* zero1_accumulate and zero1_grad_norm in one pass, for the last micro-batch
 * of a step ("ZeRO-1 风格的 Distributed Optimizer", section 6.7: the norm is
 * taken once all micro-batch gradients are in .grad).  The gradient written
 * is bit-identical to zero1_accumulate's and the norm record to
 * zero1_grad_norm's (same tiles, same summation order; with grad_divisor 1),
 * but the gradient is
 * not read back for the norm: 4 bytes per element less traffic.
 *   grad, micro_bf16, n_micro, overwrite_first   as for zero1_accumulate
 *   grad_divisor  after the last addition each element is divided by this
 *                 (rounded to fp32; one IEEE division), before its square is
 *                 taken: the average over data-parallel ranks that FSDP2
 *                 runs as a single divide kernel after the fp32
 *                 reduce-scatter ("TorchTitan 生产级预训练方案", appendix B.1).
 *                 1 keeps the plain sum (no division); must be finite > 0,
 *                 and stay so once rounded to fp32 (else ZERO1_EINVAL)
 *   extra_sumsq, workspace, workspace_bytes, d_out  as for zero1_grad_norm
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_accumulate_norm(const zero1_plan* plan, float* grad, const uint16_t* const* micro_bf16,
                          int32_t n_micro, int32_t overwrite_first, double grad_divisor, double extra_sumsq,
                          void* workspace, size_t workspace_bytes, zero1_norm_out* d_out, void* stream);

/* Fused clip + AdamW + bf16 copy over the local shard ("ZeRO-1 风格的
 * Distributed Optimizer", sections 6.2-6.3: each rank updates only its own
 * fp32 master / m / v and then all-gathers the updated bf16 weights; section
 * 6.6 for the hyper-parameters).  Decoupled weight decay applied to p before
 * the bias-corrected Adam update, eps outside the square root:
 *     coef = clip/(norm+1e-6) if that is < 1 and clip > 0, else 1
 *     g = grad*coef;  p = p*dfac;  m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g)
 *     d = sqrt(v)/sqrt(1-b2^t) + eps;  p = p - lr/(1-b1^t) * (m/d);  w = bf16_rne(p)
 * where each parameter group g uses lr_g = lr*lr_scale[g] in place of lr and
 * dfac = 1 - lr_g*weight_decay*wd_scale[g] (by default group 0 decays and
 * group 1 does not); each fp32 operation is rounded once (IEEE divide and
 * square root), the step scalars are computed in double and rounded once to
 * fp32.  The clipped gradient is not written back.
 *   master, exp_avg, exp_avg_sq   device fp32 arenas, read and written
 *   grad                          device fp32 arena, read only
 *   weight_bf16                   device bf16 arena (uint16 bits), written;
 *                                 may be NULL to skip the copy
 *   hp                            HOST pointer
 *   step_t                        1-based step count used by bias correction
 *   d_norm                        device result of zero1_grad_norm (its
 *                                 sumsq possibly summed across ranks), or
 *                                 NULL for no clipping; norm = sqrt(sumsq) in
 *                                 double; if status is not ZERO1_OK or sumsq
 *                                 is not finite the kernel writes nothing
 *                                 (the step is skipped)
 * Errors: ZERO1_EINVAL (step_t < 1, non-finite or out-of-range
 * hyper-parameters, ...), ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_step(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq,
               const float* grad, uint16_t* weight_bf16, const zero1_hparams* hp, int64_t step_t,
               const zero1_norm_out* d_norm, void* stream);

/* ---- the step of a single micro-batch in two passes ----------------------
 * With one micro-batch the fp32 gradient is float(micro) / grad_divisor, known
 * before it is written ("ZeRO-1 风格的 Distributed Optimizer", section 6.7:
 * the micro-batch gradient goes into .grad, then the reduction and the step).
 * So the norm can be taken from the 2-byte micro-batch, and the step can read
 * the micro-batch instead of the 4-byte gradient and write the gradient in
 * the same pass: 2 + 32 bytes per element instead of 6 + 30 for
 * zero1_accumulate_norm + zero1_step, with the same gradient, norm record,
 * master, m, v and bf16 copy, bit for bit. */

/* The norm record zero1_accumulate_norm(n_micro = 1, overwrite_first = 1)
 * would write, without writing the gradient: the sum of squares of
 * float(micro[j]) / grad_divisor over the arena, with the same tiles and
 * summation order, plus extra_sumsq.
 *   micro_bf16   device bf16 arena (or readable host memory, as for
 *                zero1_accumulate)
 *   grad_divisor, extra_sumsq, workspace, workspace_bytes, d_out
 *                as for zero1_accumulate_norm
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_micro_norm(const zero1_plan* plan, const uint16_t* micro_bf16, double grad_divisor, double extra_sumsq,
                     void* workspace, size_t workspace_bytes, zero1_norm_out* d_out, void* stream);

/* zero1_step for the gradient of one micro-batch, accumulated in the same
 * pass: every element's gradient float(micro[j]) / grad_divisor is written to
 * grad (what zero1_accumulate_norm would write) and feeds that element's
 * clipped AdamW update and bf16 copy, exactly as zero1_step would.  d_norm is
 * normally zero1_micro_norm's record of the same micro-batch (its sumsq
 * possibly summed across ranks).  When the step is skipped (a non-finite
 * norm) the gradient is still written and nothing else is.
 *   grad         device fp32 arena, written (not read)
 *   micro_bf16   device bf16 arena (or readable host memory), read
 *   grad_divisor as for zero1_accumulate_norm
 *   master, exp_avg, exp_avg_sq, weight_bf16, hp, step_t, d_norm
 *                as for zero1_step
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_step_accumulate(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq, float* grad,
                          const uint16_t* micro_bf16, double grad_divisor, uint16_t* weight_bf16,
                          const zero1_hparams* hp, int64_t step_t, const zero1_norm_out* d_norm, void* stream);

/* The whole local step of one rank in one call ("ZeRO-1 风格的 Distributed
 * Optimizer", section 6.7: every micro-batch's gradient accumulated into the
 * fp32 .grad, then the reduction and the optimizer step; sections 6.2-6.3 and
 * 6.6 for the step): zero1_accumulate_norm over all n_micro micro-batches
 * with the first one overwriting grad, then zero1_step reading the norm
 * record that pass wrote; for a single micro-batch, zero1_micro_norm then
 * zero1_step_accumulate instead.  Either way the results are those two calls'
 * bit for bit; it saves a caller, a binding above all, one crossing of the ABI
 * and its per-call checks, which is what bounds the step of a small shard.
 * Every argument of both passes is checked before the first launch, so an
 * error leaves every buffer unchanged.  There is no point between the two
 * passes to sum the sum of squares across ranks: pass the other ranks' share
 * as extra_sumsq when it is known, else use the two calls.
 *   grad, micro_bf16, n_micro, grad_divisor, extra_sumsq, workspace,
 *   workspace_bytes, d_norm       as for zero1_accumulate_norm (d_norm must
 *                                 not be NULL)
 *   master, exp_avg, exp_avg_sq, weight_bf16, hp, step_t   as for zero1_step
 * Errors: those of zero1_accumulate_norm and zero1_step. */
int zero1_local_step(const zero1_plan* plan, float* grad, const uint16_t* const* micro_bf16, int32_t n_micro,
                     double grad_divisor, double extra_sumsq, void* workspace, size_t workspace_bytes,
                     zero1_norm_out* d_norm, float* master, float* exp_avg, float* exp_avg_sq,
                     uint16_t* weight_bf16, const zero1_hparams* hp, int64_t step_t, void* stream);

/* Largest plan zero1_grad_norm_static serves: its fixed scratch holds one
 * 8-byte partial per 16384-element tile, 262144 tiles (2 MiB per GPU), i.e.
 * arenas of up to 2^32 elements. */
#define ZERO1_STATIC_NORM_MAX_TILES 262144
#define ZERO1_STATIC_NORM_MAX_NUMEL ((int64_t)ZERO1_STATIC_NORM_MAX_TILES * 16384)

/* zero1_grad_norm without a workspace argument: same result, bit for bit, but
 * the per-tile partial sums live in a fixed array inside the library, so the
 * call allocates nothing and the caller needs no scratch buffer.  The pages
 * have no counterpart of this call; it exists for callers that cannot supply
 * or allocate device scratch: a plain C program with no device allocator of
 * its own, a process whose framework allocator already holds nearly all of
 * the GPU's memory, or a step that must not call cudaMalloc/cudaFree (which
 * can synchronise the device).
 *   grad, extra_sumsq, d_out, stream   as for zero1_grad_norm
 * Limits and sharing: arenas above ZERO1_STATIC_NORM_MAX_NUMEL elements are
 * rejected with ZERO1_ETOOBIG before any launch.  The 2 MiB array stays
 * allocated on every GPU that loads the library until the process exits.
 * All calls on a device share it; nothing in it needs to start at zero
 * (each call writes every partial it reads first), but calls whose kernels
 * overlap on the GPU (different streams or threads) race on it, so the
 * caller must serialise them.  The first call on each device looks up the
 * array's device address with that device current; make that first call
 * before any stream capture.  The address is kept with the ID of the CUDA
 * context it belongs to and looked up again when another context is current
 * (after cudaDeviceReset, or a driver-API caller's own context); make the
 * first call in such a context before any capture too.
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ETOOBIG, ZERO1_ECUDA. */
int zero1_grad_norm_static(const zero1_plan* plan, const float* grad, double extra_sumsq,
                           zero1_norm_out* d_out, void* stream);

/* ---- the step with its scalars in device memory (for CUDA graphs) ------- */

/* The fp32 scalars zero1_step derives from (hparams, plan groups, step_t):
 * per group the step size lr_g/(1-beta1^t) and the decay factor
 * 1 - lr_g*wd_g, then beta1, beta2, 1-beta1, 1-beta2, eps, sqrt(1-beta2^t)
 * (each computed in double and rounded once), and clip_grad. */
typedef struct zero1_step_scalars {
    float stepsize[ZERO1_MAX_GROUPS];
    float dfac[ZERO1_MAX_GROUPS];
    float b1, b2, omb1, omb2, eps, sqrtbc2;
    double clip;
} zero1_step_scalars; /* 96 bytes */

/* Host only: the scalars zero1_step would use for (plan, hp, step_t).
 * Errors: ZERO1_EINVAL, as zero1_step's hyper-parameter checks. */
int zero1_step_scalars_fill(const zero1_plan* plan, const zero1_hparams* hp, int64_t step_t,
                            zero1_step_scalars* out);

/* zero1_step with the scalars read from DEVICE memory (d_scalars, 16-byte
 * aligned) when the kernel runs, not passed at launch.  A CUDA graph that
 * captured this call can therefore replay every step: the caller writes the
 * next step's scalars (zero1_step_scalars_fill) where a captured copy picks
 * them up.  Same arithmetic and results as zero1_step.  The pages have no
 * counterpart of this call; it exists so the local step can be replayed as
 * one graph launch.
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_step_dev(const zero1_plan* plan, float* master, float* exp_avg, float* exp_avg_sq,
                   const float* grad, uint16_t* weight_bf16, const zero1_step_scalars* d_scalars,
                   const zero1_norm_out* d_norm, void* stream);

/* Copy a device zero1_norm_out to the host, synchronising `stream` first.
 * Errors: ZERO1_EINVAL, ZERO1_ECUDA. */
int zero1_read_norm(const zero1_norm_out* d_norm, void* stream, zero1_norm_out* host_out);

/* ---- model layout <-> arena (the exchanges around the step) -------------- */

/* The data movement on either side of the local step ("ZeRO-1 风格的
 * Distributed Optimizer", section 6.3: after backward, gradients are
 * reduce-scattered to the rank that owns each shard; after the step, the
 * updated bf16 weights are all-gathered).  The "model layout" holds every
 * parameter whole, concatenated in model order without padding (tensor i at
 * [sum of earlier numels, + numel_i)), zero1_plan_total_numel() elements.
 *
 * Packing a reduce-scatter: for each rank r, zero1_shard_gather with rank
 * r's plan copies that rank's shard of the full gradient into chunk r of the
 * send buffer (chunks of the largest arena size).  Unpacking an all-gather:
 * zero1_shard_scatter with each rank's plan copies chunk r back into the
 * full bf16 weights.  The same calls move optimizer state between a
 * checkpoint in model layout and any dp_size's shards (resharding). */

/* Device bytes of the plan's copy table (24 per run of up to 16384 shard
 * elements); 0 for an empty shard. */
size_t zero1_layout_table_bytes(const zero1_plan* plan);

/* Copy the plan's table into caller-owned device memory d_table (16-byte
 * aligned, at least zero1_layout_table_bytes bytes).  Asynchronous on
 * `stream`; the plan may be destroyed once the call returns.  The table is
 * valid only for this plan.
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_layout_table_upload(const zero1_plan* plan, void* d_table, size_t table_bytes, void* stream);

/* arena[arena_offset_i + k] = full[model_offset_i + shard_start_i + k] for
 * every tensor i and k < shard_numel_i; padding is not written.
 *   d_table     this plan's uploaded table
 *   full        device buffer in model layout (total_numel elements),
 *               aligned to elem_bytes
 *   arena       device arena (arena_numel elements), 16-byte aligned
 *   elem_bytes  2 (bf16 or any 16-bit type) or 4 (fp32); the bits are copied
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_shard_gather(const zero1_plan* plan, const void* d_table, const void* full, void* arena,
                       int32_t elem_bytes, void* stream);

/* The reverse: full[model_offset_i + shard_start_i + k] = arena[arena_offset_i
 * + k]; elements of full outside this rank's shard are not written. */
int zero1_shard_scatter(const zero1_plan* plan, const void* d_table, const void* arena, void* full,
                        int32_t elem_bytes, void* stream);

/* ---- tensor lists: one buffer per tensor shard ---------------------------- */

/* The same step over shards that live in separate buffers, one per tensor,
 * as a framework holds them when each parameter keeps its own optimizer state
 * ("ZeRO-1 风格的 Distributed Optimizer", section 6.3: every parameter is cut
 * on its own, and each rank keeps the fp32 state of its slice of every
 * parameter).  No arena and no copy into one: tensor i's buffers hold exactly
 * shard_numel_i elements (zero1_plan_tensor), with no padding.
 *
 * A "pointer list" is a DEVICE array of n_tensors pointers (8 bytes each,
 * model order), entry i pointing at tensor i's buffer of one quantity;
 * entries of tensors whose shard is empty are never read and may be NULL.
 * Build lists with zero1_list_ptrs_upload, which checks every entry.  The
 * kernels walk a chunk table (zero1_list_table_upload) that cuts each shard
 * into runs of at most 16384 elements; one thread block owns one run and
 * stages the run's descriptor and buffer addresses in shared memory, so one
 * launch serves any number and mix of tensor sizes.  A run moves 16-byte
 * vectors when all its buffers start on 16-byte boundaries and falls back to
 * element-wise accesses otherwise (same results, lower bandwidth).
 *
 * Results: the gradient, master, m, v and bf16 copy are bit-identical to the
 * arena calls' on the same values (same per-element operations in the same
 * order); the norm record is deterministic and within ~1e-13 relative of the
 * exact sum of squares, but its partial sums follow the runs rather than
 * arena tiles, so its last bits may differ from zero1_grad_norm's.  Error
 * behaviour is as for the arena calls. */

/* Device bytes of the plan's run table (16 per run: element offset in the
 * tensor's buffer, tensor index, length, group); 0 for an empty shard. */
size_t zero1_list_table_bytes(const zero1_plan* plan);

/* Copy the run table into caller-owned device memory d_table (16-byte
 * aligned, at least zero1_list_table_bytes bytes).  Asynchronous on `stream`;
 * the plan may be destroyed once the call returns.  Valid only for this plan:
 * like buffer lengths, which plan a device table came from cannot be checked
 * (the kernels only skip a run whose tensor index, length or group is out of
 * range for the plan they are called with, so a stray table cannot send them
 * past the pointer lists).
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_table_upload(const zero1_plan* plan, void* d_table, size_t table_bytes, void* stream);

/* Device workspace of the tensor-list norm passes (8 bytes per run). */
size_t zero1_list_workspace_bytes(const zero1_plan* plan);

/* Check n_lists pointer lists and copy them into device memory d_lists.
 *   host_ptrs   HOST array of n_lists * n_tensors device addresses, list k
 *               at [k*n_tensors, (k+1)*n_tensors); each entry of a tensor
 *               with a non-empty shard must be non-NULL and a multiple of
 *               elem_bytes (its natural alignment).  The array may be freed
 *               once the call returns (the library stages it first).
 *   n_lists     1 .. ZERO1_MAX_MICRO (several micro-batch lists at once)
 *   elem_bytes  4 (fp32 buffers) or 2 (bf16 buffers)
 *   d_lists     device destination, 16-byte aligned, at least
 *               n_lists * n_tensors * 8 bytes (lists_bytes)
 * Asynchronous on `stream` (not capturable into a CUDA graph: the source is
 * pageable memory).  The library cannot check the buffers' lengths: buffer i
 * must hold shard_numel_i elements.
 * Errors: ZERO1_EINVAL (a NULL entry, a bad count or size), ZERO1_EALIGN (a
 * misaligned entry or d_lists), ZERO1_ENOMEM, ZERO1_ECUDA. */
int zero1_list_ptrs_upload(const zero1_plan* plan, const void* const* host_ptrs, int32_t n_lists,
                           int32_t elem_bytes, void* d_lists, size_t lists_bytes, void* stream);

/* zero1_accumulate over tensor lists.
 *   d_table   this plan's uploaded run table
 *   d_grad    pointer list of the fp32 gradient shards, read and written
 *   d_micro   n_micro pointer lists of bf16 micro-batch gradient shards,
 *             back to back in one device array (n_micro * n_tensors entries)
 *   n_micro, overwrite_first   as for zero1_accumulate
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_accumulate(const zero1_plan* plan, const void* d_table, float* const* d_grad,
                          const uint16_t* const* d_micro, int32_t n_micro, int32_t overwrite_first, void* stream);

/* zero1_accumulate_norm over tensor lists: accumulate, optionally divide by
 * grad_divisor, and the norm record, in one pass.  workspace holds
 * zero1_list_workspace_bytes(plan) bytes; other arguments as above and as for
 * zero1_accumulate_norm.
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_accumulate_norm(const zero1_plan* plan, const void* d_table, float* const* d_grad,
                               const uint16_t* const* d_micro, int32_t n_micro, int32_t overwrite_first,
                               double grad_divisor, double extra_sumsq, void* workspace, size_t workspace_bytes,
                               zero1_norm_out* d_out, void* stream);

/* zero1_micro_norm over the tensor lists: the norm record
 * zero1_list_accumulate_norm(one micro-batch list, overwrite_first = 1) would
 * write, without writing the gradient; the same runs and summation order.
 *   d_micro   one device list of n_tensors bf16 shard pointers
 *   grad_divisor, extra_sumsq, workspace, workspace_bytes, d_out
 *             as for zero1_list_accumulate_norm
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_micro_norm(const zero1_plan* plan, const void* d_table, const uint16_t* const* d_micro,
                          double grad_divisor, double extra_sumsq, void* workspace, size_t workspace_bytes,
                          zero1_norm_out* d_out, void* stream);

/* zero1_grad_norm over a gradient pointer list (read only).
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_grad_norm(const zero1_plan* plan, const void* d_table, const float* const* d_grad,
                         double extra_sumsq, void* workspace, size_t workspace_bytes, zero1_norm_out* d_out,
                         void* stream);

/* zero1_step over tensor lists: clip + AdamW + bf16 copy, each tensor with
 * its group's step size and decay factor.
 *   d_master, d_exp_avg, d_exp_avg_sq   pointer lists of fp32 shards, read
 *                                       and written
 *   d_grad                              pointer list of fp32 shards, read
 *   d_weight_bf16                       pointer list of bf16 shards, written;
 *                                       NULL to skip the copy
 *   hp, step_t, d_norm                  as for zero1_step
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_step(const zero1_plan* plan, const void* d_table, float* const* d_master,
                    float* const* d_exp_avg, float* const* d_exp_avg_sq, const float* const* d_grad,
                    uint16_t* const* d_weight_bf16, const zero1_hparams* hp, int64_t step_t,
                    const zero1_norm_out* d_norm, void* stream);

/* zero1_step_accumulate over the tensor lists: every shard's gradient
 * float(micro) / grad_divisor is written to its gradient buffer and feeds the
 * same clipped AdamW update and bf16 copy as zero1_list_step; a skipped step
 * still writes the gradient.  The same results as zero1_list_accumulate_norm
 * (one micro-batch, overwriting) + zero1_list_step, bit for bit, in 34 bytes
 * per element instead of 36.
 *   d_grad   the gradient list, written (not read)
 *   d_micro  one device list of bf16 shard pointers, read
 *   other arguments as for zero1_list_step and zero1_list_accumulate_norm
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_step_accumulate(const zero1_plan* plan, const void* d_table, float* const* d_master,
                               float* const* d_exp_avg, float* const* d_exp_avg_sq, float* const* d_grad,
                               const uint16_t* const* d_micro, double grad_divisor, uint16_t* const* d_weight_bf16,
                               const zero1_hparams* hp, int64_t step_t, const zero1_norm_out* d_norm, void* stream);

/* zero1_list_step with the step's scalars read from DEVICE memory (d_scalars,
 * 16-byte aligned, filled by zero1_step_scalars_fill) when the kernel runs, so
 * a CUDA graph that captured the call can replay every step; the tensor-list
 * counterpart of zero1_step_dev, with the same arithmetic and results as
 * zero1_list_step.  The pages have no counterpart of this call.
 * Errors: ZERO1_EINVAL, ZERO1_EALIGN, ZERO1_ECUDA. */
int zero1_list_step_dev(const zero1_plan* plan, const void* d_table, float* const* d_master,
                        float* const* d_exp_avg, float* const* d_exp_avg_sq, const float* const* d_grad,
                        uint16_t* const* d_weight_bf16, const zero1_step_scalars* d_scalars,
                        const zero1_norm_out* d_norm, void* stream);

/* ---- diagnostics --------------------------------------------------------- */

/* Static description of a status code. */
const char* zero1_strerror(int code);

/* Kernel launches the library has issued since it was loaded, over all
 * threads: a diagnostic, so a caller can count the kernels its calls cost
 * and see that they reach the GPU.  A launch made while a stream is being
 * captured into a CUDA graph counts once, at capture; graph replays do not
 * count.  Never fails. */
uint64_t zero1_launch_count(void);

/* Text of the CUDA error behind the calling thread's last ZERO1_ECUDA
 * ("" if none). */
const char* zero1_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO1_H */
