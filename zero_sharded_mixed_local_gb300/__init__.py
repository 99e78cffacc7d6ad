"""GB300-native ZeRO-1 local-shard optimizer step (sm_103a).

One data-parallel rank's part of a ZeRO-1 mixed-precision training step, as
described for nanotron's distributed optimizer: accumulate bf16 micro-batch
gradients in fp32, take the global gradient L2 norm for clipping, run AdamW
on the fp32 master / m / v shard and write the bf16 weights the all-gather
ships.  The work runs in hand-written CUDA kernels behind the C ABI of
``libzero1.so`` (``include/zero1.h``).  ``binding`` is its thin ctypes binding;
``optim`` holds the optimizer objects built on it (arena and tensor-list
shards, CUDA-graph replay, a torch-module wrapper); ``checkpoint`` and
``schedules`` are host-side helpers; ``pipeline`` feeds the step from pinned host
memory with the copies overlapped.
"""
from .binding import (ARENA_ALIGN, MAX_GROUPS, MAX_MICRO, NORM_OUT_BYTES, ZERO1_EALIGN, ZERO1_ECUDA, ZERO1_EINVAL,
                      ZERO1_ENOMEM, ZERO1_ENONFINITE, ZERO1_ETOOBIG, ZERO1_OK, Hparams, Plan, PointerLists,
                      ShardLayout, Zero1Error, accumulate, accumulate_norm, allreduce_sumsq_, decode_norm,
                      exchange_chunk_numel, grad_norm, grad_norm_static, launch_count, list_accumulate,
                      list_accumulate_norm, list_grad_norm, list_micro_norm, list_step, list_step_accumulate,
                      list_step_dev, load_library, local_step, micro_norm, new_norm_out, step_accumulate,
                      pack_reduce_scatter, read_norm, shard_gather, shard_scatter, step, step_dev, step_scalars,
                      unpack_all_gather)
from . import checkpoint
from .optim import LocalShardAdamW, ShardListAdamW, StepGraph, Zero1AdamW, default_no_decay
from .pipeline import HostFedSteps
from .schedules import lr_at, mup_groups

__all__ = [
    # status codes and limits
    "ARENA_ALIGN", "MAX_GROUPS", "MAX_MICRO", "NORM_OUT_BYTES", "ZERO1_EALIGN", "ZERO1_ECUDA", "ZERO1_EINVAL",
    "ZERO1_ENOMEM", "ZERO1_ENONFINITE", "ZERO1_ETOOBIG", "ZERO1_OK", "Zero1Error", "load_library",
    # plan and arena calls
    "Hparams", "Plan", "ShardLayout", "accumulate", "accumulate_norm", "grad_norm", "grad_norm_static", "step",
    "local_step", "micro_norm", "step_accumulate",
    "step_dev", "step_scalars", "new_norm_out", "read_norm", "decode_norm", "allreduce_sumsq_",
    # exchanges
    "exchange_chunk_numel", "pack_reduce_scatter", "shard_gather", "shard_scatter", "unpack_all_gather",
    # tensor lists
    "PointerLists", "list_accumulate", "list_accumulate_norm", "list_grad_norm", "list_micro_norm", "list_step",
    "list_step_accumulate", "list_step_dev",
    # optimizer objects and helpers
    "LocalShardAdamW", "ShardListAdamW", "StepGraph", "Zero1AdamW", "default_no_decay", "checkpoint", "lr_at",
    "mup_groups", "HostFedSteps",
]
