"""GB300-native ZeRO-1 local-shard optimizer step (sm_103a).

One data-parallel rank's part of a ZeRO-1 mixed-precision training step, as
described for nanotron's distributed optimizer: accumulate bf16 micro-batch
gradients in fp32, take the global gradient L2 norm for clipping, run AdamW
on the fp32 master / m / v shard and write the bf16 weights the all-gather
ships.  The work runs in hand-written CUDA kernels behind the C ABI of
``libzero1.so`` (``include/zero1.h``); this package is its thin binding.
"""
from .binding import (ARENA_ALIGN, MAX_GROUPS, MAX_MICRO, NORM_OUT_BYTES, ZERO1_EALIGN, ZERO1_ECUDA,
                      ZERO1_EINVAL, ZERO1_ENOMEM, ZERO1_ENONFINITE, ZERO1_ETOOBIG, ZERO1_OK, Hparams, LocalShardAdamW, Plan,
                      ShardLayout, Zero1Error, accumulate, accumulate_norm, allreduce_sumsq_, decode_norm, exchange_chunk_numel, grad_norm, grad_norm_static, load_library,
                      pack_reduce_scatter, shard_gather, shard_scatter, unpack_all_gather, new_norm_out,
                      read_norm, step, step_dev, step_scalars, StepGraph, PointerLists, ShardListAdamW,
                      list_accumulate, list_accumulate_norm, list_grad_norm, list_step)

__all__ = [
    "ARENA_ALIGN", "MAX_GROUPS", "MAX_MICRO", "NORM_OUT_BYTES", "ZERO1_EALIGN", "ZERO1_ECUDA", "ZERO1_EINVAL",
    "ZERO1_ENOMEM", "ZERO1_ENONFINITE", "ZERO1_ETOOBIG", "ZERO1_OK", "Hparams", "LocalShardAdamW", "Plan", "ShardLayout",
    "Zero1Error", "accumulate", "accumulate_norm", "allreduce_sumsq_", "decode_norm", "exchange_chunk_numel", "grad_norm", "grad_norm_static", "load_library",
    "pack_reduce_scatter", "shard_gather", "shard_scatter", "unpack_all_gather", "new_norm_out", "read_norm", "step", "step_dev", "step_scalars", "StepGraph",
    "PointerLists", "ShardListAdamW", "list_accumulate", "list_accumulate_norm", "list_grad_norm", "list_step",
]

from . import checkpoint  # noqa: E402
from .optim import Zero1AdamW, default_no_decay  # noqa: E402
from .schedules import lr_at, mup_groups  # noqa: E402

__all__ += ["checkpoint", "lr_at", "mup_groups", "Zero1AdamW", "default_no_decay"]
