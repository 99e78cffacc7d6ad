"""One rank's whole ZeRO-1 data-parallel step: the exchanges around the local step.

"ZeRO-1 风格的 Distributed Optimizer", sections 6.2-6.3 and 6.7: every rank runs
forward and backward on its own data with the full bf16 weights; after the
backward passes the gradients are reduce-scattered so each rank holds the
sum for the numel slice of every parameter it owns; each rank steps only its
own fp32 master / m / v shard; then the updated bf16 weights are all-gathered
so every rank holds the full model again.  ``DataParallelStep`` runs that
sequence for one rank around a ``LocalShardAdamW``:

1. pack: this rank's bf16 model-layout gradient of one micro-batch is laid out
   as one chunk per destination rank, each in the destination's arena layout
   (``zero1_shard_gather``, one launch per rank);
2. reduce-scatter, deterministically: an all-to-all moves chunk r to rank r
   (the same bytes per rank as a ring reduce-scatter of bf16), and the owner adds
   the world's chunks in fp32, in (micro-batch, rank) order, with the library's
   accumulate kernels.  Nothing is rounded to bf16 between ranks, and the sum does
   not depend on the collective's algorithm: any world size gives the same bits
   as one rank adding the same gradients in the same order;
3. the last addition divides the finished sum by the world size once per element
   (FSDP2's single divide of the fp32 reduce-scattered gradient, "TorchTitan"
   appendix B.1) and takes the local sum of squares in the same pass;
4. the sums of squares are all-reduced (one double) and every rank steps its
   shard with the same clip coefficient (a non-finite sum on any rank makes every
   rank skip);
5. the step writes its bf16 copy straight into this rank's all-gather send
   buffer, and an all-gather plus ``zero1_shard_scatter`` (one launch per rank)
   give the full model-layout bf16 weights.

With NCCL the collectives run on the device buffers.  With any other backend
(gloo on CPU) they run on pinned host copies of them, so the same class drives
a CPU process group in tests; the kernels run on the GPU either way.
"""
import torch

from .binding import MAX_MICRO, exchange_chunk_numel, shard_gather, shard_scatter


class DataParallelStep:
    """The data-parallel step of the rank that owns ``opt`` (a LocalShardAdamW whose plan has
    dp_size = the group's size and dp_rank = this rank's rank in it).

    ``average`` divides the reduced gradient by the world size (the data-parallel mean);
    without it the gradient is the plain sum over ranks and micro-batches."""

    def __init__(self, opt, group=None, average=True):
        import torch.distributed as dist
        self.dist = dist
        self.opt, self.group, self.average = opt, group, bool(average)
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        plan = opt.plan
        if plan.dp_size != self.world or plan.dp_rank != self.rank:
            raise ValueError("the optimizer's plan is dp_size %d rank %d; the group has %d ranks and this is rank %d"
                             % (plan.dp_size, plan.dp_rank, self.world, self.rank))
        self.plans = [plan if r == self.rank else plan.for_rank(r) for r in range(self.world)]
        self.chunk = exchange_chunk_numel(self.plans)
        dev = self.device = opt.device
        n, bf = self.world * self.chunk, torch.bfloat16
        self.send = torch.zeros(n, dtype=bf, device=dev)   # padding zero once; the packs write only shards
        self.recv = torch.empty(n, dtype=bf, device=dev)
        self.wsend = torch.zeros(self.chunk, dtype=bf, device=dev)
        self.wrecv = torch.empty(n, dtype=bf, device=dev)
        # the step writes its bf16 copy into the all-gather send buffer: no copy before the gather
        arena = plan.arena_numel
        self.wsend[:arena].copy_(opt.weight_bf16)
        opt.weight_bf16 = self.wsend[:arena]
        self.on_device = dist.get_backend(group) == "nccl"
        if not self.on_device:
            self._host = {name: torch.empty(t.numel(), dtype=bf).pin_memory()
                          for name, t in (("send", self.send), ("recv", self.recv), ("wsend", self.wsend),
                                          ("wrecv", self.wrecv))}

    def _collective(self, fn, out_name, in_name):
        out, inp = getattr(self, out_name), getattr(self, in_name)
        if self.on_device:
            fn(out, inp, group=self.group)
            return
        h_out, h_in = self._host[out_name], self._host[in_name]
        # Synchronous copy: it waits for the stream, so the device data is complete, and so is the
        # previous call's asynchronous copy out of any pinned buffer before this one rewrites it.
        h_in.copy_(inp)
        fn(h_out, h_in, group=self.group)
        out.copy_(h_out, non_blocking=True)  # in stream order before the kernels that read it

    def allreduce_sumsq(self):
        """Step 4's exchange: the norm record's sum of squares summed over the ranks, in place."""
        rec = self.opt.norm_out[:8].view(torch.float64)
        if self.on_device:
            self.dist.all_reduce(rec, op=self.dist.ReduceOp.SUM, group=self.group)
            return
        h = rec.cpu()
        self.dist.all_reduce(h, op=self.dist.ReduceOp.SUM, group=self.group)
        rec.copy_(h)

    def reduce_scatter(self, grad_bf16, last):
        """Steps 1-3 for one micro-batch's bf16 model-layout gradient of this rank: pack, all-to-all,
        then the owner's ordered fp32 accumulation (the step's first micro-batch overwrites; with
        ``last`` the sum is divided by the world size and its norm taken)."""
        if grad_bf16.dtype != torch.bfloat16 or grad_bf16.numel() != self.opt.plan.total_numel:
            raise ValueError("the gradient must be bf16 with the model's %d elements" % self.opt.plan.total_numel)
        c = self.chunk
        for r, pl in enumerate(self.plans):
            shard_gather(pl, grad_bf16, self.send[r * c:r * c + pl.arena_numel])
        self._collective(self.dist.all_to_all_single, "recv", "send")
        arena = self.opt.plan.arena_numel
        parts = [self.recv[q * c:q * c + arena] for q in range(self.world)]
        for j in range(0, self.world, MAX_MICRO):
            final = last and j + MAX_MICRO >= self.world
            self.opt.accumulate(parts[j:j + MAX_MICRO], last=final,
                                divisor=float(self.world) if (final and self.average) else 1.0)

    def all_gather(self, weights_out=None):
        """Step 5: every rank's bf16 arena into ``weights_out`` (bf16, model layout), if given."""
        self._collective(self.dist.all_gather_into_tensor, "wrecv", "wsend")
        if weights_out is not None:
            c = self.chunk
            for r, pl in enumerate(self.plans):
                shard_scatter(pl, self.wrecv[r * c:r * c + pl.arena_numel], weights_out)

    def step(self, micro_grads, weights_out=None, lr=None, check_finite=False):
        """The whole data-parallel step for this rank's micro-batch gradients (a bf16 model-layout
        tensor or a list of them, in order), on the current CUDA stream.  Returns what
        ``LocalShardAdamW.step`` returns: with ``check_finite``, whether the step applied."""
        micro = [micro_grads] if isinstance(micro_grads, torch.Tensor) else list(micro_grads)
        if not micro:
            raise ValueError("at least one micro-batch gradient")
        for k, g in enumerate(micro):
            self.reduce_scatter(g, last=(k == len(micro) - 1))
        self.allreduce_sumsq()
        applied = self.opt.step(lr=lr, check_finite=check_finite)
        self.all_gather(weights_out)
        return applied
