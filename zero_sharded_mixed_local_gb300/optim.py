"""Optimizer objects built on the binding: one rank's ZeRO-1 AdamW state and step.

- ``LocalShardAdamW`` owns one rank's shard as flat arenas.
- ``ShardListAdamW`` owns the same state as one buffer per tensor shard (the
  tensor-list calls).
- ``StepGraph`` replays either one's step as CUDA graphs.
- ``Zero1AdamW`` wraps a torch module's parameters.

The pages' distributed optimizer ("ZeRO-1 风格的 Distributed Optimizer", sections
6.2-6.3) wraps a model's named parameters: each rank keeps the fp32 master
weights and Adam moments of its numel slice of every parameter, steps them,
and the updated bf16 weights reach the model.  ``Zero1AdamW`` does that for one
rank with no copies between the model and the optimizer:

  - the bf16 gradient of each parameter is read where autograd left it, as a
    contiguous view of ``p.grad`` covering this rank's slice;
  - the updated bf16 weights are written straight into the same slice of the
    parameter's own storage (``p.data``);
  - master, m, v and the fp32 gradient accumulator are one buffer per slice.

With ``dp_size`` > 1 the other ranks' slices of ``p.data`` are not touched; the
all-gather that would fill them (and the reduce-scatter that would sum the
gradients before) sit outside this rank's step.  Weight decay is skipped for
parameters the ``no_decay`` predicate selects (by default 1-D parameters:
norm weights and biases).
"""
import dataclasses
import math

import torch

from .binding import (_stream_ptr, accumulate, accumulate_norm, allreduce_sumsq_, grad_norm, Hparams,
                      list_accumulate, list_accumulate_norm, list_grad_norm, list_micro_norm, list_step,
                      list_step_accumulate, list_step_dev, local_step, micro_norm, new_norm_out, Plan, PointerLists,
                      read_norm, step, step_accumulate, step_dev, step_scalars, STEP_SCALARS_BYTES)


def _applied(opt, stream):
    """Whether the step just launched applied; a skipped step gives its number back, so bias
    correction stays matched to the updates m and v received.  The kernel skips on the same
    two conditions: a non-finite local norm (the record's status) or a non-finite sum of
    squares after the all-reduce (another rank's inf or NaN)."""
    rec = read_norm(opt.norm_out, stream=stream)
    if rec["status"] == 0 and math.isfinite(rec["sumsq"]):
        return True
    opt.t -= 1
    return False


class LocalShardAdamW:
    """One data-parallel rank's ZeRO-1 optimizer shard, resident on one GPU.

    Owns the arenas of the local shard (fp32 grad, master, m, v and the bf16
    copy), the norm workspace and record, and the step counter.  A training
    loop calls ``accumulate`` once per micro-batch and ``step`` once per
    global batch; both only launch kernels on the current stream.
    """

    def __init__(self, numels, no_decay=None, dp_size=1, dp_rank=0, hparams=None, device="cuda", groups=None,
                 lr_scale=None, wd_scale=None):
        self.device = torch.device(device)
        self.plan = Plan(numels, no_decay, dp_size, dp_rank, groups=groups, lr_scale=lr_scale, wd_scale=wd_scale)
        self.hp = hparams if isinstance(hparams, Hparams) else Hparams(**(hparams or {}))
        mk = self.plan.new_arena
        self.grad = mk(torch.float32, self.device)
        self.master = mk(torch.float32, self.device)
        self.exp_avg = mk(torch.float32, self.device)
        self.exp_avg_sq = mk(torch.float32, self.device)
        self.weight_bf16 = mk(torch.bfloat16, self.device)
        self.workspace = self.plan.new_workspace(self.device)
        self.norm_out = new_norm_out(self.device)
        self.t = 0
        self._micro_seen = 0

    def accumulate(self, micro, last=False, extra_sumsq=0.0, divisor=1.0, stream=None):
        """Add one (or several) bf16 micro-batch gradient arenas; the first call of a step
        overwrites.  ``last=True`` marks the step's final micro-batch: the gradient norm
        is taken in the same pass (after dividing the sum by ``divisor``, e.g. the world
        size) and step() will not read the gradient for it again."""
        first = self._micro_seen == 0
        if last:
            accumulate_norm(self.plan, self.grad, micro, self.workspace, self.norm_out, overwrite_first=first,
                            extra_sumsq=extra_sumsq, divisor=divisor, stream=stream)
        else:
            accumulate(self.plan, self.grad, micro, overwrite_first=first, stream=stream)
        self._micro_seen += 1 if isinstance(micro, torch.Tensor) else len(micro)
        self._norm_ready = bool(last)

    def step(self, extra_sumsq=0.0, lr=None, group=None, stream=None, check_finite=False):
        """Norm + clip + AdamW + bf16 copy.

        The norm is taken here unless the last accumulate() already did.  With
        ``group`` (a torch.distributed process group of the data-parallel ranks)
        the local sum of squares is all-reduced before the update.  A non-finite
        norm makes the kernel skip the update on the device; the step count ``t``
        still advances unless ``check_finite`` is set, which synchronises, leaves
        ``t`` unchanged for a skipped step and returns whether the step applied
        (otherwise the call returns None without waiting)."""
        if not getattr(self, "_norm_ready", False):
            grad_norm(self.plan, self.grad, self.workspace, self.norm_out, extra_sumsq, stream=stream)
        self._norm_ready = False
        if group is not None:
            allreduce_sumsq_(self.norm_out, group, stream=stream)
        self.t += 1
        hp = self.hp if lr is None else dataclasses.replace(self.hp, lr=lr)
        step(self.plan, self.master, self.exp_avg, self.exp_avg_sq, self.grad, self.weight_bf16, hp, self.t,
             self.norm_out, stream=stream)
        self._micro_seen = 0
        return _applied(self, stream) if check_finite else None

    def step_from(self, micro, extra_sumsq=0.0, divisor=1.0, lr=None, group=None, stream=None, check_finite=False):
        """The whole step from micro-batch gradients that are all resident (a bf16 arena or a list
        of up to MAX_MICRO, in order): accumulate with the norm in one pass, then clip + AdamW +
        bf16 copy; for one micro-batch, the norm from the micro-batch and the step that writes the
        gradient.  The same result as accumulate(micro, last=True) then step().  Without ``group``
        it is one library call (zero1_local_step); with one, the sum of squares is all-reduced
        between the two passes."""
        self.t += 1
        hp = self.hp if lr is None else dataclasses.replace(self.hp, lr=lr)
        if group is None:
            local_step(self.plan, self.grad, micro, self.workspace, self.norm_out, self.master, self.exp_avg,
                       self.exp_avg_sq, self.weight_bf16, hp, self.t, extra_sumsq=extra_sumsq, divisor=divisor,
                       stream=stream)
        else:
            mb = [micro] if isinstance(micro, torch.Tensor) else list(micro)
            if len(mb) == 1:
                micro_norm(self.plan, mb[0], self.workspace, self.norm_out, extra_sumsq, divisor, stream=stream)
                allreduce_sumsq_(self.norm_out, group, stream=stream)
                step_accumulate(self.plan, self.master, self.exp_avg, self.exp_avg_sq, self.grad, mb[0],
                                self.weight_bf16, hp, self.t, self.norm_out, divisor=divisor, stream=stream)
            else:
                accumulate_norm(self.plan, self.grad, mb, self.workspace, self.norm_out, overwrite_first=True,
                                extra_sumsq=extra_sumsq, divisor=divisor, stream=stream)
                allreduce_sumsq_(self.norm_out, group, stream=stream)
                step(self.plan, self.master, self.exp_avg, self.exp_avg_sq, self.grad, self.weight_bf16, hp, self.t,
                     self.norm_out, stream=stream)
        self._micro_seen = 0
        self._norm_ready = False
        return _applied(self, stream) if check_finite else None

    def read_norm(self, stream=None):
        return read_norm(self.norm_out, stream=stream)

    def save_checkpoint(self, path, meta=None, async_=False):
        """Write this rank's master / m / v shard and the step count (see ``checkpoint``)."""
        from . import checkpoint
        fn = checkpoint.save_async if async_ else checkpoint.save
        return fn(path, self.plan, self.master, self.exp_avg, self.exp_avg_sq, self.t, meta)

    def load_checkpoint(self, path):
        """Fill master / m / v from a checkpoint written at any dp size; restores the step count."""
        from . import checkpoint
        self.t = checkpoint.load(path, self.plan, self.master, self.exp_avg, self.exp_avg_sq)
        self._micro_seen = 0
        self._norm_ready = False
        return self.t


class StepGraph:
    """The whole local step of a LocalShardAdamW or a ShardListAdamW captured as CUDA graphs.

    One replay runs what accumulate(..., last=True) + step() launch: the
    accumulation of the micro-batch buffers given here (their contents at
    replay time), the fused norm, and the AdamW pass.  For a ShardListAdamW
    each micro-batch is a list of per-tensor bf16 shard tensors or a
    PointerLists; their pointer lists are uploaded here, before capture.  The
    step's scalars (which change with t and lr) are not baked into the graph:
    before each replay the host writes them into a pinned buffer that a
    captured copy moves to the device.  Two graphs over two pinned buffers
    alternate, so the host may write step t+1's scalars while step t still
    runs; it waits only for step t-1.  No collective is captured: use it where
    the sum of squares needs no all-reduce (one rank, or a caller that
    all-reduces the norm record in its own graph).  A replay whose norm is not
    finite leaves the state untouched (the kernel skips) while ``t`` still advances,
    as with ``step()`` without ``check_finite``.
    """

    def __init__(self, opt, micro_buffers):
        self.opt = opt
        self.lists = isinstance(opt, ShardListAdamW)
        micro = list(micro_buffers)
        if not micro:
            raise ValueError("at least one micro-batch buffer")
        if self.lists:  # uploads cannot run inside a capture
            micro = [m if isinstance(m, PointerLists) else PointerLists(opt.plan, m, torch.bfloat16, opt.device)
                     for m in micro]
        self.micro = micro
        dev = opt.device
        self.h = [torch.zeros(128, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.d = [torch.zeros(128, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.done = [torch.cuda.Event(), torch.cuda.Event()]
        self._warm_kernels(dev)
        self.graphs = [self._capture(b) for b in range(2)]

    def _warm_kernels(self, dev):
        # Load every kernel the graph uses (lazy module loading) on a throwaway one-tensor plan,
        # with the same sequence of calls, so the capture itself launches nothing for the first time.
        tiny = Plan([16], [0])
        sc = torch.frombuffer(bytearray(step_scalars(tiny, self.opt.hp, 1)), dtype=torch.uint8).to(dev)
        ws, nout = None, new_norm_out(dev)
        if self.lists:
            def one(dtype):
                return [torch.zeros(16, dtype=dtype, device=dev)]
            f32 = [PointerLists(tiny, one(torch.float32), torch.float32, dev) for _ in range(4)]
            wl = PointerLists(tiny, one(torch.bfloat16), torch.bfloat16, dev)
            mbs = [PointerLists(tiny, [one(torch.bfloat16) for _ in range(m.n_lists)], torch.bfloat16, dev)
                   for m in self.micro]
            table, ws = tiny.list_table(dev), tiny.new_list_workspace(dev)
            for k, mb in enumerate(mbs[:-1]):
                list_accumulate(tiny, table, f32[0], mb, overwrite_first=(k == 0))
            list_accumulate_norm(tiny, table, f32[0], mbs[-1], ws, nout, overwrite_first=(len(mbs) == 1))
            list_step_dev(tiny, table, f32[1], f32[2], f32[3], f32[0], wl, sc, nout)
        else:
            a = [tiny.new_arena(torch.float32, dev) for _ in range(4)]
            w = tiny.new_arena(torch.bfloat16, dev)
            mbs = [tiny.new_arena(torch.bfloat16, dev) for _ in self.micro]
            ws = tiny.new_workspace(dev)
            for k, mb in enumerate(mbs[:-1]):
                accumulate(tiny, a[0], mb, overwrite_first=(k == 0))
            accumulate_norm(tiny, a[0], mbs[-1], ws, nout, overwrite_first=(len(mbs) == 1))
            step_dev(tiny, a[1], a[2], a[3], a[0], w, sc, nout)
        torch.cuda.synchronize(dev)

    def _capture(self, b):
        o = self.opt
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.d[b].copy_(self.h[b], non_blocking=True)
            if self.lists:
                L = o._lists
                for k, mb in enumerate(self.micro[:-1]):
                    list_accumulate(o.plan, o.table, L["grad"], mb, overwrite_first=(k == 0))
                list_accumulate_norm(o.plan, o.table, L["grad"], self.micro[-1], o.workspace, o.norm_out,
                                     overwrite_first=(len(self.micro) == 1))
                list_step_dev(o.plan, o.table, L["master"], L["exp_avg"], L["exp_avg_sq"], L["grad"],
                              L["weight_bf16"], self.d[b], o.norm_out)
            else:
                for k, mb in enumerate(self.micro[:-1]):
                    accumulate(o.plan, o.grad, mb, overwrite_first=(k == 0))
                accumulate_norm(o.plan, o.grad, self.micro[-1], o.workspace, o.norm_out,
                                overwrite_first=(len(self.micro) == 1))
                step_dev(o.plan, o.master, o.exp_avg, o.exp_avg_sq, o.grad, o.weight_bf16, self.d[b], o.norm_out)
        return g

    def replay(self, lr=None):
        """One local step at t = opt.t + 1 (lr overrides the optimizer's lr for this step)."""
        o = self.opt
        t = o.t + 1
        b = t % 2
        self.done[b].synchronize()  # the replay that last read pinned buffer b (step t-2) is done
        hp = o.hp if lr is None else dataclasses.replace(o.hp, lr=lr)
        self.h[b][:STEP_SCALARS_BYTES].copy_(torch.frombuffer(bytearray(step_scalars(o.plan, hp, t)),
                                                              dtype=torch.uint8))
        self.graphs[b].replay()
        self.done[b].record()
        o.t = t


class ShardListAdamW:
    """LocalShardAdamW over per-tensor shard buffers instead of arenas.

    ``master``, ``exp_avg``, ``exp_avg_sq``, ``grad`` and ``weight_bf16`` are lists of
    tensors, one per parameter (model order, each exactly its shard's length); pass
    your own (for instance the fp32 state a framework already keeps per parameter) or
    let the constructor allocate zeroed ones.  Micro-batch gradients are lists of bf16
    shard tensors, whose device pointer lists are cached by (address, length, dtype) of every
    tensor, so a loop that reuses the same gradient buffers uploads them once; or a
    PointerLists the caller built once."""

    def __init__(self, numels, no_decay=None, dp_size=1, dp_rank=0, hparams=None, device="cuda", master=None,
                 exp_avg=None, exp_avg_sq=None, grad=None, weight_bf16=None, groups=None, lr_scale=None,
                 wd_scale=None):
        self.device = torch.device(device)
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.plan = Plan(numels, no_decay, dp_size, dp_rank, groups=groups, lr_scale=lr_scale, wd_scale=wd_scale)
        self.hp = hparams if isinstance(hparams, Hparams) else Hparams(**(hparams or {}))
        mk = self.plan.new_shards
        self.master = master if master is not None else mk(torch.float32, self.device)
        self.exp_avg = exp_avg if exp_avg is not None else mk(torch.float32, self.device)
        self.exp_avg_sq = exp_avg_sq if exp_avg_sq is not None else mk(torch.float32, self.device)
        self.grad = grad if grad is not None else mk(torch.float32, self.device)
        self.weight_bf16 = weight_bf16 if weight_bf16 is not None else mk(torch.bfloat16, self.device)
        f32 = torch.float32
        self._lists = {name: PointerLists(self.plan, getattr(self, name), f32, self.device)
                       for name in ("master", "exp_avg", "exp_avg_sq", "grad")}
        self._lists["weight_bf16"] = PointerLists(self.plan, self.weight_bf16, torch.bfloat16, self.device)
        self.table = self.plan.list_table(self.device)
        self.workspace = self.plan.new_list_workspace(self.device)
        self.norm_out = new_norm_out(self.device)
        self._micro_cache = {}
        self.t = 0
        self._micro_seen = 0
        self._norm_ready = False

    def _micro_lists(self, micro, stream=None):
        if isinstance(micro, PointerLists):
            return micro
        if len(micro) and isinstance(micro[0], torch.Tensor):
            micro = [micro]
        # A cached upload stays valid for tensors at the same addresses with the same lengths
        # and dtype (what the upload checked); it keeps no reference to them.  It was ordered on
        # the stream the kernels then ran on, so the key holds the stream as well.
        key = (_stream_ptr(stream, self.device),) + tuple(
            tuple((t.data_ptr(), t.numel(), t.dtype) for t in lst) for lst in micro)
        pl = self._micro_cache.get(key)
        if pl is None:
            if len(self._micro_cache) >= 8:
                self._micro_cache.clear()
            pl = self._micro_cache[key] = PointerLists(self.plan, micro, torch.bfloat16, self.device, stream=stream,
                                                       keep=False)
        return pl

    def accumulate(self, micro, last=False, extra_sumsq=0.0, divisor=1.0, stream=None):
        """Add one micro-batch (a list of bf16 shard tensors), several (a list of such lists), or
        a PointerLists built for them once (no per-call host work)."""
        pl = self._micro_lists(micro, stream)
        first = self._micro_seen == 0
        if last:
            list_accumulate_norm(self.plan, self.table, self._lists["grad"], pl, self.workspace, self.norm_out,
                                 overwrite_first=first, extra_sumsq=extra_sumsq, divisor=divisor, stream=stream)
        else:
            list_accumulate(self.plan, self.table, self._lists["grad"], pl, overwrite_first=first, stream=stream)
        self._micro_seen += pl.n_lists
        self._norm_ready = bool(last)

    def step(self, extra_sumsq=0.0, lr=None, group=None, stream=None, check_finite=False):
        """Norm (unless the last accumulate took it) + optional all-reduce of sumsq + clip +
        AdamW + bf16 copy; ``check_finite`` as for LocalShardAdamW.step."""
        if not self._norm_ready:
            list_grad_norm(self.plan, self.table, self._lists["grad"], self.workspace, self.norm_out, extra_sumsq,
                           stream=stream)
        self._norm_ready = False
        if group is not None:
            allreduce_sumsq_(self.norm_out, group, stream=stream)
        self.t += 1
        hp = self.hp if lr is None else dataclasses.replace(self.hp, lr=lr)
        L = self._lists
        list_step(self.plan, self.table, L["master"], L["exp_avg"], L["exp_avg_sq"], L["grad"], L["weight_bf16"],
                  hp, self.t, self.norm_out, stream=stream)
        self._micro_seen = 0
        return _applied(self, stream) if check_finite else None

    def step_from(self, micro, extra_sumsq=0.0, divisor=1.0, lr=None, group=None, stream=None, check_finite=False):
        """The whole step from micro-batch gradients that are all resident (as for accumulate):
        for one micro-batch, the norm from the micro-batch and the step that writes the gradient
        (34 bytes per element instead of 36); for several, the K-way accumulation with the norm,
        then the step.  The same result as accumulate(micro, last=True) then step(); ``group``
        all-reduces the sum of squares in between."""
        pl = self._micro_lists(micro, stream)
        L = self._lists
        hp = self.hp if lr is None else dataclasses.replace(self.hp, lr=lr)
        if pl.n_lists == 1:
            list_micro_norm(self.plan, self.table, pl, self.workspace, self.norm_out, extra_sumsq, divisor,
                            stream=stream)
        else:
            list_accumulate_norm(self.plan, self.table, L["grad"], pl, self.workspace, self.norm_out,
                                 overwrite_first=True, extra_sumsq=extra_sumsq, divisor=divisor, stream=stream)
        if group is not None:
            allreduce_sumsq_(self.norm_out, group, stream=stream)
        self.t += 1
        if pl.n_lists == 1:
            list_step_accumulate(self.plan, self.table, L["master"], L["exp_avg"], L["exp_avg_sq"], L["grad"], pl,
                                 L["weight_bf16"], hp, self.t, self.norm_out, divisor=divisor, stream=stream)
        else:
            list_step(self.plan, self.table, L["master"], L["exp_avg"], L["exp_avg_sq"], L["grad"], L["weight_bf16"],
                      hp, self.t, self.norm_out, stream=stream)
        self._micro_seen = 0
        self._norm_ready = False
        return _applied(self, stream) if check_finite else None

    def read_norm(self, stream=None):
        return read_norm(self.norm_out, stream=stream)

    @property
    def pointer_lists(self):
        """The device pointer lists of the state buffers: "master", "exp_avg", "exp_avg_sq",
        "grad" and "weight_bf16" (PointerLists), for calling the list functions directly."""
        return dict(self._lists)

    def save_checkpoint(self, path, meta=None, async_=False):
        """Write this rank's master / m / v shards and the step count (see ``checkpoint``)."""
        from . import checkpoint
        fn = checkpoint.save_async if async_ else checkpoint.save
        return fn(path, self.plan, self.master, self.exp_avg, self.exp_avg_sq, self.t, meta)

    def load_checkpoint(self, path):
        """Fill the master / m / v shards from a checkpoint written at any dp size (in either
        layout); restores the step count."""
        from . import checkpoint
        self.t = checkpoint.load(path, self.plan, self.master, self.exp_avg, self.exp_avg_sq)
        self._micro_seen = 0
        self._norm_ready = False
        return self.t


def default_no_decay(name, p):
    """Norm weights and biases (1-D parameters) are excluded from weight decay."""
    return p.dim() < 2


class Zero1AdamW:
    """Fused ZeRO-1 AdamW over ``named_params`` (an iterable of (name, parameter)).

    The parameters must be bf16 and contiguous; their gradients must be bf16 too.
    ``accumulate()`` adds the current ``p.grad`` of every parameter into the fp32
    accumulator (call it after each micro-batch's backward, then zero the grads);
    ``step()`` takes the last micro-batch from ``p.grad`` itself if ``accumulate``
    was not called since the previous step, then clips, steps and writes the bf16
    weights into the model."""

    def __init__(self, named_params, hparams=None, dp_size=1, dp_rank=0, no_decay=default_no_decay, device=None):
        self.named = [(n, p) for n, p in named_params if p.requires_grad]
        if not self.named:
            raise ValueError("no parameters to optimize")
        for n, p in self.named:
            if p.dtype != torch.bfloat16 or not p.is_contiguous() or p.device.type != "cuda":
                raise ValueError("parameter %s must be a contiguous bf16 CUDA tensor" % n)
        self.device = torch.device(device) if device is not None else self.named[0][1].device
        numels = [p.numel() for _, p in self.named]
        flags = [1 if no_decay(n, p) else 0 for n, p in self.named]
        plan = Plan(numels, flags, dp_size, dp_rank)
        L = plan.layout()
        self._slices = [(int(s), int(c)) for s, c in zip(L.shard_start, L.counts)]
        master = [p.data.view(-1)[s:s + c].float().contiguous() for (_, p), (s, c) in zip(self.named, self._slices)]
        weights = [p.data.view(-1)[s:s + c] for (_, p), (s, c) in zip(self.named, self._slices)]
        self.opt = ShardListAdamW(numels, flags, dp_size, dp_rank, hparams=hparams, device=self.device,
                                  master=master, weight_bf16=weights)
        self.no_decay = flags
        self._pending = 0
        self._grad_ident = None
        self._grad_pl = None

    @property
    def hparams(self) -> Hparams:
        return self.opt.hp

    @property
    def t(self):
        return self.opt.t

    def _grad_lists(self, stream=None):
        """Device pointer lists of every parameter's gradient slice.  Slicing thousands of
        gradients costs the host milliseconds per call, so the lists are reused while every
        p.grad is the same tensor at the same address."""
        grads = [p.grad for _, p in self.named]
        ident = [(id(g), g.data_ptr() if g is not None else 0) for g in grads]
        ident.append(_stream_ptr(stream, self.device))  # the stream the lists were uploaded on
        if ident == self._grad_ident and self._grad_pl is not None:
            return self._grad_pl
        views = []
        for (n, p), g, (s, c) in zip(self.named, grads, self._slices):
            if g is None:
                raise ValueError("parameter %s has no gradient" % n)
            if g.dtype != torch.bfloat16 or not g.is_contiguous():
                raise ValueError("gradient of %s must be contiguous bf16" % n)
            views.append(g.view(-1)[s:s + c])
        # no reference kept: the identity check above decides whether the addresses still hold
        self._grad_pl = PointerLists(self.opt.plan, views, torch.bfloat16, self.device, stream=stream, keep=False)
        self._grad_ident = ident
        return self._grad_pl

    def accumulate(self, last=False, stream=None):
        """Add every parameter's current bf16 gradient slice into the fp32 accumulator."""
        self.opt.accumulate(self._grad_lists(stream), last=last, stream=stream)
        self._pending += 1

    def step(self, lr=None, group=None, stream=None, check_finite=False):
        """Clip + AdamW on this rank's slices; the bf16 weights land in the model's parameters.
        ``group``: a torch.distributed group whose ranks' sums of squares make the global norm;
        ``check_finite`` as for LocalShardAdamW.step."""
        if self._pending == 0:  # one micro-batch: its norm, then the step that fills the accumulator
            applied = self.opt.step_from(self._grad_lists(stream), lr=lr, group=group, stream=stream,
                                         check_finite=check_finite)
        else:
            applied = self.opt.step(lr=lr, group=group, stream=stream, check_finite=check_finite)
        self._pending = 0
        return applied

    def read_norm(self, stream=None):
        """The last step's gradient norm record (synchronises)."""
        return self.opt.read_norm(stream=stream)

    def save_checkpoint(self, path, meta=None, async_=False):
        meta = dict(meta or {})
        meta.setdefault("names", [n for n, _ in self.named])
        return self.opt.save_checkpoint(path, meta=meta, async_=async_)

    def load_checkpoint(self, path):
        """Restore master / m / v and the step count, and write the restored master's bf16
        rounding into the model's parameter slices."""
        t = self.opt.load_checkpoint(path)
        with torch.no_grad():
            for w, m in zip(self.opt.weight_bf16, self.opt.master):
                if w.numel():
                    w.copy_(m.to(torch.bfloat16))
        return t
