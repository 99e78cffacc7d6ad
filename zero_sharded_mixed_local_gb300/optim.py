"""A ZeRO-1 AdamW over a torch module's parameters, on top of the tensor-list calls.

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
import torch

from .binding import Hparams, Plan, ShardListAdamW


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

    @property
    def hparams(self) -> Hparams:
        return self.opt.hp

    @property
    def t(self):
        return self.opt.t

    def _grad_views(self):
        views = []
        for (n, p), (s, c) in zip(self.named, self._slices):
            g = p.grad
            if g is None:
                raise ValueError("parameter %s has no gradient" % n)
            if g.dtype != torch.bfloat16 or not g.is_contiguous():
                raise ValueError("gradient of %s must be contiguous bf16" % n)
            views.append(g.view(-1)[s:s + c])
        return views

    def accumulate(self, last=False, stream=None):
        """Add every parameter's current bf16 gradient slice into the fp32 accumulator."""
        self.opt.accumulate(self._grad_views(), last=last, stream=stream)
        self._pending += 1

    def step(self, lr=None, group=None, stream=None):
        """Clip + AdamW on this rank's slices; the bf16 weights land in the model's parameters.
        ``group``: a torch.distributed group whose ranks' sums of squares make the global norm."""
        if self._pending == 0:
            self.opt.accumulate(self._grad_views(), last=True, stream=stream)
        self.opt.step(lr=lr, group=group, stream=stream)
        self._pending = 0

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
