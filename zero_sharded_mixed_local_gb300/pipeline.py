"""Host-fed local steps: micro-batch gradients arrive from pinned host memory.

A training loop whose gradients are produced away from the optimizer's GPU
(another device, a host-side reducer, a data loader of precomputed gradients)
feeds the local ZeRO-1 step from host memory.  ``HostFedSteps`` runs that loop
with the transfer hidden behind the kernels:

- every step's K micro-batch gradients (bf16 arenas in pinned host memory) are
  copied to the device by the copy engines on a side stream, into one of two
  staging sets, so step t+1's transfer (bound by the CPU-GPU link) overlaps step
  t's kernels (bound by HBM);
- on the step stream, the step waits for its own copy (an event), then runs the
  path as a training loop does: K-1 ``accumulate`` calls, ``accumulate_norm`` for
  the last micro-batch (or one K-way ``accumulate_norm``), the optional all-reduce
  of the sum of squares, and ``step``; with one micro-batch, ``micro_norm`` and
  ``step_accumulate`` (the same results, 34 bytes per element instead of 36);
  each kernel launched as a programmatic dependent of the previous one;
- every step's 24-byte norm record is copied back to pinned host memory on the
  step stream and read on the host one step behind, as a loop logs it.

Two gradient arenas, workspaces and norm records alternate with the staging
sets, so the copy for step t+1 never writes a buffer step t still reads, and the
side stream reuses staging set i only after the step that last read it (t-2)
is done.  The arithmetic is that of the synchronous calls, in the same order
("ZeRO-1 风格的 Distributed Optimizer", section 6.7: accumulate every
micro-batch, then the reduction and the step).
"""
import torch

from .binding import (NORM_OUT_BYTES, accumulate, accumulate_norm, allreduce_sumsq_, decode_norm, micro_norm,
                      new_norm_out, step, step_accumulate)


class HostFedSteps:
    """Host-fed local steps over one rank's arenas.

    ``master``, ``exp_avg``, ``exp_avg_sq`` and ``weight_bf16`` are the rank's state
    arenas (updated in place); ``t`` is the number of steps already taken.  Slot 0
    of the double buffering may reuse buffers the caller already holds
    (``stage0``: K bf16 arenas, ``grad0``, ``workspace0``, ``norm_out0``); the rest
    is allocated here.  ``k_way`` accumulates all K micro-batches in one pass;
    ``group`` all-reduces each step's sum of squares over a process group."""

    def __init__(self, plan, master, exp_avg, exp_avg_sq, weight_bf16, hparams, micro_batches, t=0, k_way=False,
                 group=None, stream=None, stage0=None, grad0=None, workspace0=None, norm_out0=None):
        self.plan, self.hp, self.K = plan, hparams, int(micro_batches)
        self.master, self.exp_avg, self.exp_avg_sq, self.weight_bf16 = master, exp_avg, exp_avg_sq, weight_bf16
        self.t, self.k_way, self.group = int(t), bool(k_way), group
        dev = self.device = master.device
        self.stream = stream if stream is not None else torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(dev)
        mk = plan.new_arena
        self.stage = [list(stage0) if stage0 is not None else [mk(torch.bfloat16, dev) for _ in range(self.K)],
                      [mk(torch.bfloat16, dev) for _ in range(self.K)]]
        if any(len(s) != self.K for s in self.stage):
            raise ValueError("stage0 must hold %d micro-batch arenas" % self.K)
        self.grads = [grad0 if grad0 is not None else mk(torch.float32, dev), mk(torch.float32, dev)]
        self.workspaces = [workspace0 if workspace0 is not None else plan.new_workspace(dev),
                           plan.new_workspace(dev)]
        self.norm_outs = [norm_out0 if norm_out0 is not None else new_norm_out(dev), new_norm_out(dev)]
        self.host_records = [torch.empty(32, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.copied = [torch.cuda.Event(), torch.cuda.Event()]
        self.step_done = [torch.cuda.Event(), torch.cuda.Event()]
        self.copy_times = []   # (start, end) timing events of each step's host copy, when asked for
        self._n = 0            # steps run through this object: selects the slot

    def run(self, host_micros, n_steps, first_event=None, time_copies=False):
        """Run ``n_steps`` local steps and return their norm records (dicts), in order.

        ``host_micros`` is a list of K pinned host bf16 arenas used for every step, or a
        callable ``f(i)`` returning step i's list (i counts from 0 within this call).
        Copies read those buffers asynchronously: leave them unchanged until ``run``
        returns.  ``first_event`` (a CUDA event) gates the first copy, e.g. the start
        of a timed region; ``time_copies`` records timing events around each copy
        (``copy_times``)."""
        get = host_micros if callable(host_micros) else (lambda i: host_micros)
        plan, K, stream, side = self.plan, self.K, self.stream, self.side
        records = []
        for i in range(n_steps):
            s = self._n % 2
            micros = list(get(i))
            if len(micros) != K:
                raise ValueError("step %d has %d micro-batch gradients, expected %d" % (i, len(micros), K))
            for k, h in enumerate(micros):
                if h.device.type != "cpu" or not h.is_pinned():
                    raise ValueError("micro-batch %d of step %d must be in pinned host memory" % (k, i))
            with torch.cuda.stream(side):
                if self._n >= 2:
                    side.wait_event(self.step_done[s])  # staging set s is free once step n-2 is done
                if i == 0 and first_event is not None:
                    side.wait_event(first_event)  # later copies follow it on the side stream
                if time_copies:
                    self.copy_times.append((torch.cuda.Event(enable_timing=True),
                                            torch.cuda.Event(enable_timing=True)))
                    self.copy_times[-1][0].record(side)
                for k in range(K):
                    self.stage[s][k].copy_(micros[k], non_blocking=True)
                if time_copies:
                    self.copy_times[-1][1].record(side)
                self.copied[s].record(side)
            stream.wait_event(self.copied[s])
            # the step's kernels, the all-reduce and the record's copy back all in order on `stream`
            # (the binding and the collective take torch's current stream)
            with torch.cuda.stream(stream):
                self._step(s)
                self.host_records[s].copy_(self.norm_outs[s], non_blocking=True)
            self.step_done[s].record(stream)
            if i >= 1:  # the previous step's record, one step behind
                self.step_done[1 - s].synchronize()
                records.append(decode_norm(self.host_records[1 - s]))
            self._n += 1
        if n_steps:
            last = (self._n - 1) % 2
            self.step_done[last].synchronize()
            records.append(decode_norm(self.host_records[last]))
        return records

    def _step(self, s):
        plan, K, stream = self.plan, self.K, self.stream
        grad, ws, nout, stage = self.grads[s], self.workspaces[s], self.norm_outs[s], self.stage[s]
        if K == 1 and not self.k_way:  # the norm from the micro-batch; the step writes the gradient
            micro_norm(plan, stage[0], ws, nout, stream=stream)
            if self.group is not None:
                allreduce_sumsq_(nout, self.group)
            self.t += 1
            step_accumulate(plan, self.master, self.exp_avg, self.exp_avg_sq, grad, stage[0], self.weight_bf16,
                            self.hp, self.t, nout, stream=stream)
            return
        if self.k_way:
            accumulate_norm(plan, grad, stage, ws, nout, overwrite_first=True, stream=stream)
        else:
            for k in range(K - 1):
                accumulate(plan, grad, stage[k], overwrite_first=(k == 0), stream=stream)
            accumulate_norm(plan, grad, stage[K - 1], ws, nout, overwrite_first=(K == 1), stream=stream)
        if self.group is not None:
            allreduce_sumsq_(nout, self.group)
        self.t += 1
        step(plan, self.master, self.exp_avg, self.exp_avg_sq, grad, self.weight_bf16, self.hp, self.t, nout,
             stream=stream)

    @property
    def h2d_bytes_per_step(self):
        return sum(a.numel() * a.element_size() for a in self.stage[0])

    d2h_bytes_per_step = NORM_OUT_BYTES
