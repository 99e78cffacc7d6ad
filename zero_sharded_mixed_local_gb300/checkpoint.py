"""Checkpoint of the sharded optimizer state, readable at any data-parallel size.

The state is stored in model layout: each of master, exp_avg (m) and
exp_avg_sq (v) is one raw little-endian fp32 file holding every parameter
whole, concatenated in model order (tensor i at element offset
sum(numels[:i])), plus ``meta.json`` (tensor sizes, step count, optional
names, hyper-parameters and groups).  A rank writes only its own shard runs,
with positional writes into files sized up front, so all ranks of a job can
save concurrently without any collective; a rank of a job with another
dp_size reads back its own shard runs of the same files.  This is the
resharding-on-load that TorchTitan's distributed checkpointing provides
("TorchTitan 生产级预训练方案", section 2.3.1), done here for the ZeRO-1 shard
plan.

``save_async`` copies the arenas to host memory before returning (training
may go on changing them) and writes the files in a background thread, the
asynchronous checkpointing the same section describes.

Each quantity is given either as an arena (one padded fp32 tensor laid out by
the plan) or as a list of per-tensor shard tensors in model order (the form
the tensor-list calls step); the files are the same either way.
"""
import concurrent.futures
import json
import os
import sys

import numpy as np
import torch

FORMAT = "zero1-optimizer-shards-model-layout-v1"
QUANTITIES = ("master", "exp_avg", "exp_avg_sq")
_executor = concurrent.futures.ThreadPoolExecutor(max_workers=2, thread_name_prefix="zero1-ckpt")


def _numels(plan):
    """Per-tensor total numels (the whole tensors, all ranks)."""
    return plan.numels


def _runs(plan):
    """(model element offset, arena offset, count) of every non-empty shard run."""
    L = plan.layout()
    numels = np.asarray(_numels(plan), np.int64)
    model_off = np.concatenate([[0], np.cumsum(numels)[:-1]]) if len(numels) else numels
    return [(int(model_off[i] + L.shard_start[i]), int(L.offsets[i]), int(L.counts[i]))
            for i in range(len(numels)) if L.counts[i]]


def _host_copy(plan, x):
    """Host fp32 array in arena layout from an arena tensor or a list of shard tensors."""
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.float32:
            raise TypeError("optimizer state arenas are fp32")
        t = x.detach()
        return t.cpu().numpy() if t.device.type != "cpu" else t.numpy().copy()
    L = plan.layout()
    shards = list(x)
    if len(shards) != len(L.counts):
        raise ValueError("%d shard tensors for a plan of %d tensors" % (len(shards), len(L.counts)))
    host = np.zeros(plan.arena_numel, np.float32)
    for i, (t, o, c) in enumerate(zip(shards, L.offsets, L.counts)):
        o, c = int(o), int(c)
        if c == 0:
            continue
        if t.dtype != torch.float32 or t.numel() != c:
            raise ValueError("shard %d must be fp32 with %d elements" % (i, c))
        host[o:o + c] = t.detach().reshape(-1).cpu().numpy()
    return host


def _write(path, plan, snap, step_t, meta):
    total = int(sum(_numels(plan)))
    runs = _runs(plan)
    for q in QUANTITIES:
        fd = os.open(os.path.join(path, q + ".bin"), os.O_RDWR | os.O_CREAT, 0o644)
        try:
            if os.fstat(fd).st_size != 4 * total:
                os.ftruncate(fd, 4 * total)
            host = snap[q]
            for model_off, arena_off, n in runs:
                buf = memoryview(host[arena_off:arena_off + n]).cast("B")
                written = 0
                while written < len(buf):
                    written += os.pwrite(fd, buf[written:], 4 * model_off + written)
            os.fsync(fd)
        finally:
            os.close(fd)
    if plan.dp_rank == 0:
        info = {"format": FORMAT, "numels": [int(n) for n in _numels(plan)], "step": int(step_t),
                "dtype": "float32", "byte_order": "little", "written_by_dp_size": plan.dp_size}
        info.update(meta or {})
        tmp = os.path.join(path, "meta.json.tmp.%d" % os.getpid())
        with open(tmp, "w") as f:
            json.dump(info, f)
        os.replace(tmp, os.path.join(path, "meta.json"))


def save(path, plan, master, exp_avg, exp_avg_sq, step_t, meta=None):
    """Write this rank's shard of master, m and v into the checkpoint at ``path``.

    Every rank of the job calls it with its own plan; rank 0 also writes
    meta.json.  ``meta`` adds entries (names, hyper-parameters, ...)."""
    if sys.byteorder != "little":  # pragma: no cover - every supported host is little-endian
        raise RuntimeError("little-endian host expected")
    os.makedirs(path, exist_ok=True)
    snap = {q: _host_copy(plan, a) for q, a in zip(QUANTITIES, (master, exp_avg, exp_avg_sq))}
    _write(path, plan, snap, step_t, meta)


def save_async(path, plan, master, exp_avg, exp_avg_sq, step_t, meta=None):
    """As save(), but only the device-to-host snapshot happens before returning; the
    files are written in a background thread.  Returns a concurrent.futures.Future."""
    os.makedirs(path, exist_ok=True)
    snap = {q: _host_copy(plan, a) for q, a in zip(QUANTITIES, (master, exp_avg, exp_avg_sq))}
    return _executor.submit(_write, path, plan, snap, step_t, meta)


def read_meta(path):
    with open(os.path.join(path, "meta.json")) as f:
        info = json.load(f)
    if info.get("format") != FORMAT:
        raise ValueError("not a %s checkpoint: %s" % (FORMAT, path))
    return info


def load(path, plan, master, exp_avg, exp_avg_sq):
    """Fill this rank's arenas or shard lists (any dp_size) from the checkpoint; returns its
    step count.  Arena padding elements are set to zero."""
    info = read_meta(path)
    if [int(n) for n in info["numels"]] != [int(n) for n in _numels(plan)]:
        raise ValueError("checkpoint tensor sizes do not match the plan")
    runs = _runs(plan)
    L = plan.layout()
    for q, arena in zip(QUANTITIES, (master, exp_avg, exp_avg_sq)):
        if isinstance(arena, torch.Tensor):
            if arena.dtype != torch.float32 or arena.numel() != plan.arena_numel:
                raise ValueError("%s arena must be fp32 with %d elements" % (q, plan.arena_numel))
        else:
            arena = list(arena)
            if len(arena) != len(L.counts) or any(
                    int(c) and (t.dtype != torch.float32 or t.numel() != int(c)) for t, c in zip(arena, L.counts)):
                raise ValueError("%s shards must be fp32 tensors of the plan's shard sizes" % q)
        host = np.zeros(plan.arena_numel, np.float32)
        fd = os.open(os.path.join(path, q + ".bin"), os.O_RDONLY)
        try:
            for model_off, arena_off, n in runs:
                view = memoryview(host[arena_off:arena_off + n]).cast("B")
                got = 0
                while got < len(view):
                    k = os.preadv(fd, [view[got:]], 4 * model_off + got)
                    if k <= 0:
                        raise IOError("checkpoint file %s is short" % q)
                    got += k
        finally:
            os.close(fd)
        if isinstance(arena, torch.Tensor):
            arena.copy_(torch.from_numpy(host))
        else:
            for t, o, c in zip(arena, L.offsets, L.counts):
                if int(c):
                    t.copy_(torch.from_numpy(host[int(o):int(o) + int(c)]).view_as(t))
    return int(info["step"])

