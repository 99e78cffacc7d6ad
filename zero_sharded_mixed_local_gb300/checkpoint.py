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

State on the GPU is copied through page-locked host buffers: one copy per
arena (or per shard) on the current stream and one synchronisation, at the
speed of the CPU-GPU link rather than of pageable staging.  The buffers are
kept for the next checkpoint (pinning many GB costs more than the copy), at
most one set per arena size while no save is in flight; ``prepare_staging()``
pins them ahead of the first checkpoint and ``release_staging()`` frees them.

Each quantity is given either as an arena (one padded fp32 tensor laid out by
the plan) or as a list of per-tensor shard tensors in model order (the form
the tensor-list calls step); the files are the same either way.
"""
import concurrent.futures
import json
import os
import sys
import threading

import numpy as np
import torch

FORMAT = "zero1-optimizer-shards-model-layout-v1"
QUANTITIES = ("master", "exp_avg", "exp_avg_sq")
_executor = concurrent.futures.ThreadPoolExecutor(max_workers=2, thread_name_prefix="zero1-ckpt")


class _StagingPool:
    """Page-locked fp32 host buffers by length, reused across checkpoints."""

    def __init__(self):
        self._lock = threading.Lock()
        self._free = {}

    def take(self, n):
        with self._lock:
            bufs = self._free.get(n)
            if bufs:
                return bufs.pop()
        return torch.empty(n, dtype=torch.float32, pin_memory=True)

    def give(self, buf):
        with self._lock:
            bufs = self._free.setdefault(buf.numel(), [])
            if len(bufs) < len(QUANTITIES):  # one checkpoint's worth per size
                bufs.append(buf)

    def clear(self):
        with self._lock:
            self._free.clear()


_staging = _StagingPool()


def prepare_staging(plan):
    """Pin one checkpoint's worth of staging buffers for ``plan`` now (at start-up, say), so the
    first snapshot does not pay for pinning.  Needs CUDA."""
    bufs = [_staging.take(plan.arena_numel) for _ in QUANTITIES]
    for b in bufs:
        _staging.give(b)


def release_staging():
    """Free the page-locked buffers kept for later checkpoints."""
    _staging.clear()


def _on_gpu(x):
    if isinstance(x, torch.Tensor):
        return x.device.type == "cuda"
    return any(isinstance(t, torch.Tensor) and t.device.type == "cuda" for t in x)


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


def _check_state(plan, x, name):
    """An fp32 arena of the plan, or a list of fp32 shard tensors of its shard sizes; returns the list
    form's shards (None for an arena)."""
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.float32 or x.numel() != plan.arena_numel:
            raise ValueError("%s arena must be fp32 with %d elements" % (name, plan.arena_numel))
        return None
    L = plan.layout()
    shards = list(x)
    if len(shards) != len(L.counts):
        raise ValueError("%s: %d shard tensors for a plan of %d tensors" % (name, len(shards), len(L.counts)))
    for i, (t, c) in enumerate(zip(shards, L.counts)):
        if int(c) and (t.dtype != torch.float32 or t.numel() != int(c)):
            raise ValueError("%s shard %d must be fp32 with %d elements" % (name, i, int(c)))
    return shards


def _snapshot(plan, states):
    """Host copies, in arena layout, of the named states (arenas or shard lists).  Returns
    ({name: numpy array}, [page-locked buffers to give back once written])."""
    L = plan.layout()
    snap, staged = {}, []
    gpu = any(_on_gpu(x) for x in states.values())
    checked = {name: _check_state(plan, x, name) for name, x in states.items()}  # before any copy
    for name, x in states.items():
        shards = checked[name]
        if gpu:
            buf = _staging.take(plan.arena_numel)
            staged.append(buf)
            if shards is None:
                buf.copy_(x.detach(), non_blocking=True)
            else:
                for t, o, c in zip(shards, L.offsets, L.counts):
                    if int(c):
                        buf[int(o):int(o) + int(c)].copy_(t.detach().reshape(-1), non_blocking=True)
            snap[name] = buf.numpy()
        elif shards is None:
            snap[name] = x.detach().numpy().copy()
        else:
            host = np.zeros(plan.arena_numel, np.float32)
            for t, o, c in zip(shards, L.offsets, L.counts):
                if int(c):
                    host[int(o):int(o) + int(c)] = t.detach().reshape(-1).numpy()
            snap[name] = host
    if gpu:  # the copies were queued behind the work already on the stream
        torch.cuda.current_stream().synchronize()
    return snap, staged


def _write_file(path, q, host, runs, total):
    fd = os.open(os.path.join(path, q + ".bin"), os.O_RDWR | os.O_CREAT, 0o644)
    try:
        if os.fstat(fd).st_size != 4 * total:
            os.ftruncate(fd, 4 * total)
        for model_off, arena_off, n in runs:
            buf = memoryview(host[arena_off:arena_off + n]).cast("B")
            written = 0
            while written < len(buf):
                written += os.pwrite(fd, buf[written:], 4 * model_off + written)
        os.fsync(fd)
    finally:
        os.close(fd)


def _write(path, plan, snap, step_t, meta):
    total = int(sum(_numels(plan)))
    runs = _runs(plan)
    # one thread per file: the writes and fsyncs release the GIL and keep the disk's queue fuller
    with concurrent.futures.ThreadPoolExecutor(len(QUANTITIES)) as ex:
        for f in [ex.submit(_write_file, path, q, snap[q], runs, total) for q in QUANTITIES]:
            f.result()
    if plan.dp_rank == 0:
        info = {"format": FORMAT, "numels": [int(n) for n in _numels(plan)], "step": int(step_t),
                "dtype": "float32", "byte_order": "little", "written_by_dp_size": plan.dp_size}
        info.update(meta or {})
        tmp = os.path.join(path, "meta.json.tmp.%d" % os.getpid())
        with open(tmp, "w") as f:
            json.dump(info, f)
        os.replace(tmp, os.path.join(path, "meta.json"))


def _write_and_release(path, plan, snap, step_t, meta, staged):
    try:
        _write(path, plan, snap, step_t, meta)
    finally:
        for b in staged:
            _staging.give(b)


def save(path, plan, master, exp_avg, exp_avg_sq, step_t, meta=None):
    """Write this rank's shard of master, m and v into the checkpoint at ``path``.

    Every rank of the job calls it with its own plan; rank 0 also writes
    meta.json.  ``meta`` adds entries (names, hyper-parameters, ...).  The
    state is read in the order of the current CUDA stream."""
    if sys.byteorder != "little":  # pragma: no cover - every supported host is little-endian
        raise RuntimeError("little-endian host expected")
    os.makedirs(path, exist_ok=True)
    snap, staged = _snapshot(plan, dict(zip(QUANTITIES, (master, exp_avg, exp_avg_sq))))
    _write_and_release(path, plan, snap, step_t, meta, staged)


def save_async(path, plan, master, exp_avg, exp_avg_sq, step_t, meta=None):
    """As save(), but only the device-to-host snapshot happens before returning; the
    files are written in a background thread.  Returns a concurrent.futures.Future."""
    if sys.byteorder != "little":  # pragma: no cover
        raise RuntimeError("little-endian host expected")
    os.makedirs(path, exist_ok=True)
    snap, staged = _snapshot(plan, dict(zip(QUANTITIES, (master, exp_avg, exp_avg_sq))))
    return _executor.submit(_write_and_release, path, plan, snap, step_t, meta, staged)


def read_meta(path):
    with open(os.path.join(path, "meta.json")) as f:
        info = json.load(f)
    if info.get("format") != FORMAT:
        raise ValueError("not a %s checkpoint: %s" % (FORMAT, path))
    return info


def _read_file(path, q, host, runs):
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


def load(path, plan, master, exp_avg, exp_avg_sq):
    """Fill this rank's arenas or shard lists (any dp_size) from the checkpoint; returns its
    step count.  Arena padding elements are set to zero.  GPU state is filled through
    page-locked buffers, in the order of the current CUDA stream, and the call returns once
    the copies are done."""
    info = read_meta(path)
    if [int(n) for n in info["numels"]] != [int(n) for n in _numels(plan)]:
        raise ValueError("checkpoint tensor sizes do not match the plan")
    runs = _runs(plan)
    L = plan.layout()
    states = dict(zip(QUANTITIES, (master, exp_avg, exp_avg_sq)))
    shards = {q: _check_state(plan, x, q) for q, x in states.items()}
    gpu = {q: _on_gpu(x) for q, x in states.items()}
    staged, hosts = [], {}
    try:
        for q in QUANTITIES:
            if gpu[q]:
                buf = _staging.take(plan.arena_numel)
                staged.append(buf)
                host = buf.numpy()
                pos = 0  # a reused buffer: zero what the runs leave out (the arena padding)
                for arena_off, n in sorted((a, n) for _, a, n in runs):
                    host[pos:arena_off] = 0.0
                    pos = arena_off + n
                host[pos:] = 0.0
                hosts[q] = (buf, host)
            else:
                host = np.zeros(plan.arena_numel, np.float32)
                hosts[q] = (torch.from_numpy(host), host)
        with concurrent.futures.ThreadPoolExecutor(len(QUANTITIES)) as ex:  # one reader per file
            for f in [ex.submit(_read_file, path, q, hosts[q][1], runs) for q in QUANTITIES]:
                f.result()
        for q in QUANTITIES:
            src = hosts[q][0]
            if shards[q] is None:
                states[q].copy_(src, non_blocking=gpu[q])
            else:
                for t, o, c in zip(shards[q], L.offsets, L.counts):
                    if int(c):
                        t.copy_(src[int(o):int(o) + int(c)].view_as(t), non_blocking=gpu[q])
    finally:
        if staged:  # the buffers are reused: the copies out of them must be done
            torch.cuda.current_stream().synchronize()
        for b in staged:
            _staging.give(b)
    return int(info["step"])
