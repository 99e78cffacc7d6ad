"""Optimizer-shard checkpoints (CPU): written by the ranks of one data-parallel
size, read back by the ranks of another.  The expected arenas come from the
shard definition (the oracle's plan) applied to model-layout arrays."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle

NUMELS = [1000, 3, 64, 4097, 11, 0, 257, 1, 16385]
ND = [0, 1, 0, 0, 1, 0, 0, 1, 0]


@pytest.fixture(scope="module")
def z():
    from zero_sharded_mixed_local_gb300 import build
    build.build_library()
    import zero_sharded_mixed_local_gb300 as z
    z.load_library()
    return z


def _full_state(seed=0):
    rng = np.random.default_rng(seed)
    n = sum(NUMELS)
    return {q: rng.standard_normal(n).astype(np.float32) for q in ("master", "exp_avg", "exp_avg_sq")}


def _arena_from_full(plan, full, dp, rank):
    """Rank's arena by the shard definition: tensor i's slice [start, start+count) at its arena offset."""
    start, count, _ = oracle.plan(NUMELS, dp, rank)
    model_off = np.concatenate([[0], np.cumsum(NUMELS)[:-1]])
    L = plan.layout()
    a = np.zeros(plan.arena_numel, np.float32)
    for i in range(len(NUMELS)):
        a[L.offsets[i]:L.offsets[i] + count[i]] = full[model_off[i] + start[i]:model_off[i] + start[i] + count[i]]
    return torch.from_numpy(a)


def _save_all(z, path, full, dp, use_async=False):
    futs = []
    for r in range(dp):
        plan = z.Plan(NUMELS, ND, dp, r)
        arenas = [_arena_from_full(plan, full[q], dp, r) for q in ("master", "exp_avg", "exp_avg_sq")]
        if use_async:
            futs.append(z.checkpoint.save_async(path, plan, *arenas, step_t=7, meta={"note": "test"}))
            for a in arenas:  # training goes on: the snapshot must already have been taken
                a.fill_(-1.0)
        else:
            z.checkpoint.save(path, plan, *arenas, step_t=7, meta={"note": "test"})
    for f in futs:
        f.result()


@pytest.mark.parametrize("dp_save,dp_load,use_async", [(4, 3, False), (1, 8, False), (8, 1, True), (3, 3, True)])
def test_checkpoint_reshards(z, tmp_path, dp_save, dp_load, use_async):
    full = _full_state(dp_save * 10 + dp_load)
    path = str(tmp_path / "ckpt")
    _save_all(z, path, full, dp_save, use_async)
    meta = z.checkpoint.read_meta(path)
    assert meta["step"] == 7 and meta["note"] == "test" and meta["numels"] == NUMELS
    for q in ("master", "exp_avg", "exp_avg_sq"):
        raw = np.fromfile(os.path.join(path, q + ".bin"), dtype="<f4")
        assert np.array_equal(raw, full[q])  # model layout on disk, whole
    for r in range(dp_load):
        plan = z.Plan(NUMELS, ND, dp_load, r)
        arenas = [torch.full((plan.arena_numel,), 5.0) for _ in range(3)]
        assert z.checkpoint.load(path, plan, *arenas) == 7
        for q, a in zip(("master", "exp_avg", "exp_avg_sq"), arenas):
            assert torch.equal(a, _arena_from_full(plan, full[q], dp_load, r))  # padding zeroed too


def test_checkpoint_rejects_a_different_model(z, tmp_path):
    path = str(tmp_path / "ckpt")
    _save_all(z, path, _full_state(), 2)
    other = z.Plan(NUMELS[:-1] + [16384], ND, 2, 0)
    arenas = [torch.zeros(other.arena_numel) for _ in range(3)]
    with pytest.raises(ValueError):
        z.checkpoint.load(path, other, *arenas)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_saves(rank, world, port, path, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import zero_sharded_mixed_local_gb300 as z
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        full = _full_state(99)
        plan = z.Plan(NUMELS, ND, world, rank)
        arenas = [_arena_from_full(plan, full[k], world, rank) for k in ("master", "exp_avg", "exp_avg_sq")]
        dist.barrier()
        z.checkpoint.save(path, plan, *arenas, step_t=3)
        dist.barrier()
        q.put((rank, "ok"))
    finally:
        dist.destroy_process_group()


def test_ranks_save_concurrently_with_gloo(z, tmp_path):
    """Two processes write their shards into the same files at once; one rank reads it all back."""
    path = str(tmp_path / "ckpt")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_saves, args=(r, 2, port, path, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, "ok"), (1, "ok")]
    full = _full_state(99)
    plan = z.Plan(NUMELS, ND, 1, 0)
    arenas = [torch.zeros(plan.arena_numel) for _ in range(3)]
    assert z.checkpoint.load(path, plan, *arenas) == 3
    for k, a in zip(("master", "exp_avg", "exp_avg_sq"), arenas):
        assert torch.equal(a, _arena_from_full(plan, full[k], 1, 0))


def test_checkpoint_from_and_into_shard_lists(z, tmp_path):
    """Per-tensor shard lists (the tensor-list form) save the same files as arenas and load
    back at another dp size, in either form."""
    full = _full_state(42)
    path = str(tmp_path / "ckpt")
    model_off = np.concatenate([[0], np.cumsum(NUMELS)[:-1]])

    def shards(plan, dp, r, q):
        start, count, _ = oracle.plan(NUMELS, dp, r)
        return [torch.from_numpy(full[q][model_off[i] + start[i]:model_off[i] + start[i] + count[i]].copy())
                for i in range(len(NUMELS))]

    for r in range(3):
        plan = z.Plan(NUMELS, ND, 3, r)
        z.checkpoint.save(path, plan, *[shards(plan, 3, r, q) for q in ("master", "exp_avg", "exp_avg_sq")], step_t=9)
    for q in ("master", "exp_avg", "exp_avg_sq"):
        assert np.array_equal(np.fromfile(os.path.join(path, q + ".bin"), dtype="<f4"), full[q])
    for r in range(5):
        plan = z.Plan(NUMELS, ND, 5, r)
        lists = [[torch.full((int(c),), 5.0) for c in plan.layout().counts] for _ in range(3)]
        assert z.checkpoint.load(path, plan, *lists) == 9
        for q, lst in zip(("master", "exp_avg", "exp_avg_sq"), lists):
            for a, b in zip(lst, shards(plan, 5, r, q)):
                assert torch.equal(a, b)
        arenas = [torch.full((plan.arena_numel,), 5.0) for _ in range(3)]
        z.checkpoint.load(path, plan, *arenas)
        for q, a in zip(("master", "exp_avg", "exp_avg_sq"), arenas):
            assert torch.equal(a, _arena_from_full(plan, full[q], 5, r))
    plan = z.Plan(NUMELS, ND, 5, 0)
    bad = [torch.zeros(int(c) + 1) for c in plan.layout().counts]
    with pytest.raises(ValueError):
        z.checkpoint.load(path, plan, bad, bad, bad)
