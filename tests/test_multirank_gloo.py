"""The step's one exchange across data-parallel ranks, on CPU with gloo.

Two processes each hold one shard (dp_size 2) of a small parameter list.
Each computes its local sum of squares into a norm record, the ranks sum the
record's ``sumsq`` field in place with the binding's allreduce_sumsq_ (the
call a multi-GPU job makes between zero1_grad_norm and zero1_step), and each
then steps its shard with the global clip coefficient.  The gathered shards
must equal the unsharded step bit for bit, and a NaN on one rank must make
both ranks skip.  The per-rank arithmetic is the oracle's (this runs without
a GPU); what is under test is the exchange and the rank bookkeeping.
"""
import os
import socket
import struct

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
NUMELS = [1000, 3, 64, 4097, 11, 257, 1]
NO_DECAY = [0, 1, 0, 0, 1, 0, 1]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem(seed=0, nan_rank=None):
    rng = np.random.default_rng(seed)
    N = sum(NUMELS)
    micros = [torch.from_numpy(rng.standard_normal(N).astype(np.float32) * 0.3).to(torch.bfloat16)
              .view(torch.int16).numpy().view(np.uint16) for _ in range(2)]
    p0 = (rng.standard_normal(N) * 0.02).astype(np.float32)
    return micros, p0


def _shard_index(dp, rank):
    import oracle
    start, count, _ = oracle.plan(NUMELS, dp, rank)
    tstart = np.concatenate([[0], np.cumsum(NUMELS)[:-1]])
    idx = np.concatenate([np.arange(tstart[i] + start[i], tstart[i] + start[i] + count[i])
                          for i in range(len(NUMELS))]).astype(np.int64)
    return count, idx


def _worker(rank, world, port, nan_rank, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import oracle
    from zero_sharded_mixed_local_gb300.binding import allreduce_sumsq_, decode_norm

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        micros, p0 = _problem()
        count, idx = _shard_index(world, rank)
        mic = [m[idx].copy() for m in micros]
        if rank == nan_rank:
            mic[0][3] = 0x7FC0
        g = np.zeros(idx.size, np.float32)
        oracle.accumulate_all(g, mic)
        record = torch.zeros(32, dtype=torch.uint8)
        record[:24] = torch.frombuffer(bytearray(struct.pack("<ddii", oracle.sumsq(g), 0.0, 0, 0)), dtype=torch.uint8)
        allreduce_sumsq_(record)
        total = decode_norm(record)["sumsq"]
        ok, norm, coef = oracle.clip_coef(total, 1.0)
        p, m, v, w = p0[idx].copy(), np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32), \
            np.zeros(idx.size, np.uint16)
        if ok:
            oracle.adamw(p, m, v, g, count, np.array(NO_DECAY, np.uint8), HP, 1, coef, w=w)
        q.put((rank, ok, float(coef), idx, p, m, v, w))
    finally:
        dist.destroy_process_group()


def _run(world, nan_rank=None):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, nan_rank, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    return sorted(out, key=lambda x: x[0])


def test_sumsq_allreduce_two_ranks_equals_unsharded_step():
    import oracle
    results = _run(2)
    micros, p0 = _problem()
    N = p0.size
    P, M, V, W = p0.copy(), np.zeros(N, np.float32), np.zeros(N, np.float32), np.zeros(N, np.uint16)
    ref = oracle.full_step(P, M, V, micros, np.array(NUMELS, np.int64), np.array(NO_DECAY, np.uint8), HP, 1,
                           1.0, w=W)
    assert ref["coef"] < 1.0  # clipping active: the global norm matters
    got = [np.zeros(N, np.float32), np.zeros(N, np.float32), np.zeros(N, np.float32), np.zeros(N, np.uint16)]
    for rank, ok, coef, idx, p, m, v, w in results:
        assert ok and np.float32(coef) == ref["coef"]
        for dst, src in zip(got, (p, m, v, w)):
            dst[idx] = src
    for a, b in zip(got, (P, M, V, W)):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_nonfinite_on_one_rank_makes_every_rank_skip():
    results = _run(2, nan_rank=1)
    assert [ok for _, ok, *_ in results] == [False, False]


def _worker_drops_out(rank, world, port, q):
    import sys
    import datetime
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    from zero_sharded_mixed_local_gb300.binding import allreduce_sumsq_

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
    def leave(msg):
        q.put((rank, msg))
        q.close()
        q.join_thread()  # flush the message before the hard exit
        os._exit(0)

    if rank == 1:
        leave("left")  # this rank dies between steps: it never joins the exchange
    record = torch.zeros(32, dtype=torch.uint8)
    try:
        allreduce_sumsq_(record)
        msg = "no error"
    except Exception as e:  # the survivor learns of it instead of hanging
        msg = "error: " + type(e).__name__
    leave(msg)


def test_a_rank_that_drops_out_is_detected_not_waited_for():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_drops_out, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
    assert out[1] == "left"
    assert out[0].startswith("error"), out[0]
