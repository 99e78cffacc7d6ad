"""The whole ZeRO-1 data-parallel step with real collectives (``DataParallelStep``).

Two (or three) processes, one per data-parallel rank, each run the library's kernels on
the one GPU of this machine (independent kernels, nothing waits on the other
process) while a gloo process group carries the collectives over pinned host
copies: the all-to-all of the packed bf16 gradients, the one-double all-reduce
of the sum of squares, and the all-gather of the bf16 weights.  Each rank has
its own K = 2 micro-batch gradients per step.  After three steps:
  - every rank's all-gathered model-layout bf16 weights, and
  - every rank's own master / m / v shard
equal, bit for bit, one unsharded oracle step over all ranks' gradients (added
in fp32 in (micro-batch, rank) order, divided by the world size, clipped with
the global norm).  A NaN in one rank's gradient makes both ranks skip that
step and keep their step count.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)
K, STEPS = 2, 3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _model():
    import sys
    sys.path.insert(0, ROOT)
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    w = get_workload("toy")
    numels = list(w.params.numels) + [13, 3]  # two small tensors: shards of 7/6 and 2/1 elements
    return numels, list(w.params.no_decay) + [0, 1]


def _grad(t, rank, k, total, nan):
    """Rank `rank`'s micro-batch k gradient of step t (model layout, bf16), drawn on the host."""
    g = torch.Generator().manual_seed(1000 * t + 10 * rank + k)
    x = (torch.randn(total, generator=g) * 0.05).to(torch.bfloat16)  # clip active at this size
    if nan:
        x[12345] = float("nan")
    return x


def _master0(total):
    return torch.randn(total, generator=torch.Generator().manual_seed(7)) * 0.02


def _worker(rank, world, port, nan_at, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import zero_sharded_mixed_local_gb300 as z
    from zero_sharded_mixed_local_gb300.exchange import DataParallelStep

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        numels, nd = _model()
        total = sum(numels)
        opt = z.LocalShardAdamW(numels, nd, world, rank, hparams=z.Hparams(**HP))
        z.shard_gather(opt.plan, _master0(total).cuda(), opt.master)
        opt.weight_bf16.copy_(opt.master.to(torch.bfloat16))
        dps = DataParallelStep(opt)
        weights = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        applied = []
        for t in range(1, STEPS + 1):
            micro = [_grad(t, rank, k, total, nan=(t == nan_at and rank == 1 and k == 1)).cuda() for k in range(K)]
            applied.append(dps.step(micro, weights_out=weights, check_finite=True))
        torch.cuda.synchronize()
        out = {}
        for name, a in (("master", opt.master), ("m", opt.exp_avg), ("v", opt.exp_avg_sq)):
            full = torch.full((total,), float("nan"), device="cuda")  # NaN where other ranks own the elements
            z.shard_scatter(opt.plan, a, full)
            out[name] = full.cpu().numpy()
        q.put((rank, applied, opt.t, weights.view(torch.int16).cpu().numpy(), out))
    except Exception as e:  # report, so the parent does not wait for a result that never comes
        q.put((rank, "error: %r" % (e,), None, None, None))
        raise
    finally:
        dist.destroy_process_group()


def _run(world, nan_at=None):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, nan_at, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
    for r in got:
        assert not isinstance(r[1], str), r[1]
    for p in procs:
        assert p.exitcode == 0
    return sorted(got, key=lambda x: x[0])


def _oracle(world, nan_at=None):
    """One rank stepping the whole model on every rank's micro-batches, (micro-batch, rank) order."""
    import oracle
    numels, nd = _model()
    total = sum(numels)
    P = _master0(total).numpy().copy()
    M, V, W = np.zeros(total, np.float32), np.zeros(total, np.float32), np.zeros(total, np.uint16)
    t_applied, flags = 0, []
    for t in range(1, STEPS + 1):
        micros = [_grad(t, r, k, total, nan=(t == nan_at and r == 1 and k == 1)).view(torch.int16).numpy()
                  .view(np.uint16) for k in range(K) for r in range(world)]
        G = np.zeros(total, np.float32)
        oracle.accumulate_all(G, micros)
        oracle.divide(G, world)
        ok, norm, coef = oracle.clip_coef(oracle.sumsq(G), HP["clip_grad"])
        flags.append(ok)
        if ok:
            assert coef < 1.0  # clipping is active: the global norm matters
            t_applied += 1
            oracle.adamw(P, M, V, G, np.array(numels, np.int64), np.array(nd, np.uint8), HP, t_applied, coef, w=W)
    return P, M, V, W, flags, t_applied


def _check(world, nan_at=None):
    got = _run(world, nan_at)
    P, M, V, W, flags, t_applied = _oracle(world, nan_at)
    seen = np.zeros(P.size, bool)
    for rank, applied, t, weights, out in got:
        assert applied == flags and t == t_applied
        assert np.array_equal(weights.view(np.uint16), W), rank
        mine = ~np.isnan(out["master"])
        assert not (seen & mine).any()
        seen |= mine
        for name, ref in (("master", P), ("m", M), ("v", V)):
            assert np.array_equal(out[name][mine].view(np.uint32), ref[mine].view(np.uint32)), (rank, name)
    assert seen.all()  # the ranks' shards cover the model


def test_two_rank_data_parallel_step_equals_the_unsharded_oracle_step():
    _check(2)


def test_three_rank_data_parallel_step_equals_the_unsharded_oracle_step():
    """With three ranks the order of the owner's fp32 additions matters (two values add the same
    either way): (micro-batch, rank) order, as the oracle adds them."""
    _check(3)


def test_a_nan_on_one_rank_makes_both_ranks_skip():
    _check(2, nan_at=1)


def _one_rank_nccl_worker(q):
    import socket as _s
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import zero_sharded_mixed_local_gb300 as z
    from zero_sharded_mixed_local_gb300.exchange import DataParallelStep

    torch.cuda.set_device(0)
    sock = _s.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    try:
        numels, nd = _model()
        total = sum(numels)
        hp = z.Hparams(**HP)
        a = z.LocalShardAdamW(numels, nd, 1, 0, hparams=hp)   # through DataParallelStep (NCCL buffers)
        b = z.LocalShardAdamW(numels, nd, 1, 0, hparams=hp)   # the local calls alone
        for o in (a, b):
            z.shard_gather(o.plan, _master0(total).cuda(), o.master)
            o.weight_bf16.copy_(o.master.to(torch.bfloat16))
        dps = DataParallelStep(a)
        assert dps.on_device
        weights = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        mb = b.plan.new_arena(torch.bfloat16)
        for t in range(1, STEPS + 1):
            micro = [_grad(t, 0, k, total, nan=False).cuda() for k in range(K)]
            dps.step(micro, weights_out=weights)
            for k, g in enumerate(micro):
                z.shard_gather(b.plan, g, mb)
                b.accumulate(mb, last=(k == K - 1))
            b.step()
        ref_w = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        z.shard_scatter(b.plan, b.weight_bf16, ref_w)
        same = [torch.equal(x.view(torch.int32), y.view(torch.int32))
                for x, y in ((a.master, b.master), (a.exp_avg, b.exp_avg), (a.exp_avg_sq, b.exp_avg_sq))]
        same.append(torch.equal(weights.view(torch.int16), ref_w.view(torch.int16)))
        q.put(same)
    except Exception as e:
        q.put("error: %r" % (e,))
        raise
    finally:
        dist.destroy_process_group()


def test_one_rank_nccl_group_equals_the_local_step():
    """The NCCL branch (collectives on device buffers) in a one-rank group on this GPU: the
    all-to-all, the all-reduce and the all-gather are identities, so three data-parallel steps
    must equal the plain local calls bit for bit (a division by 1 changes nothing)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_one_rank_nccl_worker, args=(q,))
    p.start()
    got = q.get(timeout=300)
    p.join(timeout=120)
    assert got == [True, True, True, True], got
    assert p.exitcode == 0


def _step_from_group_worker(rank, world, port, q):
    """step_from with a process group, on a side stream: the norm pass, the all-reduce of the sums of
    squares and the step, against the same rank stepping alone with the other rank's sum of squares as
    ``extra_sumsq`` (two doubles add the same in either order)."""
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import zero_sharded_mixed_local_gb300 as z

    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        numels, nd = _model()
        total = sum(numels)
        hp = z.Hparams(**HP)
        side = torch.cuda.Stream()
        results = []
        for kind in ("arena", "list"):
            for k_micro in (1, 3):
                make = z.LocalShardAdamW if kind == "arena" else z.ShardListAdamW
                a, b, c = (make(numels, nd, world, rank, hparams=hp) for _ in range(3))
                plan = a.plan
                m0 = plan.new_arena()
                z.shard_gather(plan, _master0(total).cuda(), m0)
                for o in (a, b):
                    if kind == "arena":
                        o.master.copy_(m0)
                    else:
                        for dst, src in zip(o.master, plan.shard_views(m0)):
                            dst.copy_(src)
                sums = []
                for t in range(1, STEPS + 1):
                    micro = []
                    for k in range(k_micro):
                        arena = plan.new_arena(torch.bfloat16)
                        z.shard_gather(plan, _grad(t, rank, k, total, nan=False).cuda(), arena)
                        micro.append(arena if kind == "arena" else [v.clone() for v in plan.shard_views(arena)])
                    if kind == "arena" and k_micro == 1:
                        micro = micro[0]
                    c.step_from(micro)  # this rank's own sum of squares, read back
                    own = z.read_norm(c.norm_out)["sumsq"]
                    got = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
                    dist.all_gather(got, torch.tensor([own], dtype=torch.float64))
                    extra = sum(float(g[0]) for r, g in enumerate(got) if r != rank)
                    side.wait_stream(torch.cuda.current_stream())
                    a.step_from(micro, group=dist.group.WORLD, stream=side)
                    torch.cuda.current_stream().wait_stream(side)
                    b.step_from(micro, extra_sumsq=extra)
                    torch.cuda.synchronize()
                    sums.append(z.read_norm(a.norm_out)["sumsq"] == z.read_norm(b.norm_out)["sumsq"])
                if kind == "arena":
                    pairs = [(a.master, b.master), (a.exp_avg, b.exp_avg), (a.exp_avg_sq, b.exp_avg_sq),
                             (a.grad, b.grad)]
                else:
                    pairs = [(torch.cat(list(x)), torch.cat(list(y))) for x, y in
                             ((a.master, b.master), (a.exp_avg, b.exp_avg), (a.exp_avg_sq, b.exp_avg_sq),
                              (a.grad, b.grad))]
                same = [torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in pairs]
                wa = a.weight_bf16 if kind == "arena" else torch.cat(list(a.weight_bf16))
                wb = b.weight_bf16 if kind == "arena" else torch.cat(list(b.weight_bf16))
                same.append(torch.equal(wa.view(torch.int16), wb.view(torch.int16)))
                results.append((kind, k_micro, all(sums), same, a.t))
        q.put((rank, results))
    except Exception as e:
        q.put((rank, "error: %r" % (e,)))
        raise
    finally:
        dist.destroy_process_group()


def test_step_from_with_a_group_on_a_side_stream_equals_the_local_step_with_extra_sumsq():
    """Two gloo ranks, each with its own shard and gradients: LocalShardAdamW.step_from and
    ShardListAdamW.step_from with the group (one micro-batch: the micro-batch norm, the all-reduce,
    the step that writes the gradient; three: the accumulating pass, the all-reduce, the step), on a
    stream that is not the current one, give every rank the global sum of squares and the same
    master, m, v, gradient and bf16 copy, bit for bit, as its local step given the other rank's
    share."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_step_from_group_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=120)
    for r in range(2):
        assert not isinstance(got[r], str), got[r]
        for kind, k_micro, sums_equal, same, t in got[r]:
            assert sums_equal, (r, kind, k_micro)
            assert same == [True] * 5, (r, kind, k_micro, same)
            assert t == STEPS
    for p in procs:
        assert p.exitcode == 0
