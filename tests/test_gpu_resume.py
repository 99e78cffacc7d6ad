"""Checkpoint and resume through the optimizer classes on a GB300: stepping twice, saving,
loading into a fresh optimizer and stepping once more equals three uninterrupted steps,
bit for bit, for both layouts and with parameter groups."""
import pytest
import torch

import zero_sharded_mixed_local_gb300 as z

pytestmark = pytest.mark.gpu

NUMELS = [1000, 7, 4096, 33, 16385, 40000]
GROUPS = [0, 1, 2, 1, 0, 2]
LR_SCALE = [1.0, 1.0, 0.25, 1, 1, 1, 1, 1]
WD_SCALE = [1.0, 0.0, 0.5, 1, 1, 1, 1, 1]
HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)


def _make(kind):
    kw = dict(dp_size=2, dp_rank=0, hparams=HP, groups=GROUPS, lr_scale=LR_SCALE, wd_scale=WD_SCALE)
    return z.LocalShardAdamW(NUMELS, **kw) if kind == "arena" else z.ShardListAdamW(NUMELS, **kw)


def _micro(opt, step):
    g = torch.Generator(device="cuda").manual_seed(100 + step)
    if isinstance(opt, z.LocalShardAdamW):
        a = opt.plan.new_arena(torch.bfloat16)
        for v in opt.plan.shard_views(a):
            v.copy_(torch.randn(v.numel(), device="cuda", generator=g) * 1e-2)
        return a
    return [(torch.randn(int(c), device="cuda", generator=g) * 1e-2).to(torch.bfloat16)
            for c in opt.plan.layout().counts]


def _init(opt):
    g = torch.Generator(device="cuda").manual_seed(7)
    views = opt.plan.shard_views(opt.master) if isinstance(opt, z.LocalShardAdamW) else opt.master
    for v in views:
        v.copy_(torch.randn(v.numel(), device="cuda", generator=g) * 0.02)


def _state(opt):
    if isinstance(opt, z.LocalShardAdamW):
        return [torch.cat([v.clone() for v in opt.plan.shard_views(a)]) for a in (opt.master, opt.exp_avg,
                                                                                 opt.exp_avg_sq)]
    return [torch.cat([t.clone() for t in lst]) for lst in (opt.master, opt.exp_avg, opt.exp_avg_sq)]


@pytest.mark.parametrize("kind", ["arena", "list"])
@pytest.mark.parametrize("use_async", [False, True])
def test_resume_equals_uninterrupted(kind, use_async, tmp_path):
    a = _make(kind)
    _init(a)
    for s in range(3):
        a.accumulate(_micro(a, s), last=True)
        a.step()
    b = _make(kind)
    _init(b)
    for s in range(2):
        b.accumulate(_micro(b, s), last=True)
        b.step()
    fut = b.save_checkpoint(str(tmp_path / "ck"), meta={"kind": kind}, async_=use_async)
    if use_async:
        fut.result()
    c = _make(kind)  # a fresh process's optimizer
    assert c.load_checkpoint(str(tmp_path / "ck")) == 2
    c.accumulate(_micro(c, 2), last=True)
    c.step()
    for x, y in zip(_state(a), _state(c)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_list_checkpoint_loads_into_arenas_at_another_dp(tmp_path):
    lst = _make("list")
    _init(lst)
    lst.accumulate(_micro(lst, 0), last=True)
    lst.step()
    lst.save_checkpoint(str(tmp_path / "ck"))
    # rank 0 of dp 2 saved its own runs (and meta.json); the same rank reads them back as arenas
    arena = z.LocalShardAdamW(NUMELS, dp_size=2, dp_rank=0, hparams=HP, groups=GROUPS, lr_scale=LR_SCALE,
                              wd_scale=WD_SCALE)
    assert arena.load_checkpoint(str(tmp_path / "ck")) == 1
    for x, y in zip(_state(lst), _state(arena)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("kind", ["arena", "list"])
def test_skipped_step_keeps_the_step_count_with_check_finite(kind):
    """A non-finite gradient skips the step on the device; with check_finite the step count
    stays, so the next finite step is step 1 and equals a fresh optimizer's first step."""
    a, b = _make(kind), _make(kind)
    _init(a)
    _init(b)
    bad = _micro(a, 0)
    if kind == "arena":
        bad[0] = float("inf")
    else:
        bad[0][0] = float("inf")
    a.accumulate(bad, last=True)
    assert a.step(check_finite=True) is False and a.t == 0
    a.accumulate(_micro(a, 1), last=True)
    assert a.step(check_finite=True) is True and a.t == 1
    b.accumulate(_micro(b, 1), last=True)
    b.step()
    for x, y in zip(_state(a), _state(b)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("kind", ["arena", "list"])
def test_another_ranks_nonfinite_sum_skips_the_step(kind, monkeypatch):
    """After the all-reduce of the sums of squares the local record's status is still OK, but
    the sum is inf because another rank's gradient overflowed: the kernel skips the update,
    and check_finite reports the skip and keeps the step count."""
    import zero_sharded_mixed_local_gb300.optim as optim

    def allreduce_with_an_inf_rank(norm_out, group, stream=None):  # what the sum over the ranks gives
        norm_out[:8].view(torch.float64).fill_(float("inf"))

    monkeypatch.setattr(optim, "allreduce_sumsq_", allreduce_with_an_inf_rank)
    a = _make(kind)
    _init(a)
    before = _state(a)
    a.accumulate(_micro(a, 0), last=True)
    assert a.step(group=object(), check_finite=True) is False and a.t == 0
    assert z.read_norm(a.norm_out)["status"] == 0  # the local norm itself was finite
    for x, y in zip(_state(a), before):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("kind", ["arena", "list"])
def test_overlapping_checkpoints_keep_their_own_snapshots(kind, tmp_path):
    """Two asynchronous saves in flight at once, the state stepped in between: each takes its
    own page-locked staging, so each checkpoint holds the state of the moment it was taken."""
    a = _make(kind)
    _init(a)
    z.checkpoint.prepare_staging(a.plan)
    s0 = _state(a)
    f0 = a.save_checkpoint(str(tmp_path / "c0"), async_=True)
    a.accumulate(_micro(a, 0), last=True)
    a.step()
    s1 = _state(a)
    f1 = a.save_checkpoint(str(tmp_path / "c1"), async_=True)
    a.accumulate(_micro(a, 1), last=True)
    a.step()  # changes the state while the second save may still be writing
    f0.result()
    f1.result()
    for path, want, t in (("c0", s0, 0), ("c1", s1, 1)):
        b = _make(kind)
        assert b.load_checkpoint(str(tmp_path / path)) == t
        for x, y in zip(_state(b), want):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    z.checkpoint.release_staging()
