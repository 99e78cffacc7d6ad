"""The data movement around the local step, on a GB300: model layout <-> arena
copies (zero1_shard_gather / zero1_shard_scatter), and a whole ZeRO-1
data-parallel step emulated on one GPU with dp ranks.

In the emulation every collective is replaced by its definition: a
reduce-scatter is each owner accumulating the ranks' packed chunks in rank
order (zero1_accumulate, fp32, deterministic), the all-reduce of the sum of
squares is a host sum, and an all-gather is each rank's bf16 arena unpacked
into the full weights.  The result must equal the unsharded step bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_local_gb300 as z

pytestmark = pytest.mark.gpu

HP = z.Hparams(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gather_scatter_follow_the_shard_definition(dtype):
    numels = [1, 7, 8, 9, 100, 16384 * 2 + 5, 3, 40000, 0, 16384]
    nd = [1, 0, 0, 1, 0, 0, 1, 0, 0, 1]
    total = sum(numels)
    g = torch.Generator(device="cuda").manual_seed(3)
    full = (torch.randn(total, device="cuda", generator=g) * 3).to(dtype)
    full_np = _bits(full).cpu().numpy()
    model_off = np.concatenate([[0], np.cumsum(numels)[:-1]])
    sentinel = -777
    for dp in (1, 3, 8):
        rebuilt = torch.full((total,), sentinel, dtype=_bits(full).dtype, device="cuda").view(dtype)
        for r in range(dp):
            plan = z.Plan(numels, nd, dp, r)
            arena = plan.new_arena(dtype)
            z.shard_gather(plan, full, arena)
            start, count, _ = oracle.plan(numels, dp, r)
            L = plan.layout()
            expect = np.zeros(plan.arena_numel, full_np.dtype)
            mine = np.zeros(total, bool)
            for i in range(len(numels)):
                src = model_off[i] + start[i]
                expect[L.offsets[i]:L.offsets[i] + count[i]] = full_np[src:src + count[i]]
                mine[src:src + count[i]] = True
            assert np.array_equal(_bits(arena).cpu().numpy(), expect), (dp, r)
            z.shard_scatter(plan, arena, rebuilt)
            if r == 0:  # positions of the other ranks are untouched
                rb = _bits(rebuilt).cpu().numpy()
                assert np.all(rb[~mine] == sentinel) and np.array_equal(rb[mine], full_np[mine])
        assert torch.equal(_bits(rebuilt), _bits(full)), dp


def test_pack_and_unpack_helpers():
    numels = [5000, 13, 64, 2049]
    nd = [0, 1, 0, 0]
    dp = 3
    plans = [z.Plan(numels, nd, dp, r) for r in range(dp)]
    chunk = z.exchange_chunk_numel(plans)
    full = torch.arange(sum(numels), device="cuda", dtype=torch.float32)
    send = torch.full((dp, chunk), -1.0, device="cuda")
    z.pack_reduce_scatter(plans, full, send)
    for r, pl in enumerate(plans):
        a = pl.new_arena()
        z.shard_gather(pl, full, a)
        assert torch.equal(send[r, :pl.arena_numel], a) and not send[r, pl.arena_numel:].any()
    out = torch.zeros_like(full)
    z.unpack_all_gather(plans, send, out)
    assert torch.equal(out, full)


def test_pack_on_a_side_stream_fills_the_padding_before_its_gathers():
    """pack_reduce_scatter on a stream that is not the current one: the padding's zero fill is
    ordered with the gathers on that stream, so a buffer holding stale values ends up as the pack on
    the current stream gives it."""
    numels = [5000, 13, 64, 2049, 1 << 20]
    nd = [0, 1, 0, 0, 0]
    dp = 3
    plans = [z.Plan(numels, nd, dp, r) for r in range(dp)]
    chunk = z.exchange_chunk_numel(plans)
    full = torch.arange(sum(numels), device="cuda", dtype=torch.float32)
    ref = torch.empty((dp, chunk), device="cuda")
    z.pack_reduce_scatter(plans, full, ref)
    side = torch.cuda.Stream()
    for _ in range(3):
        send = torch.full((dp, chunk), 7.0, device="cuda")  # stale values, written on the current stream
        side.wait_stream(torch.cuda.current_stream())
        z.pack_reduce_scatter(plans, full, send, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        assert torch.equal(send, ref)


def _layouts(numels, nd, dp):
    return [z.Plan(numels, nd, dp, r) for r in range(dp)]


def test_data_parallel_step_emulated_on_one_gpu():
    """dp=4 ranks, each with its own K=2 bf16 micro-batch gradients in model layout, through
    reduce-scatter (pack + ordered accumulate), global norm, local steps and all-gather, for
    three steps: identical to one rank stepping the whole model on all 8 micro-batches."""
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    w = get_workload("toy")
    numels, nd = w.params.numels, w.params.no_decay
    total = sum(numels)
    dp, K = 4, 2
    gen = torch.Generator(device="cuda").manual_seed(11)
    master_full = torch.randn(total, device="cuda", generator=gen) * 0.02

    plans = _layouts(numels, nd, dp)
    ref_plan = z.Plan(numels, nd, 1, 0)

    def state(plan):
        s = {k: plan.new_arena() for k in ("master", "m", "v", "grad")}
        z.shard_gather(plan, master_full, s["master"])
        s["w"] = plan.new_arena(torch.bfloat16)
        s["ws"], s["nout"] = plan.new_workspace(), z.new_norm_out()
        return s

    ranks = [state(p) for p in plans]
    ref = state(ref_plan)
    chunk = z.exchange_chunk_numel(plans)
    for t in range(1, 4):
        # every rank's micro-batch gradients, model layout, bf16 (clip active: sigma 0.05)
        grads = [[(torch.randn(total, device="cuda", generator=gen) * 0.05).to(torch.bfloat16) for _ in range(K)]
                 for _ in range(dp)]
        # reduce-scatter: each rank packs; owner r accumulates the chunks in (rank, micro-batch) order
        packed = []
        for q in range(dp):
            for k in range(K):
                send = torch.empty((dp, chunk), dtype=torch.bfloat16, device="cuda")
                z.pack_reduce_scatter(plans, grads[q][k], send)
                packed.append(send)
        for r, (pl, st) in enumerate(zip(plans, ranks)):
            for n, send in enumerate(packed):
                z.accumulate(pl, st["grad"], send[r, :pl.arena_numel], overwrite_first=(n == 0))
            z.grad_norm(pl, st["grad"], st["ws"], st["nout"])
        # all-reduce of the sum of squares (in place, as allreduce_sumsq_ does)
        local = [z.read_norm(st["nout"])["sumsq"] for st in ranks]
        for r, (pl, st) in enumerate(zip(plans, ranks)):
            z.grad_norm(pl, st["grad"], st["ws"], st["nout"], extra_sumsq=sum(local) - local[r] if dp > 1 else 0.0)
            z.step(pl, st["master"], st["m"], st["v"], st["grad"], st["w"], HP, t, st["nout"])
        # the unsharded reference: one rank, all dp*K micro-batches in the same order
        n = 0
        for q in range(dp):
            for k in range(K):
                a = ref_plan.new_arena(torch.bfloat16)
                z.shard_gather(ref_plan, grads[q][k], a)
                z.accumulate(ref_plan, ref["grad"], a, overwrite_first=(n == 0))
                n += 1
        z.grad_norm(ref_plan, ref["grad"], ref["ws"], ref["nout"])
        z.step(ref_plan, ref["master"], ref["m"], ref["v"], ref["grad"], ref["w"], HP, t, ref["nout"])
        assert z.read_norm(ref["nout"])["norm"] > 1.0  # clipping is active

        # all-gather of the bf16 weights into model layout
        recv = torch.zeros((dp, chunk), dtype=torch.bfloat16, device="cuda")
        for r, (pl, st) in enumerate(zip(plans, ranks)):
            recv[r, :pl.arena_numel] = st["w"]
        weights = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        z.unpack_all_gather(plans, recv, weights)
        ref_weights = torch.zeros_like(weights)
        z.shard_scatter(ref_plan, ref["w"], ref_weights)
        assert torch.equal(_bits(weights), _bits(ref_weights)), t
        for key in ("master", "m", "v"):
            full = torch.zeros(total, device="cuda")
            for pl, st in zip(plans, ranks):
                z.shard_scatter(pl, st[key], full)
            ref_full = torch.zeros(total, device="cuda")
            z.shard_scatter(ref_plan, ref[key], ref_full)
            assert torch.equal(_bits(full), _bits(ref_full)), (t, key)


def test_checkpoint_resume_at_another_data_parallel_size(tmp_path):
    """Train 2 steps as 4 ranks, checkpoint, resume as 3 ranks for 2 more steps: master, m, v and
    the bf16 weights equal 4 steps of one rank on the whole model, bit for bit."""
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    w = get_workload("toy")
    numels, nd = w.params.numels, w.params.no_decay
    total = sum(numels)
    gen = torch.Generator(device="cuda").manual_seed(21)
    master_full = torch.randn(total, device="cuda", generator=gen) * 0.02
    grads = [(torch.randn(total, device="cuda", generator=gen) * 0.05).to(torch.bfloat16) for _ in range(4)]

    def make(plan):
        s = {k: plan.new_arena() for k in ("master", "m", "v", "grad")}
        z.shard_gather(plan, master_full, s["master"])
        s["w"], s["ws"], s["nout"], s["mb"] = (plan.new_arena(torch.bfloat16), plan.new_workspace(),
                                              z.new_norm_out(), plan.new_arena(torch.bfloat16))
        return s

    def run_steps(plans, states, ts):
        for t in ts:
            for pl, st in zip(plans, states):
                z.shard_gather(pl, grads[t - 1], st["mb"])
                z.accumulate_norm(pl, st["grad"], st["mb"], st["ws"], st["nout"])
            local = [z.read_norm(st["nout"])["sumsq"] for st in states]
            for r, (pl, st) in enumerate(zip(plans, states)):
                z.accumulate_norm(pl, st["grad"], st["mb"], st["ws"], st["nout"],
                                  extra_sumsq=sum(local) - local[r])
                z.step(pl, st["master"], st["m"], st["v"], st["grad"], st["w"], HP, t, st["nout"])

    def full_of(plans, states, key, dtype=torch.float32):
        out = torch.zeros(total, dtype=dtype, device="cuda")
        for pl, st in zip(plans, states):
            z.shard_scatter(pl, st[key], out)
        return out

    ref_plan = [z.Plan(numels, nd, 1, 0)]
    ref = [make(ref_plan[0])]
    run_steps(ref_plan, ref, (1, 2, 3, 4))

    plans4 = _layouts(numels, nd, 4)
    s4 = [make(p) for p in plans4]
    run_steps(plans4, s4, (1, 2))
    path = str(tmp_path / "ckpt")
    futs = [z.checkpoint.save_async(path, pl, st["master"], st["m"], st["v"], step_t=2) for pl, st in zip(plans4, s4)]
    for f in futs:
        f.result()
    plans3 = _layouts(numels, nd, 3)
    s3 = [make(p) for p in plans3]
    for pl, st in zip(plans3, s3):
        assert z.checkpoint.load(path, pl, st["master"], st["m"], st["v"]) == 2
    run_steps(plans3, s3, (3, 4))

    for key, dt in (("master", torch.float32), ("m", torch.float32), ("v", torch.float32), ("w", torch.bfloat16)):
        assert torch.equal(_bits(full_of(plans3, s3, key, dt)), _bits(full_of(ref_plan, ref, key, dt))), key
