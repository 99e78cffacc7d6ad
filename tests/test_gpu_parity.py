"""CUDA path vs the CPU oracle, through the C ABI, on a GB300.

Small cases compare every arena element; the full-size workloads compare
sampled elements (tensor edges, padding, a million random positions) while
the gradient arena, the norm and the bf16 copy are still checked in full.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_local_gb300 as z
from zero_sharded_mixed_local_gb300.workloads import ParamList, Workload

from parity import MAX_ULP, Problem, oracle_grad, rne_of, run_parity, u16, ulp_diff

pytestmark = pytest.mark.gpu

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    z.load_library()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _custom(numels, no_decay, dp=1, rank=0, K=2, steps=3, sigma=1e-3, name="custom", hp=None, groups=None,
            lr_scale=None, wd_scale=None):
    return Workload(name, name, ParamList(["p%d" % i for i in range(len(numels))], list(numels), list(no_decay)),
                    dp, rank, K, steps, sigma, hp=dict(hp or HP), groups=groups, lr_scale=lr_scale,
                    wd_scale=wd_scale)


def test_parameter_groups_with_lr_and_wd_scales():
    """Eight tensors in five groups (two empty groups in between), each group with its own
    lr and weight-decay multiplier, clip active, every arena element compared."""
    numels = [5000, 17, 16384 + 3, 64, 1, 999, 4096, 40]
    groups = [3, 0, 3, 7, 1, 0, 5, 1]
    lr_scale = [1.0, 0.5, 1.0, 1 / 64, 1.0, 2.0, 1.0, 1 / 576]
    wd_scale = [1.0, 0.0, 1.0, 0.25, 1.0, 0.0, 1.0, 3.0]
    for dp, r in ((1, 0), (3, 2)):
        res = run_parity(_custom(numels, [0] * 8, dp, r, K=2, steps=4, sigma=0.05, groups=groups,
                                 lr_scale=lr_scale, wd_scale=wd_scale))
        assert res["master"] <= MAX_ULP


def test_smollm135m_mup_groups_full_size_sampled():
    res = run_parity("smollm135m_mup", sample="sampled")
    assert res["local_numel"] > 67_000_000


# ---------------------------------------------------------------- workloads
def test_toy_full_parity():
    res = run_parity("toy")
    assert res["master"] <= MAX_ULP


def test_toy_200_steps_every_element():
    """A long run: 200 steps of the toy shard with fresh gradients every step (K = 2, clipping
    decided anew each step); every arena element still equal to the oracle's at the end."""
    res = run_parity("toy", steps=200, fresh_grads=True)
    assert res["master"] == 0 and res["m"] == 0 and res["v"] == 0
    assert res["compared"] == Problem("toy").n


def test_toy_full_parity_unfused_calls():
    run_parity("toy", fused=False)


def test_fused_accumulate_norm_equals_separate_calls():
    """zero1_accumulate_norm writes the same gradient and the same norm record, bit for bit,
    as zero1_accumulate followed by zero1_grad_norm (same tiles, same summation order)."""
    for numels, K in (([16384 * 3 + 8 * 5 + 3, 1000, 77], 1), ([40000, 17, 16384], 3), ([9], 2)):
        pb = Problem(_custom(numels, [0, 1, 0][:len(numels)], K=K, steps=1, sigma=0.1))
        micros = pb.gen.micro_grads()
        recs = []
        grads = []
        for fused in (False, True):
            if fused:
                for k, mb in enumerate(micros[:-1]):
                    z.accumulate(pb.plan, pb.grad, mb, overwrite_first=(k == 0))
                z.accumulate_norm(pb.plan, pb.grad, micros[-1], pb.ws, pb.nout, overwrite_first=(K == 1),
                                  extra_sumsq=0.5)
            else:
                for k, mb in enumerate(micros):
                    z.accumulate(pb.plan, pb.grad, mb, overwrite_first=(k == 0))
                z.grad_norm(pb.plan, pb.grad, pb.ws, pb.nout, 0.5)
            recs.append(z.read_norm(pb.nout))
            grads.append(pb.grad.clone())
        assert recs[0] == recs[1]
        assert torch.equal(grads[0].view(torch.int32), grads[1].view(torch.int32))
    # several micro-batches in the fused call itself
    pb = Problem(_custom([33333, 64], [0, 1], K=4, steps=1, sigma=0.3))
    micros = pb.gen.micro_grads()
    z.accumulate_norm(pb.plan, pb.grad, micros, pb.ws, pb.nout, overwrite_first=True)
    r1 = z.read_norm(pb.nout)
    g1 = pb.grad.clone()
    z.accumulate(pb.plan, pb.grad, micros, overwrite_first=True)
    z.grad_norm(pb.plan, pb.grad, pb.ws, pb.nout)
    assert z.read_norm(pb.nout) == r1 and torch.equal(g1, pb.grad)


def test_wide_and_narrow_gradient_stores_agree():
    """The passes that write the gradient without reading it first store it with 256-bit accesses
    when the arena is 32-byte aligned and with two 128-bit ones when it is only 16-byte aligned (the
    ABI's minimum). Both keep each thread's elements, so the gradient and the norm record must be
    the same bits: the one-micro-batch fused pass, and the overwriting accumulate with adds after."""
    pb = Problem(_custom([16384 * 3 + 8 * 5 + 3, 1000, 77], [0, 1, 0], K=3, steps=1, sigma=0.1))
    micros = pb.gen.micro_grads()
    wide = pb.plan.new_arena()
    back = torch.zeros(pb.n + 4, device="cuda")
    narrow = back[4:]  # 16 bytes past an aligned start
    assert wide.data_ptr() % 32 == 0 and narrow.data_ptr() % 32 == 16
    recs = []
    for g in (wide, narrow):
        z.accumulate_norm(pb.plan, g, micros[0], pb.ws, pb.nout, overwrite_first=True)
        recs.append(z.read_norm(pb.nout))
    assert recs[0] == recs[1]
    assert torch.equal(wide.view(torch.int32), narrow.view(torch.int32))
    for g in (wide, narrow):
        z.accumulate(pb.plan, g, micros, overwrite_first=True)
    assert torch.equal(wide.view(torch.int32), narrow.view(torch.int32))
    ref = oracle_grad(pb.n, [u16(m) for m in micros])
    assert np.array_equal(narrow.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_smollm135m_full_size_sampled():
    res = run_parity("smollm135m", sample="sampled")
    assert res["local_numel"] == 134_515_008


def test_smollm1p7b_full_size_sampled_clip_active():
    res = run_parity("smollm1p7b", sample="sampled")
    assert res["local_numel"] == 213_922_048
    t, gpu_norm, ref_norm, coef = res["norms"][0]
    assert 3.0 < ref_norm < 5.0 and coef < 1.0  # the grads were scaled so clipping is active


def test_llama8b_full_size_sampled():
    """The bench's configuration for K = 1: the norm from the micro-batch, then the step that
    writes the gradient (the gradient is still checked in full against the oracle)."""
    res = run_parity("llama8b", steps=10, sample="sampled", micro_step=True)
    assert res["local_numel"] == 1_003_782_656


def test_ragged_full_size_sampled():
    res = run_parity("ragged", sample="sampled")
    _, gpu_norm, ref_norm, coef = res["norms"][0]
    assert ref_norm > 1.0 and coef < 1.0


# ---------------------------------------------------------------- edge cases
def test_tiny_and_ragged_tensors_all_ranks():
    numels = list(range(1, 18)) + [0, 1023, 1025, 16384 * 3 + 5]
    nd = [i % 3 == 0 for i in range(len(numels))]
    for dp in (1, 2, 3, 4, 8):
        for r in range(dp):
            run_parity(_custom(numels, nd, dp, r, K=3, steps=4, sigma=0.05))


def test_multi_tile_with_ragged_tail():
    # several 16384-element norm tiles and a tail that is not a multiple of 16
    numels = [16384 * 5 + 8 * 3 + 7, 100003, 6]
    run_parity(_custom(numels, [0, 0, 1], K=2, steps=3, sigma=0.02))


def test_empty_plan_is_a_no_op():
    plan = z.Plan([0, 0, 0], [0, 1, 0], 1, 0)
    assert plan.arena_numel == 0 and plan.workspace_bytes == 0
    nout = z.new_norm_out()
    # zero-length arenas: nothing to launch for the element-wise calls
    g = torch.zeros(0, device="cuda")
    z.accumulate(plan, g, torch.zeros(0, dtype=torch.bfloat16, device="cuda"))
    z.grad_norm(plan, g, torch.zeros(16, dtype=torch.uint8, device="cuda"), nout, extra_sumsq=9.0)
    r = z.read_norm(nout)
    assert r["sumsq"] == 9.0 and r["norm"] == 3.0 and r["status"] == 0 and r["n_partials"] == 0
    z.step(plan, g, g.clone(), g.clone(), g, torch.zeros(0, dtype=torch.bfloat16, device="cuda"), z.Hparams(), 1,
           nout)


def test_shards_with_fewer_elements_than_ranks():
    # numel < dp: some ranks own nothing of a tensor
    numels = [1, 2, 3, 5, 7]
    for r in range(8):
        plan = z.Plan(numels, [0] * 5, 8, r)
        _, counts, _ = oracle.plan(numels, 8, r)
        assert plan.local_numel == int(counts.sum())
        if plan.arena_numel:
            run_parity(_custom(numels, [0] * 5, 8, r, K=1, steps=2, sigma=0.1))


def test_nonfinite_gradient_skips_the_step():
    for bad in (float("nan"), float("inf")):
        pb = Problem(_custom([1000, 64], [0, 1], K=2, steps=1))
        micros = pb.gen.micro_grads()
        micros[1][123] = bad
        before = [t.clone() for t in (pb.master, pb.m, pb.v, pb.wbf)]
        got = pb.gpu_step(micros, 1)
        assert got["status"] == z.ZERO1_ENONFINITE
        for a, b in zip(before, (pb.master, pb.m, pb.v, pb.wbf)):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_clip_below_threshold_equals_no_clip_and_no_norm():
    outs = []
    for clip, use_norm in ((1.0, True), (0.0, True), (1.0, False)):
        pb = Problem(_custom([4096, 512, 33], [0, 1, 0], K=2, steps=1, hp=dict(HP, clip_grad=clip)))
        micros = pb.gen.micro_grads()
        z.accumulate(pb.plan, pb.grad, micros)
        z.grad_norm(pb.plan, pb.grad, pb.ws, pb.nout)
        assert z.read_norm(pb.nout)["norm"] < 1.0
        z.step(pb.plan, pb.master, pb.m, pb.v, pb.grad, pb.wbf, pb.hp, 1, pb.nout if use_norm else None)
        outs.append([t.cpu() for t in (pb.master, pb.m, pb.v, pb.wbf)])
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_zero_gradient_is_pure_decay_bit_exact():
    pb = Problem(_custom([1000, 256, 77], [0, 1, 0], K=1, steps=1))
    p0 = pb.master.clone()
    zero = torch.zeros_like(pb.wbf)
    pb.gpu_step([zero], 1)
    dfac = np.float32(1.0 - HP["lr"] * HP["weight_decay"])
    b = pb.group1
    exp = p0.cpu().numpy().copy()
    exp[:b] = exp[:b] * dfac
    assert np.array_equal(pb.master.cpu().numpy().view(np.uint32), exp.view(np.uint32))
    assert not pb.m.any() and not pb.v.any()


def test_step_without_bf16_copy_matches():
    pa = Problem(_custom([5000, 31], [0, 1], K=1, steps=1))
    pb = Problem(_custom([5000, 31], [0, 1], K=1, steps=1))
    mic = pa.gen.micro_grads()
    for pr, w in ((pa, pa.wbf), (pb, None)):
        z.accumulate(pr.plan, pr.grad, mic)
        z.grad_norm(pr.plan, pr.grad, pr.ws, pr.nout)
        z.step(pr.plan, pr.master, pr.m, pr.v, pr.grad, w, pr.hp, 1, pr.nout)
    assert torch.equal(pa.master, pb.master) and torch.equal(pa.m, pb.m) and torch.equal(pa.v, pb.v)
    assert not pb.wbf.view(torch.int16).any()


def test_accumulate_many_micro_batches_in_one_call():
    pb = Problem(_custom([40000, 17], [0, 1], K=16, steps=1, sigma=0.5))
    micros = pb.gen.micro_grads()
    z.accumulate(pb.plan, pb.grad, micros, overwrite_first=True)
    ref = oracle_grad(pb.n, [u16(m) for m in micros])
    assert np.array_equal(pb.grad.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    # and without overwrite: grad += sum
    z.accumulate(pb.plan, pb.grad, micros[:3], overwrite_first=False)
    for m in micros[:3]:
        oracle.accumulate(ref, u16(m), overwrite=False)
    assert np.array_equal(pb.grad.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("K", [2, 3, 4, 5, 6, 7, 8, 9])
def test_k_way_fused_pass_matches_the_oracle(K):
    """All K micro-batches in one fused accumulate-and-norm call (the K-specialised kernels for
    K <= 8, the general one above): the gradient bit for bit, the norm record equal to the
    separate calls', with and without the world-size divisor; several tiles and a ragged tail."""
    pb = Problem(_custom([40000, 17, 3 * 16384 + 40], [0, 1, 0], K=K, steps=1, sigma=0.5))
    micros = pb.gen.micro_grads()
    ref = oracle_grad(pb.n, [u16(m) for m in micros])
    for divisor in (1.0, 3.0):
        z.accumulate_norm(pb.plan, pb.grad, micros, pb.ws, pb.nout, overwrite_first=True, divisor=divisor)
        got = z.read_norm(pb.nout)
        exp = ref.copy()
        if divisor != 1.0:
            oracle.divide(exp, divisor)
        assert np.array_equal(pb.grad.cpu().numpy().view(np.uint32), exp.view(np.uint32)), divisor
        # the same gradient through the separate norm call: identical record
        nout2 = z.new_norm_out()
        z.grad_norm(pb.plan, pb.grad, pb.ws, nout2)
        assert z.read_norm(nout2)["sumsq"] == got["sumsq"]
        s = oracle.sumsq(exp)
        assert abs(got["sumsq"] - s) <= 1e-12 * s


def test_norm_is_deterministic_and_extra_sumsq_adds():
    pb = Problem(_custom([16384 * 7 + 40, 9], [0, 1], K=1, steps=1, sigma=0.3))
    z.accumulate(pb.plan, pb.grad, pb.gen.micro_grads())
    vals = []
    for extra in (0.0, 0.0, 2.5):
        z.grad_norm(pb.plan, pb.grad, pb.ws, pb.nout, extra)
        vals.append(z.read_norm(pb.nout))
    assert vals[0] == vals[1]
    assert vals[2]["sumsq"] == vals[0]["sumsq"] + 2.5
    assert vals[0]["n_partials"] == 8


def test_shard_concatenation_on_gpu():
    """All dp ranks stepped on the one GPU, each with the other ranks' sum of squares,
    reproduce the unsharded step bit for bit."""
    numels = [1000, 3, 64, 4097, 11, 257]
    nd = [0, 1, 0, 0, 1, 0]
    dp = 4
    N = sum(numels)
    tstart = np.concatenate([[0], np.cumsum(numels)[:-1]])
    rng = torch.Generator(device="cuda").manual_seed(5)
    full_micro = [(torch.randn(N, device="cuda", generator=rng) * 0.2).to(torch.bfloat16) for _ in range(2)]
    full_p = torch.randn(N, device="cuda", generator=rng) * 0.02

    def run(dp_size, rank, extra=None):
        plan = z.Plan(numels, nd, dp_size, rank)
        L = plan.layout()
        sel = [np.arange(tstart[i] + L.shard_start[i], tstart[i] + L.shard_start[i] + L.counts[i])
               for i in range(len(numels))]
        def arena_of(full, dtype):
            a = plan.new_arena(dtype)
            for i, s in enumerate(sel):
                if len(s):
                    a[int(L.offsets[i]):int(L.offsets[i]) + len(s)] = full[torch.from_numpy(s).cuda()]
            return a
        master, m, v, g = arena_of(full_p, torch.float32), plan.new_arena(), plan.new_arena(), plan.new_arena()
        wbf = plan.new_arena(torch.bfloat16)
        z.accumulate(plan, g, [arena_of(mb, torch.bfloat16) for mb in full_micro])
        ws, nout = plan.new_workspace(), z.new_norm_out()
        z.grad_norm(plan, g, ws, nout, 0.0)
        local = z.read_norm(nout)["sumsq"]
        if extra is not None:
            z.grad_norm(plan, g, ws, nout, extra)
            z.step(plan, master, m, v, g, wbf, z.Hparams(**HP), 1, nout)
        return plan, sel, local, (master, m, v, wbf)

    ref_plan, ref_sel, ref_sumsq, ref_out = run(1, 0, 0.0)
    locals_ = [run(dp, r)[2] for r in range(dp)]
    for r in range(dp):
        plan, sel, _, out = run(dp, r, sum(s for q, s in enumerate(locals_) if q != r))
        L, RL = plan.layout(), ref_plan.layout()
        for i, s in enumerate(sel):
            if not len(s):
                continue
            o = int(L.offsets[i])
            ro = int(RL.offsets[i]) + int(L.shard_start[i])
            for a, b in zip(out, ref_out):
                assert torch.equal(a[o:o + len(s)].view(torch.uint8) if a.dtype != torch.bfloat16 else
                                   a[o:o + len(s)].view(torch.int16),
                                   b[ro:ro + len(s)].view(torch.uint8) if b.dtype != torch.bfloat16 else
                                   b[ro:ro + len(s)].view(torch.int16))


def test_micro_batches_read_from_pinned_host_memory():
    """Pinned host arenas are read by the kernels directly (no staging copy): same gradient
    and norm record, bit for bit, as from device memory."""
    pb = Problem(_custom([40000, 1000, 17], [0, 1, 0], K=3, steps=1, sigma=0.2))
    micros = pb.gen.micro_grads()
    host = [m.cpu().pin_memory() for m in micros]
    outs = []
    for src in (micros, host):
        z.accumulate(pb.plan, pb.grad, src[0], overwrite_first=True)
        z.accumulate(pb.plan, pb.grad, src[1], overwrite_first=False)
        z.accumulate_norm(pb.plan, pb.grad, src[2], pb.ws, pb.nout, overwrite_first=False)
        outs.append((pb.grad.clone(), z.read_norm(pb.nout)))
    assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32))
    assert outs[0][1] == outs[1][1]
    # a plain (pageable) CPU tensor is refused by the binding
    with pytest.raises(ValueError, match="pinned"):
        z.accumulate(pb.plan, pb.grad, micros[0].cpu())


def test_misaligned_and_wrong_size_buffers_are_rejected():
    plan = z.Plan([100], [0], 1, 0)
    g = plan.new_arena()
    n = plan.arena_numel
    big = torch.zeros(n + 4, device="cuda")
    mb = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError, match="16-byte"):
        z.accumulate(plan, big[1:1 + n], mb)  # 4-byte offset
    with pytest.raises(ValueError, match="elements"):
        z.accumulate(plan, big, mb)           # wrong size
    # straight through the C ABI: misalignment is caught before any launch
    lib = z.load_library()
    arr = (ctypes.c_void_p * 1)(torch.zeros(112, dtype=torch.bfloat16, device="cuda").data_ptr() + 2)
    assert lib.zero1_accumulate(plan.handle, ctypes.c_void_p(g.data_ptr()), arr, 1, 1, None) == z.ZERO1_EALIGN


@pytest.mark.parametrize("guard_bytes", [256, 272])
def test_no_call_writes_outside_its_buffers(guard_bytes):
    """Every buffer sits between two guard zones filled with a pattern; after every entry point has
    run on it, the guards are unchanged.  256-byte guards leave the buffers 32-byte aligned (the
    256-bit gradient stores), 272-byte ones only 16-byte aligned (the 128-bit stores)."""
    numels = [1000, 7, 16384 + 9, 33]
    nd = [0, 1, 0, 1]
    plan = z.Plan(numels, nd, 3, 1)
    n, total = plan.arena_numel, plan.total_numel

    def guarded(count, dtype):
        G = guard_bytes // torch.empty(0, dtype=dtype).element_size()
        buf = torch.empty(count + 2 * G, dtype=dtype, device="cuda")
        buf.view(torch.uint8).fill_(0xA5)
        return buf, buf[G:G + count]

    def zero_mid(pair):
        pair[1].zero_()
        return pair

    bufs = {k: zero_mid(guarded(n, torch.float32)) for k in ("grad", "master", "m", "v")}
    bufs["w"] = zero_mid(guarded(n, torch.bfloat16))
    bufs["mb"] = zero_mid(guarded(n, torch.bfloat16))
    bufs["ws"] = guarded(max(plan.workspace_bytes, 16), torch.uint8)
    bufs["nout"] = guarded(32, torch.uint8)
    bufs["full32"] = guarded(total, torch.float32)
    bufs["full16"] = guarded(total, torch.bfloat16)
    g = torch.Generator(device="cuda").manual_seed(9)
    L = plan.layout()
    for o, c in zip(L.offsets, L.counts):
        bufs["mb"][1][int(o):int(o) + int(c)] = (torch.randn(int(c), device="cuda", generator=g) * 0.1).to(
            torch.bfloat16)
        bufs["master"][1][int(o):int(o) + int(c)] = torch.randn(int(c), device="cuda", generator=g) * 0.02
    bufs["full32"][1].normal_(generator=g)
    bufs["full16"][1].normal_(generator=g)
    B = {k: v[1] for k, v in bufs.items()}
    assert (B["grad"].data_ptr() % 32 == 0) == (guard_bytes % 32 == 0)
    z.accumulate_norm(plan, B["grad"], B["mb"], B["ws"], B["nout"])
    z.local_step(plan, B["grad"], [B["mb"], B["mb"]], B["ws"], B["nout"], B["master"], B["m"], B["v"], B["w"],
                 z.Hparams(), 1)
    z.accumulate(plan, B["grad"], B["mb"])
    z.accumulate(plan, B["grad"], [B["mb"], B["mb"]], overwrite_first=False)
    z.accumulate_norm(plan, B["grad"], B["mb"], B["ws"], B["nout"], overwrite_first=False)
    z.grad_norm(plan, B["grad"], B["ws"], B["nout"])
    z.grad_norm_static(plan, B["grad"], B["nout"])
    z.step(plan, B["master"], B["m"], B["v"], B["grad"], B["w"], z.Hparams(), 1, B["nout"])
    z.shard_gather(plan, B["full32"], B["master"])
    z.shard_scatter(plan, B["master"], B["full32"])
    z.shard_gather(plan, B["full16"], B["w"])
    z.shard_scatter(plan, B["w"], B["full16"])
    torch.cuda.synchronize()
    for k, (buf, mid) in bufs.items():
        raw = buf.view(torch.uint8)
        eb = buf.element_size()
        head, tail = raw[:guard_bytes], raw[guard_bytes + mid.numel() * eb:]
        assert bool((head == 0xA5).all()) and bool((tail == 0xA5).all()), k


def test_other_hyperparameters_and_late_steps():
    """lr 1e-2, betas (0.8, 0.999), eps 1e-6, weight decay 0.01, clip 0.5, steps 1000-1003
    (bias corrections near 1) and steps 1-4, every element compared."""
    hp = dict(lr=1e-2, beta1=0.8, beta2=0.999, eps=1e-6, weight_decay=0.01, clip_grad=0.5)
    w = _custom([5000, 3, 16384 + 40, 100], [0, 1, 0, 1], dp=2, rank=1, K=3, steps=4, sigma=0.02, hp=hp)
    res = run_parity(w)
    assert res["master"] <= MAX_ULP
    pb = Problem(w)
    P = pb.master.cpu().numpy().copy()
    M = np.zeros(pb.n, np.float32)
    V = np.zeros(pb.n, np.float32)
    from parity import group_counts, oracle_pass
    idx = np.arange(pb.n, dtype=np.int64)
    counts = group_counts(idx, pb.plan)
    lr_s, wd_s = w.group_scales()
    for t in (1000, 1001, 1002, 1003):
        micros = pb.gen.micro_grads()
        got = pb.gpu_step(micros, t)
        g_idx, ref = oracle_pass(micros, pb.grad, idx)
        ok, norm, coef = oracle.clip_coef(ref, hp["clip_grad"])
        oracle.adamw_scaled(P, M, V, g_idx, counts, lr_s, wd_s, hp, t, coef)
    for a, b in ((pb.master, P), (pb.m, M), (pb.v, V)):
        assert ulp_diff(a.cpu().numpy(), b).max() <= MAX_ULP


def test_fused_pass_divides_by_the_world_size():
    """zero1_accumulate_norm with grad_divisor d: grad = (sum of micro-batches) / d, one IEEE
    division per element after the last addition, bit for bit against the oracle; the norm is
    the norm of the divided gradient."""
    for K, d in ((1, 2.0), (3, 3.0), (2, 8.0), (4, 7.0)):
        pb = Problem(_custom([16384 * 2 + 13, 77, 1000], [0, 1, 0], K=K, steps=1, sigma=0.3))
        micros = pb.gen.micro_grads()
        for k, mb in enumerate(micros[:-1]):
            z.accumulate(pb.plan, pb.grad, mb, overwrite_first=(k == 0))
        z.accumulate_norm(pb.plan, pb.grad, micros[-1], pb.ws, pb.nout, overwrite_first=(K == 1), divisor=d)
        got = z.read_norm(pb.nout)
        ref = oracle_grad(pb.n, [u16(m) for m in micros])
        oracle.divide(ref, d)
        assert np.array_equal(pb.grad.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (K, d)
        s = oracle.sumsq(ref)
        assert abs(got["sumsq"] - s) <= 1e-12 * s


def test_data_parallel_average_emulated_on_one_gpu():
    """dp=4 ranks reduce-scatter their gradients and divide by the world size in the fused pass
    (the FSDP2-style average), take the global norm and step: equal to one rank stepping on the
    average of all ranks' gradients, bit for bit."""
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    w = get_workload("toy")
    numels, nd = w.params.numels, w.params.no_decay
    total, dp = sum(numels), 4
    gen = torch.Generator(device="cuda").manual_seed(31)
    master_full = torch.randn(total, device="cuda", generator=gen) * 0.02
    plans = [z.Plan(numels, nd, dp, r) for r in range(dp)]
    ref_plan = z.Plan(numels, nd, 1, 0)
    chunk = z.exchange_chunk_numel(plans)

    def state(plan):
        s = {k: plan.new_arena() for k in ("master", "m", "v", "grad")}
        z.shard_gather(plan, master_full, s["master"])
        s["w"], s["ws"], s["nout"] = plan.new_arena(torch.bfloat16), plan.new_workspace(), z.new_norm_out()
        return s

    ranks, ref = [state(p) for p in plans], state(ref_plan)
    hp = z.Hparams(**w.hp)
    for t in (1, 2):
        grads = [(torch.randn(total, device="cuda", generator=gen) * 0.1).to(torch.bfloat16) for _ in range(dp)]
        sends = []
        for q in range(dp):
            send = torch.empty((dp, chunk), dtype=torch.bfloat16, device="cuda")
            z.pack_reduce_scatter(plans, grads[q], send)
            sends.append(send)
        for r, (pl, st) in enumerate(zip(plans, ranks)):
            for q in range(dp - 1):
                z.accumulate(pl, st["grad"], sends[q][r, :pl.arena_numel], overwrite_first=(q == 0))
            z.accumulate_norm(pl, st["grad"], sends[dp - 1][r, :pl.arena_numel], st["ws"], st["nout"],
                              overwrite_first=False, divisor=dp)
        local = [z.read_norm(st["nout"])["sumsq"] for st in ranks]
        for r, (pl, st) in enumerate(zip(plans, ranks)):
            z.grad_norm(pl, st["grad"], st["ws"], st["nout"], extra_sumsq=sum(local) - local[r])
            z.step(pl, st["master"], st["m"], st["v"], st["grad"], st["w"], hp, t, st["nout"])
        for q in range(dp):
            a = ref_plan.new_arena(torch.bfloat16)
            z.shard_gather(ref_plan, grads[q], a)
            if q < dp - 1:
                z.accumulate(ref_plan, ref["grad"], a, overwrite_first=(q == 0))
            else:
                z.accumulate_norm(ref_plan, ref["grad"], a, ref["ws"], ref["nout"], overwrite_first=False,
                                  divisor=dp)
        z.step(ref_plan, ref["master"], ref["m"], ref["v"], ref["grad"], ref["w"], hp, t, ref["nout"])
    for key in ("master", "m", "v"):
        full, ref_full = torch.zeros(total, device="cuda"), torch.zeros(total, device="cuda")
        for pl, st in zip(plans, ranks):
            z.shard_scatter(pl, st[key], full)
        z.shard_scatter(ref_plan, ref[key], ref_full)
        assert torch.equal(full.view(torch.int32), ref_full.view(torch.int32)), key


def test_arena_beyond_2_to_32_elements():
    """Maximum size: one tensor of 2^32 + 2^20 + 5 elements (dp 1; 86 GB resident) and a tiny
    excluded one.  Every gradient element is 2^-8 (exact in bf16), so the sum of squares is
    N * 2^-16 exactly; elements around 2^31, 2^32 and the tail are stepped by the oracle.  Through the
    two-pass calls, then through the one-micro-batch pair on the same buffers."""
    n0 = (1 << 32) + (1 << 20) + 5
    plan = z.Plan([n0, 3], [0, 1], 1, 0)
    n, N = plan.arena_numel, plan.local_numel
    dev = torch.device("cuda")
    mb = torch.full((n,), 2.0 ** -8, dtype=torch.bfloat16, device=dev)
    mb[n0:plan.group_range(1)[0]] = 0  # padding after tensor 0
    mb[plan.group_range(1)[0] + 3:] = 0
    g = torch.Generator(device=dev).manual_seed(3)
    master = torch.zeros(n, dtype=torch.float32, device=dev)
    master[:n0].normal_(0.0, 0.02, generator=g)
    b1 = plan.group_range(1)[0]
    master[b1:b1 + 3] = 1.0
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    grad = torch.empty_like(master)
    wbf = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    ws, nout = plan.new_workspace(dev), z.new_norm_out(dev)
    edges = [(1 << 31) - 12, (1 << 32) - 12, n0 - 12, b1]
    idx = np.unique(np.concatenate([np.arange(e, e + 24) for e in edges] +
                                   [np.random.default_rng(0).integers(0, n0, 100000)]))
    idx = idx[(idx < n0) | ((idx >= b1) & (idx < b1 + 3))]
    it = torch.from_numpy(idx).to(dev)
    P0 = master[it].cpu().numpy().copy()
    z.accumulate_norm(plan, grad, mb, ws, nout)
    hp = dict(HP)
    z.step(plan, master, m, v, grad, wbf, z.Hparams(**hp), 1, nout)
    got = z.read_norm(nout)
    assert got["status"] == 0
    assert got["sumsq"] == N * 2.0 ** -16, (got["sumsq"], N * 2.0 ** -16)
    G = grad[it].cpu().numpy()
    assert np.all(G == np.float32(2.0 ** -8))
    ok, norm, coef = oracle.clip_coef(N * 2.0 ** -16, hp["clip_grad"])
    P, M, V = P0.copy(), np.zeros_like(P0), np.zeros_like(P0)
    dec = int(np.sum(idx < n0))
    oracle.adamw(P, M, V, G, [dec, idx.size - dec], [0, 1], hp, 1, coef)
    for name, t, ref in (("master", master, P), ("m", m, M), ("v", v, V)):
        assert np.array_equal(t[it].cpu().numpy().view(np.uint32), ref.view(np.uint32)), name
    assert np.array_equal(u16(wbf[it]), oracle.bf16_rne(P))
    # the same step through the one-micro-batch pair (norm from the micro-batch, then the step that
    # writes the gradient), on the same buffers restored to the initial state
    g = torch.Generator(device=dev).manual_seed(3)
    master.zero_()
    master[:n0].normal_(0.0, 0.02, generator=g)
    master[b1:b1 + 3] = 1.0
    assert np.array_equal(master[it].cpu().numpy(), P0)
    m.zero_()
    v.zero_()
    grad.fill_(float("nan"))
    wbf.zero_()
    z.micro_norm(plan, mb, ws, nout)
    z.step_accumulate(plan, master, m, v, grad, mb, wbf, z.Hparams(**hp), 1, nout)
    got = z.read_norm(nout)
    assert got["status"] == 0 and got["sumsq"] == N * 2.0 ** -16
    assert np.all(grad[it].cpu().numpy() == np.float32(2.0 ** -8))
    for name, t, ref in (("master", master, P), ("m", m, M), ("v", v, V)):
        assert np.array_equal(t[it].cpu().numpy().view(np.uint32), ref.view(np.uint32)), name
    assert np.array_equal(u16(wbf[it]), oracle.bf16_rne(P))
    del mb, master, m, v, grad, wbf
    torch.cuda.empty_cache()


def test_four_element_worked_example_on_the_gpu():
    """The hand-worked four-element case of the oracle pins (two tensors, clipping at norm 1.625,
    a repeated and a sign-flipped gradient), through the C ABI: the same numbers."""
    from test_oracle_pins import FOUR_G, FOUR_HP, FOUR_P, FOUR_P0
    plan = z.Plan([2, 2], [0, 1], 1, 0)
    offs = plan.layout().offsets
    n = plan.arena_numel
    dev = torch.device("cuda")
    master = torch.zeros(n, device=dev)
    for i, o in enumerate(offs):
        master[int(o):int(o) + 2] = torch.tensor(FOUR_P0[2 * i:2 * i + 2])
    m, v, grad = torch.zeros_like(master), torch.zeros_like(master), torch.zeros_like(master)
    wbf = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    ws, nout = plan.new_workspace(dev), z.new_norm_out(dev)
    hp = z.Hparams(**FOUR_HP, clip_grad=1.0)
    for t, (g, expect) in enumerate(zip(FOUR_G, FOUR_P), start=1):
        mb = torch.zeros(n, dtype=torch.bfloat16, device=dev)
        for i, o in enumerate(offs):
            mb[int(o):int(o) + 2] = torch.tensor(g[2 * i:2 * i + 2]).to(torch.bfloat16)
        z.accumulate_norm(plan, grad, mb, ws, nout)
        z.step(plan, master, m, v, grad, wbf, hp, t, nout)
        got = z.read_norm(nout)
        assert got["sumsq"] == 2.640625 and got["norm"] == 1.625
        vals = torch.cat([master[int(o):int(o) + 2] for o in offs]).cpu().numpy()
        np.testing.assert_allclose(vals, expect, rtol=0, atol=2.5e-7)


def test_launch_count_counts_each_kernel():
    """zero1_launch_count grows by the kernels each call launches: a plain accumulate one, the
    fused last pass two (the tile pass and the final reduction), the step one, a separate norm
    two; a call rejected before any launch none."""
    pb = Problem(_custom([16384 * 2 + 13, 77], [0, 1], K=2, steps=1, sigma=0.1))
    micros = pb.gen.micro_grads()
    c0 = z.launch_count()
    z.accumulate(pb.plan, pb.grad, micros[0])
    assert z.launch_count() - c0 == 1
    z.accumulate_norm(pb.plan, pb.grad, micros[1], pb.ws, pb.nout, overwrite_first=False)
    assert z.launch_count() - c0 == 3
    z.step(pb.plan, pb.master, pb.m, pb.v, pb.grad, pb.wbf, pb.hp, 1, pb.nout)
    assert z.launch_count() - c0 == 4
    z.grad_norm(pb.plan, pb.grad, pb.ws, pb.nout)
    assert z.launch_count() - c0 == 6
    with pytest.raises(z.Zero1Error):
        z.step(pb.plan, pb.master, pb.m, pb.v, pb.grad, pb.wbf, pb.hp, 0, pb.nout)  # t < 1
    assert z.launch_count() - c0 == 6


def test_random_configurations_match_the_oracle():
    """Forty seeded random configurations, every element compared over two steps: 1-12 tensors of 0 to
    70,000 elements (a fifth of them under 20, so below the rank count or inside one vector), dp 1-8 at
    a random rank, 1-6 micro-batches, four groups with random lr and weight-decay multipliers, and the
    hyper-parameters drawn too (lr, both betas, eps, weight decay, clip off or on), with gradient scales
    from far below to far above the clip threshold. Draws of one micro-batch take the micro-batch norm
    and the step that writes the gradient."""
    rng = np.random.default_rng(2024)
    k1 = 0
    for case in range(40):
        nt = int(rng.integers(1, 13))
        small = rng.random(nt) < 0.2
        numels = [int(x) for x in np.where(small, rng.integers(0, 20, nt), rng.integers(0, 70000, nt))]
        dp = int(rng.integers(1, 9))
        numels[0] += 1000 * dp  # at least one shard on every rank
        rank = int(rng.integers(0, dp))
        hp = dict(lr=float(10 ** rng.uniform(-5, -2)), beta1=float(rng.uniform(0.8, 0.99)),
                  beta2=float(rng.uniform(0.9, 0.9999)), eps=float(10 ** rng.uniform(-10, -6)),
                  weight_decay=float(rng.uniform(0.0, 0.2)), clip_grad=float(rng.choice([0.0, 0.5, 1.0, 5.0])))
        w = _custom(numels, [0] * nt, dp, rank, K=int(rng.integers(1, 7)), steps=2,
                    sigma=float(10 ** rng.uniform(-4, -1)), name="random%d" % case, hp=hp,
                    groups=[int(g) for g in rng.integers(0, 4, nt)],
                    lr_scale=[float(x) for x in rng.uniform(0.1, 2.0, 8)],
                    wd_scale=[float(x) for x in rng.choice([0.0, 0.5, 1.0, 2.0], 8)])
        # one micro-batch goes the bench's way for K = 1: its norm, then the step that writes the gradient
        res = run_parity(w, seed=case, micro_step=(w.micro_batches == 1))
        assert res["master"] == 0 and res["m"] == 0 and res["v"] == 0, (case, res)
        k1 += w.micro_batches == 1
    assert k1 >= 4  # several draws take the one-micro-batch path
