"""zero1_local_step, the whole local step in one call, on a GB300.

It must equal zero1_accumulate_norm (every micro-batch, the first overwriting)
followed by zero1_step, bit for bit: gradient, norm record, master, m, v and
the bf16 copy, with and without the divisor, the other ranks' share of the sum
of squares and parameter groups; it must match the oracle; and a rejected
argument of either pass must leave every buffer untouched with no kernel
launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_local_gb300 as z

from parity import MAX_ULP, Problem, oracle_grad, ulp_diff

pytestmark = pytest.mark.gpu

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _pair(numels, no_decay, K, sigma, seed=0, **plan_kw):
    plan = z.Plan(numels, no_decay, **plan_kw) if plan_kw else z.Plan(numels, no_decay)
    g = torch.Generator(device="cuda").manual_seed(seed)
    master = torch.randn(plan.arena_numel, device="cuda", generator=g) * 0.02
    L = plan.layout()
    pad = torch.ones(plan.arena_numel, dtype=torch.bool, device="cuda")
    for o, c in zip(L.offsets, L.counts):
        pad[int(o):int(o) + int(c)] = False
    master[pad] = 0.0

    def state():
        return {"grad": plan.new_arena(), "master": master.clone(), "m": plan.new_arena(), "v": plan.new_arena(),
                "w": plan.new_arena(torch.bfloat16), "ws": plan.new_workspace(), "nout": z.new_norm_out()}

    def micros():
        out = []
        for _ in range(K):
            x = (torch.randn(plan.arena_numel, device="cuda", generator=g) * sigma).to(torch.bfloat16)
            x[pad] = 0
            out.append(x)
        return out
    return plan, state(), state(), micros


@pytest.mark.parametrize("K,divisor,extra", [(1, 1.0, 0.0), (3, 1.0, 0.0), (4, 8.0, 2.5), (16, 3.0, 0.0)])
def test_local_step_equals_the_two_calls(K, divisor, extra):
    numels = [16384 * 3 + 8 * 5 + 3, 1000, 77, 1, 0, 4096]
    plan, one, two, micros = _pair(numels, [0, 1, 0, 1, 0, 0], K, 0.05)
    hp = z.Hparams(**HP)
    for t in (1, 2, 3):
        mb = micros()
        z.local_step(plan, one["grad"], mb, one["ws"], one["nout"], one["master"], one["m"], one["v"], one["w"], hp,
                     t, extra_sumsq=extra, divisor=divisor)
        z.accumulate_norm(plan, two["grad"], mb, two["ws"], two["nout"], overwrite_first=True, extra_sumsq=extra,
                          divisor=divisor)
        z.step(plan, two["master"], two["m"], two["v"], two["grad"], two["w"], hp, t, two["nout"])
        assert z.read_norm(one["nout"]) == z.read_norm(two["nout"])
    for k in ("grad", "master", "m", "v", "w"):
        assert torch.equal(_bits(one[k]), _bits(two[k])), k


def test_local_step_with_groups_matches_the_oracle():
    """Every element, three steps of the toy shard through LocalShardAdamW.step_from with
    clipping active, against the oracle."""
    pb = Problem("toy")
    w = pb.w
    opt = z.LocalShardAdamW(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank, hparams=pb.hp)
    opt.master.copy_(pb.master)
    n = pb.n
    P = pb.master.cpu().numpy().copy()
    M, V = np.zeros(n, np.float32), np.zeros(n, np.float32)
    lr_scale, wd_scale = w.group_scales()
    counts = np.array([pb.group1, n - pb.group1] + [0] * 6, np.int64)
    for t in (1, 2, 3):
        micros = [m * 40 for m in pb.gen.micro_grads()]  # clip active
        opt.step_from(micros)
        G = oracle_grad(n, [m.view(torch.int16).cpu().numpy().view(np.uint16) for m in micros])
        assert np.array_equal(opt.grad.cpu().numpy().view(np.uint32), G.view(np.uint32))
        ok, norm, coef = oracle.clip_coef(oracle.sumsq(G), w.hp["clip_grad"])
        assert ok and coef < 1.0
        oracle.adamw_scaled(P, M, V, G, counts, lr_scale, wd_scale, w.hp, t, coef)
    for name, a, ref in (("master", opt.master, P), ("m", opt.exp_avg, M), ("v", opt.exp_avg_sq, V)):
        assert int(ulp_diff(a.cpu().numpy(), ref).max()) <= MAX_ULP, name
    assert torch.equal(_bits(opt.weight_bf16), _bits(opt.master.to(torch.bfloat16)))
    assert opt.t == 3


def test_local_step_rejects_before_any_launch():
    """A bad argument of the second pass (a misaligned master, a step count of 0) is refused
    before the first pass launches: no kernel runs and the gradient is untouched."""
    lib = z.load_library()
    plan, one, _, micros = _pair([5000, 64], [0, 1], 2, 0.05)
    mb = micros()
    one["grad"].fill_(7.0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    arr = (ctypes.c_void_p * 2)(*[m.data_ptr() for m in mb])
    hp = z.Hparams(**HP)._c()

    def call(master_ptr, t):
        return lib.zero1_local_step(plan.handle, one["grad"].data_ptr(), arr, 2, 1.0, 0.0, one["ws"].data_ptr(),
                                    one["ws"].numel(), one["nout"].data_ptr(), master_ptr, one["m"].data_ptr(),
                                    one["v"].data_ptr(), one["w"].data_ptr(), ctypes.byref(hp), t, stream)

    before = z.launch_count()
    assert call(one["master"].data_ptr() + 4, 1) == z.ZERO1_EALIGN
    assert call(one["master"].data_ptr(), 0) == z.ZERO1_EINVAL
    assert z.launch_count() == before
    torch.cuda.synchronize()
    assert bool((one["grad"] == 7.0).all())
    assert call(one["master"].data_ptr(), 1) == z.ZERO1_OK
    assert z.launch_count() == before + 3  # the K-way pass, its final reduction, the step
