"""The one-micro-batch step in two passes (zero1_micro_norm + zero1_step_accumulate), on a GB300.

With one micro-batch the norm is taken from the micro-batch and the step writes
the gradient it uses. Against zero1_accumulate_norm (overwrite) + zero1_step on
the same inputs, bit for bit: the gradient, the norm record, master, m, v and
the bf16 copy, over several steps and sizes (empty, tiny and multi-tile
tensors with ragged tails), with the divisor and another ranks' share of the
sum of squares, parameter groups, no bf16 copy, 32- and 16-byte-aligned
gradient arenas, host-resident micro-batches, and a non-finite gradient (the
step is skipped, the gradient still written). Rejected arguments launch
nothing. The micro-batch norm's record equals the accumulating pass's and the
plain norm's on values that take its exact-square form, the general one, or
both in one tile.
"""
import ctypes

import numpy as np
import pytest
import torch

import zero_sharded_mixed_local_gb300 as z

pytestmark = pytest.mark.gpu

HP = z.Hparams(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


class _State:
    def __init__(self, plan, master, grad=None):
        self.plan = plan
        self.grad = plan.new_arena() if grad is None else grad
        self.master, self.m, self.v = master.clone(), plan.new_arena(), plan.new_arena()
        self.w = plan.new_arena(torch.bfloat16)
        self.ws, self.nout = plan.new_workspace(), z.new_norm_out()


def _setup(numels, no_decay=None, sigma=0.05, seed=0, groups=None):
    kw = {"groups": groups, "lr_scale": [1.0, 0.5, 2.0, 1.0, 1.0, 1.0, 1.0, 1.0],
          "wd_scale": [1.0, 0.0, 3.0, 1.0, 1.0, 1.0, 1.0, 1.0]} if groups else {"no_decay": no_decay}
    plan = z.Plan(numels, **kw)
    g = torch.Generator(device="cuda").manual_seed(seed)
    L = plan.layout()
    pad = torch.ones(plan.arena_numel, dtype=torch.bool, device="cuda")
    for o, c in zip(L.offsets, L.counts):
        pad[int(o):int(o) + int(c)] = False
    master = torch.randn(plan.arena_numel, device="cuda", generator=g) * 0.02
    master[pad] = 0.0

    def micro():
        x = (torch.randn(plan.arena_numel, device="cuda", generator=g) * sigma).to(torch.bfloat16)
        x[pad] = 0
        return x
    return plan, master, micro


def _two_calls(s, mb, t, divisor=1.0, extra=0.0, with_w=True):
    z.accumulate_norm(s.plan, s.grad, mb, s.ws, s.nout, overwrite_first=True, extra_sumsq=extra, divisor=divisor)
    z.step(s.plan, s.master, s.m, s.v, s.grad, s.w if with_w else None, HP, t, s.nout)


def _micro_pair(s, mb, t, divisor=1.0, extra=0.0, with_w=True):
    z.micro_norm(s.plan, mb, s.ws, s.nout, extra_sumsq=extra, divisor=divisor)
    z.step_accumulate(s.plan, s.master, s.m, s.v, s.grad, mb, s.w if with_w else None, HP, t, s.nout,
                      divisor=divisor)


def _same(a, b):
    torch.cuda.synchronize()
    # the records' bytes: a skipped step's sum of squares is NaN, which no float comparison equates
    assert bytes(a.nout[:z.NORM_OUT_BYTES].cpu().numpy()) == bytes(b.nout[:z.NORM_OUT_BYTES].cpu().numpy())
    for k in ("grad", "master", "m", "v", "w"):
        assert torch.equal(_bits(getattr(a, k)), _bits(getattr(b, k))), k


@pytest.mark.parametrize("divisor,extra", [(1.0, 0.0), (4.0, 0.0), (1.0, 3.5), (3.0, 0.25)])
def test_micro_pair_equals_accumulate_norm_and_step(divisor, extra):
    numels = [16384 * 3 + 8 * 5 + 3, 1000, 0, 1, 7, 77, 16384]
    plan, master, micro = _setup(numels, [0, 1, 0, 1, 0, 0, 1], sigma=0.05)
    a, b = _State(plan, master), _State(plan, master)
    for t in (1, 2, 3):
        mb = micro()
        _micro_pair(a, mb, t, divisor, extra)
        _two_calls(b, mb, t, divisor, extra)
        _same(a, b)
    assert z.read_norm(a.nout)["norm"] > 1.0  # clipping active


def test_micro_pair_with_groups_no_bf16_copy_and_a_narrow_gradient_arena():
    plan, master, micro = _setup([5000, 17, 16384 + 3, 64, 999], groups=[2, 1, 0, 2, 1], sigma=0.3, seed=4)
    back = torch.zeros(plan.arena_numel + 4, device="cuda")
    narrow = back[4:]  # 16 bytes past an aligned start: the 128-bit gradient stores
    assert narrow.data_ptr() % 32 == 16
    a, b, c = _State(plan, master, grad=narrow), _State(plan, master), _State(plan, master)
    for t in (1, 2):
        mb = micro()
        _micro_pair(a, mb, t, with_w=False)
        _micro_pair(c, mb, t)
        _two_calls(b, mb, t, with_w=False)
        assert torch.equal(_bits(a.grad), _bits(c.grad))
    for k in ("grad", "master", "m", "v"):
        assert torch.equal(_bits(getattr(a, k)), _bits(getattr(b, k))), k
        assert torch.equal(_bits(getattr(c, k)), _bits(getattr(b, k))), k
    assert not a.w.any() and torch.equal(_bits(c.w), _bits(c.master.to(torch.bfloat16)))


def test_micro_pair_reads_a_host_micro_batch():
    plan, master, micro = _setup([40000, 33], [0, 1], sigma=0.1, seed=5)
    a, b = _State(plan, master), _State(plan, master)
    mb = micro()
    _micro_pair(a, mb.cpu().pin_memory(), 1)
    _two_calls(b, mb, 1)
    _same(a, b)


def test_nonfinite_micro_batch_skips_the_step_and_still_writes_the_gradient():
    plan, master, micro = _setup([20000, 64], [0, 1], seed=6)
    a, b = _State(plan, master), _State(plan, master)
    mb = micro()
    _micro_pair(a, mb, 1)
    _two_calls(b, mb, 1)
    bad = micro()
    bad[123] = float("inf")
    _micro_pair(a, bad, 2)
    _two_calls(b, bad, 2)
    assert z.read_norm(a.nout)["status"] == z.ZERO1_ENONFINITE
    _same(a, b)
    assert torch.equal(_bits(a.grad), _bits(bad.float()))  # the gradient is the new micro-batch


def test_local_step_with_one_micro_batch_takes_the_micro_pair():
    """zero1_local_step with one micro-batch launches the micro-batch norm (2 kernels) and the step
    (1 kernel), and gives the two calls' results."""
    plan, master, micro = _setup([16384 * 2 + 5, 300], [0, 1], seed=7)
    a, b = _State(plan, master), _State(plan, master)
    mb = micro()
    before = z.launch_count()
    z.local_step(plan, a.grad, [mb], a.ws, a.nout, a.master, a.m, a.v, a.w, HP, 1)
    assert z.launch_count() - before == 3
    _two_calls(b, mb, 1)
    _same(a, b)


@pytest.mark.parametrize("kind", ["exact", "outside", "zeros", "large", "inf"])
@pytest.mark.parametrize("divisor", [1.0, 3.0])
def test_micro_norm_record_equals_the_accumulating_pass_on_any_bf16_values(kind, divisor):
    """Without a divisor the micro-batch norm drops the residual of squares it checks to be exact; the
    record stays the bits of zero1_accumulate_norm's pass and of zero1_grad_norm over the gradient it
    writes, whatever mix of exact and inexact squares (subnormals, zeros, overflowing sums) a tile
    holds.  With a divisor every square takes the general form."""
    from parity import bf16_norm_pattern
    numels = [16384 * 5 + 77, 1000, 16384 * 2, 3, 40000]
    plan, master, micro = _setup(numels, [0, 1, 0, 1, 0], sigma=0.05, seed=9)
    L = plan.layout()
    mb = bf16_norm_pattern(micro(), kind, torch.Generator(device="cuda").manual_seed(10))
    keep = torch.zeros(plan.arena_numel, dtype=torch.bool, device="cuda")
    for o, c in zip(L.offsets, L.counts):
        keep[int(o):int(o) + int(c)] = True
    mb[~keep] = 0  # the arena's padding stays zero
    a, b = _State(plan, master), _State(plan, master)
    z.micro_norm(plan, mb, a.ws, a.nout, divisor=divisor)
    z.accumulate_norm(plan, b.grad, mb, b.ws, b.nout, overwrite_first=True, divisor=divisor)
    c_out = z.new_norm_out()
    z.grad_norm(plan, b.grad, b.ws, c_out)
    torch.cuda.synchronize()
    ra, rb, rc = (bytes(r[:z.NORM_OUT_BYTES].cpu().numpy()) for r in (a.nout, b.nout, c_out))
    assert ra == rb == rc
    rec = z.read_norm(a.nout)
    if kind in ("large", "inf"):
        assert rec["status"] == z.ZERO1_ENONFINITE
    else:
        assert rec["status"] == 0
        ref = float(np.sum((b.grad.double() ** 2).cpu().numpy()))
        assert abs(rec["sumsq"] - ref) <= 1e-12 * ref


def test_micro_pair_rejects_bad_arguments_before_any_launch():
    lib = z.load_library()
    plan, master, micro = _setup([5000, 64], [0, 1], seed=8)
    s = _State(plan, master)
    mb = micro()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    hp = HP._c()
    before = z.launch_count()
    assert lib.zero1_micro_norm(plan.handle, mb.data_ptr() + 2, 1.0, 0.0, s.ws.data_ptr(), s.ws.numel(),
                                s.nout.data_ptr(), stream) == z.ZERO1_EALIGN
    assert lib.zero1_micro_norm(plan.handle, mb.data_ptr(), 0.0, 0.0, s.ws.data_ptr(), s.ws.numel(),
                                s.nout.data_ptr(), stream) == z.ZERO1_EINVAL
    assert lib.zero1_micro_norm(plan.handle, mb.data_ptr(), 1.0, 0.0, s.ws.data_ptr(), 0, s.nout.data_ptr(),
                                stream) == z.ZERO1_EINVAL
    args = [s.master.data_ptr(), s.m.data_ptr(), s.v.data_ptr(), s.grad.data_ptr()]
    assert lib.zero1_step_accumulate(plan.handle, *args, mb.data_ptr() + 2, 1.0, s.w.data_ptr(), ctypes.byref(hp), 1,
                                     s.nout.data_ptr(), stream) == z.ZERO1_EALIGN
    assert lib.zero1_step_accumulate(plan.handle, *args, mb.data_ptr(), float("nan"), s.w.data_ptr(),
                                     ctypes.byref(hp), 1, s.nout.data_ptr(), stream) == z.ZERO1_EINVAL
    assert lib.zero1_step_accumulate(plan.handle, *args, mb.data_ptr(), 1.0, s.w.data_ptr(), ctypes.byref(hp), 0,
                                     s.nout.data_ptr(), stream) == z.ZERO1_EINVAL
    assert z.launch_count() == before


def test_micro_pair_matches_the_oracle_on_the_toy_shard_with_one_micro_batch():
    """Every element of the toy shard with K = 1, five steps, through the bench's K = 1 path."""
    from parity import run_parity
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    w = get_workload("toy")
    w.micro_batches = 1
    w.grad_sigma = 0.05  # clipping active
    res = run_parity(w, steps=5, micro_step=True)
    assert res["master"] == 0 and res["m"] == 0 and res["v"] == 0
    assert res["norms"][0][3] < 1.0


def test_arena_calls_write_nothing_outside_their_buffers():
    """Every arena buffer sits between 64-element guard zones filled with a pattern (the buffer stays
    32-byte aligned); after zero1_accumulate (K = 3), the fused and the separate norm, the step, the
    micro-batch pair and one-call steps, with and without the bf16 copy and with a divisor, every guard
    is unchanged.  The sizes leave ragged tails in the last norm tile and the last block."""
    numels = [16384 * 2 + 8 * 3 + 5, 77, 1, 1000]
    plan, master, micro = _setup(numels, [0, 1, 0, 1], sigma=0.05, seed=12)
    n = plan.arena_numel
    G = 64

    def guarded(dtype, fill):
        back = torch.empty(n + 2 * G, dtype=dtype, device="cuda")
        back.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).fill_(fill)
        return back, back[G:G + n]

    bufs = {name: guarded(dt, fill) for name, dt, fill in (
        ("grad", torch.float32, 0x5A5A5A5A), ("master", torch.float32, 0x3C3C3C3C), ("m", torch.float32, 0x11111111),
        ("v", torch.float32, 0x22222222), ("w", torch.bfloat16, 0x7777))}
    for name in ("master", "m", "v", "grad"):
        bufs[name][1].copy_(master if name == "master" else torch.zeros_like(master))
    bufs["w"][1].zero_()
    mbs = [guarded(torch.bfloat16, 0x6666) for _ in range(3)]
    for (_, view) in mbs:
        view.copy_(micro())
    ws_back = torch.full((plan.new_workspace().numel() + 2 * 16,), 0x5B, dtype=torch.uint8, device="cuda")
    ws = ws_back[16:16 + plan.new_workspace().numel()]
    nout_back = torch.full((z.NORM_OUT_BYTES + 64,), 0x4D, dtype=torch.uint8, device="cuda")
    nout = nout_back[16:48]
    before = {k: b.clone() for k, (b, _) in bufs.items()}
    mb_before = [b.clone() for b, _ in mbs]
    ws_before, nout_before = ws_back.clone(), nout_back.clone()
    g, p, m_, v_, w_ = (bufs[k][1] for k in ("grad", "master", "m", "v", "w"))
    views = [v for _, v in mbs]
    z.accumulate(plan, g, views[0], overwrite_first=True)
    z.accumulate(plan, g, views[1], overwrite_first=False)
    z.accumulate_norm(plan, g, views[2], ws, nout, overwrite_first=False, divisor=3.0)
    z.grad_norm(plan, g, ws, nout)
    z.step(plan, p, m_, v_, g, w_, HP, 1, nout)
    z.step(plan, p, m_, v_, g, None, HP, 2, nout)
    z.micro_norm(plan, views[0], ws, nout, divisor=2.0)
    z.step_accumulate(plan, p, m_, v_, g, views[0], w_, HP, 3, nout, divisor=2.0)
    z.local_step(plan, g, views, ws, nout, p, m_, v_, w_, HP, 4)
    z.local_step(plan, g, views[:1], ws, nout, p, m_, v_, None, HP, 5)
    torch.cuda.synchronize()
    for k, (b, _) in bufs.items():
        assert torch.equal(b[:G], before[k][:G]) and torch.equal(b[G + n:], before[k][G + n:]), k
    for (b, _), b0 in zip(mbs, mb_before):
        assert torch.equal(b, b0)  # micro-batches are only read
    end = 16 + ws.numel()
    assert torch.equal(ws_back[:16], ws_before[:16]) and torch.equal(ws_back[end:], ws_before[end:])
    assert torch.equal(nout_back[:16], nout_before[:16]) and torch.equal(nout_back[48:], nout_before[48:])
