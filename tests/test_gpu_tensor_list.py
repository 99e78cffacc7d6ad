"""The tensor-list calls (one buffer per tensor shard, a run table walked by the
kernels) against the CPU oracle and against the arena calls, on a GB300.

The oracle sees the shards concatenated in model order with no padding, which
is exactly what the list kernels walk; gradients and the moments must match it
bit for bit, the norm within 1e-12 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_local_gb300 as z

from parity import u16

pytestmark = pytest.mark.gpu

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)
# sizes around every boundary the kernels have: 8-element vectors, 2048-element block
# passes, 16384-element runs; an empty tensor and one with fewer elements than ranks
NUMELS = [1000, 7, 4096, 33, 16385, 40000, 1, 0, 65539, 2, 49152, 16384 * 3 + 8]
NO_DECAY = [0, 1, 0, 1, 0, 0, 1, 0, 0, 1, 0, 0]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    z.load_library()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _buffers(counts, dtype, misaligned, dev):
    """One buffer per shard; with `misaligned`, each starts one element past a 16-byte
    boundary (a view into a larger allocation), which forces the element-wise path."""
    out = []
    for c in counts:
        c = int(c)
        if misaligned and c:
            out.append(torch.zeros(c + 8, dtype=dtype, device=dev)[1:1 + c])
        else:
            out.append(torch.zeros(c, dtype=dtype, device=dev))
    return out


class ListProblem:
    def __init__(self, numels, no_decay, dp=3, rank=1, misaligned=False, hp=None, seed=0, sigma=1e-3):
        self.dev = torch.device("cuda")
        self.hp = dict(hp or HP)
        self.no_decay = np.asarray(no_decay, np.uint8)
        self.plan = z.Plan(numels, self.no_decay, dp, rank)
        self.counts = self.plan.layout().counts
        self.gen = torch.Generator(device=self.dev).manual_seed(seed)
        self.sigma = sigma
        mk = lambda dt: _buffers(self.counts, dt, misaligned, self.dev)  # noqa: E731
        self.master, self.m, self.v, self.grad = mk(torch.float32), mk(torch.float32), mk(torch.float32), mk(
            torch.float32)
        self.w = mk(torch.bfloat16)
        for t, c, nd in zip(self.master, self.counts, self.no_decay):
            if c:
                t.copy_(torch.ones_like(t) if nd else torch.randn(int(c), generator=self.gen, device=self.dev) * 0.02)
        self.opt = z.ShardListAdamW(numels, self.no_decay, dp, rank, hparams=self.hp, master=self.master,
                                    exp_avg=self.m, exp_avg_sq=self.v, grad=self.grad, weight_bf16=self.w)
        self.misaligned = misaligned

    def micro(self):
        return [(torch.randn(int(c), generator=self.gen, device=self.dev) * self.sigma).to(torch.bfloat16)
                if c else torch.zeros(0, dtype=torch.bfloat16, device=self.dev) for c in self.counts]

    def micro_like(self, lst):
        """Same values in buffers with this problem's alignment."""
        out = _buffers(self.counts, torch.bfloat16, self.misaligned, self.dev)
        for a, b in zip(out, lst):
            a.copy_(b)
        return out

    def flat(self, lst):
        return torch.cat([t.reshape(-1) for t in lst]).cpu()


def _oracle_state(pb):
    return (pb.flat(pb.master).numpy().copy(), np.zeros(int(pb.counts.sum()), np.float32),
            np.zeros(int(pb.counts.sum()), np.float32))


def _eq(a, b):
    a = np.asarray(a)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("misaligned", [False, True])
def test_list_step_matches_the_oracle_bit_for_bit(misaligned):
    pb = ListProblem(NUMELS, NO_DECAY, misaligned=misaligned)
    P, M, V = _oracle_state(pb)
    n = P.size
    for t in range(1, 4):
        micros = [pb.micro_like(pb.micro()) for _ in range(2)]
        pb.opt.accumulate(micros[0])
        pb.opt.accumulate(micros[1], last=True)
        pb.opt.step()
        got = pb.opt.read_norm()
        G = np.zeros(n, np.float32)
        for k, mb in enumerate(micros):
            oracle.accumulate(G, u16(pb.flat(mb)), overwrite=(k == 0))
        assert _eq(pb.flat(pb.grad).numpy(), G), "gradient differs from the oracle at step %d" % t
        ref = oracle.sumsq(G)
        assert got["status"] == 0 and abs(got["sumsq"] - ref) <= 1e-12 * ref, (t, got["sumsq"], ref)
        ok, _, coef = oracle.clip_coef(ref, HP["clip_grad"])
        oracle.adamw(P, M, V, G, pb.counts, pb.no_decay, HP, t, coef)
    for name, lst, ref in (("master", pb.master, P), ("m", pb.m, M), ("v", pb.v, V)):
        assert _eq(pb.flat(lst).numpy(), ref), name
    assert np.array_equal(u16(pb.flat(pb.w)), oracle.bf16_rne(P))


def test_list_calls_equal_the_arena_calls():
    """No clipping (so both sides use coef 1): every state element bit-identical to the
    arena path's on the same values; the norms agree to 1e-12."""
    hp = dict(HP, clip_grad=0.0)
    pb = ListProblem(NUMELS, NO_DECAY, hp=hp, seed=3)
    arena = z.LocalShardAdamW(NUMELS, NO_DECAY, 3, 1, hparams=hp)
    for view, t in zip(arena.plan.shard_views(arena.master), pb.master):
        view.copy_(t)
    for step in range(2):
        micros = [pb.micro() for _ in range(3)]
        arenas = []
        for mb in micros:
            a = arena.plan.new_arena(torch.bfloat16)
            for view, t in zip(arena.plan.shard_views(a), mb):
                view.copy_(t)
            arenas.append(a)
        pb.opt.accumulate(micros[:2])
        pb.opt.accumulate(micros[2], last=True)
        arena.accumulate(arenas[:2])
        arena.accumulate(arenas[2], last=True)
        pb.opt.step()
        arena.step()
        a_norm, l_norm = arena.read_norm(), pb.opt.read_norm()
        assert abs(a_norm["sumsq"] - l_norm["sumsq"]) <= 1e-12 * a_norm["sumsq"]
    for name in ("grad", "master", "exp_avg", "exp_avg_sq", "weight_bf16"):
        views = arena.plan.shard_views(getattr(arena, name))
        for i, (a, b) in enumerate(zip(views, getattr(pb.opt, name))):
            assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                               b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)), (name, i)


def test_divisor_and_separate_norm_call():
    """Fused pass with a world-size divisor equals the oracle's sum then divide; the
    standalone norm call reproduces the fused record bit for bit, twice."""
    pb = ListProblem(NUMELS, NO_DECAY, dp=2, rank=0, seed=5, sigma=1e-2)
    micros = [pb.micro() for _ in range(2)]
    pb.opt.accumulate(micros[0])
    pb.opt.accumulate(micros[1], last=True, divisor=8.0)
    fused = pb.opt.read_norm()
    G = np.zeros(int(pb.counts.sum()), np.float32)
    for k, mb in enumerate(micros):
        oracle.accumulate(G, u16(pb.flat(mb)), overwrite=(k == 0))
    oracle.divide(G, 8.0)
    assert _eq(pb.flat(pb.grad).numpy(), G)
    ref = oracle.sumsq(G)
    assert abs(fused["sumsq"] - ref) <= 1e-12 * ref
    nout = z.new_norm_out()
    for _ in range(2):
        z.list_grad_norm(pb.opt.plan, pb.opt.table, pb.opt.pointer_lists["grad"], pb.opt.workspace, nout)
        again = z.read_norm(nout)
        assert again["sumsq"] == fused["sumsq"] and again["n_partials"] == fused["n_partials"]
    runs = int(np.sum((pb.counts + 16383) // 16384))
    assert fused["n_partials"] == runs


def test_nonfinite_gradient_skips_the_list_step():
    pb = ListProblem(NUMELS, NO_DECAY, seed=7)
    mb = pb.micro()
    mb[4][100] = float("inf")
    before = [t.clone() for t in pb.master]
    pb.opt.accumulate(mb, last=True)
    pb.opt.step()
    got = pb.opt.read_norm()
    assert got["status"] == z.ZERO1_ENONFINITE
    for a, b in zip(before, pb.master):
        assert torch.equal(a, b)
    assert all(int(t.abs().sum()) == 0 for t in pb.m if t.numel())


def test_list_step_without_bf16_copy():
    pb = ListProblem(NUMELS, NO_DECAY, seed=9)
    mb = pb.micro()
    pb.opt.accumulate(mb, last=True)
    L = pb.opt.pointer_lists
    twin = [t.clone() for t in pb.master]
    z.list_step(pb.opt.plan, pb.opt.table, L["master"], L["exp_avg"], L["exp_avg_sq"], L["grad"], None,
                z.Hparams(**HP), 1, pb.opt.norm_out)
    # the same step through the oracle on the cloned master
    G = pb.flat(pb.grad).numpy()
    P = torch.cat([t.reshape(-1) for t in twin]).cpu().numpy().copy()
    M = np.zeros_like(P)
    V = np.zeros_like(P)
    ref = oracle.sumsq(G)
    _, _, coef = oracle.clip_coef(ref, HP["clip_grad"])
    oracle.adamw(P, M, V, G, pb.counts, pb.no_decay, HP, 1, coef)
    assert _eq(pb.flat(pb.master).numpy(), P)
    assert all(int(t.view(torch.int16).abs().sum()) == 0 for t in pb.w if t.numel())  # no copy written


def test_parameter_groups_through_the_run_table():
    """Four groups with their own lr and weight-decay multipliers, interleaved in model
    order: each run steps with its tensor's group scalars."""
    groups = [0, 1, 2, 3, 0, 2, 1, 3, 2, 1, 0, 3]
    lr_scale = [1.0, 1.0, 0.25, 2.0, 1, 1, 1, 1]
    wd_scale = [1.0, 0.0, 1.0, 0.5, 1, 1, 1, 1]
    dev = torch.device("cuda")
    plan = z.Plan(NUMELS, dp_size=3, dp_rank=1, groups=groups, lr_scale=lr_scale, wd_scale=wd_scale)
    counts = plan.layout().counts
    g = torch.Generator(device=dev).manual_seed(13)
    master = [torch.randn(int(c), generator=g, device=dev) * 0.02 for c in counts]
    grads = [torch.randn(int(c), generator=g, device=dev) * 1e-2 for c in counts]
    m, v, w = plan.new_shards(), plan.new_shards(), plan.new_shards(torch.bfloat16)
    P = torch.cat(master).cpu().numpy().copy()
    G = torch.cat(grads).cpu().numpy().copy()
    M, V = np.zeros_like(P), np.zeros_like(P)
    lists = [z.PointerLists(plan, x, torch.float32) for x in (master, m, v, grads)]
    wl = z.PointerLists(plan, w, torch.bfloat16)
    table, ws, nout = plan.list_table(), plan.new_list_workspace(), z.new_norm_out()
    for t in (1, 2):
        z.list_grad_norm(plan, table, lists[3], ws, nout)
        z.list_step(plan, table, *lists, wl, z.Hparams(**HP), t, nout)
        ref = oracle.sumsq(G)
        _, _, coef = oracle.clip_coef(ref, HP["clip_grad"])
        oracle.adamw_scaled(P, M, V, G, counts, np.asarray(lr_scale)[groups], np.asarray(wd_scale)[groups], HP, t,
                            coef)
    assert _eq(torch.cat(master).cpu().numpy(), P) and _eq(torch.cat(m).cpu().numpy(), M)
    assert np.array_equal(u16(torch.cat(w)), oracle.bf16_rne(P))


def test_many_small_tensors_log_uniform():
    """3000 tensors with sizes log-uniform in [1, 2^16] (the ragged mix, scaled down),
    10% without decay, dp 2 rank 1, clipping active."""
    rng = np.random.default_rng(11)
    numels = np.floor(np.exp(rng.uniform(0, 16 * np.log(2), 3000))).astype(np.int64)
    no_decay = (rng.random(3000) < 0.1).astype(np.uint8)
    pb = ListProblem(numels, no_decay, dp=2, rank=1, seed=11, sigma=1e-2)
    P, M, V = _oracle_state(pb)
    for t in (1, 2):
        mb = pb.micro()
        pb.opt.accumulate(mb, last=True)
        pb.opt.step()
        got = pb.opt.read_norm()
        G = np.zeros(P.size, np.float32)
        oracle.accumulate(G, u16(pb.flat(mb)), overwrite=True)
        ref = oracle.sumsq(G)
        assert abs(got["sumsq"] - ref) <= 1e-12 * ref
        ok, norm, coef = oracle.clip_coef(ref, HP["clip_grad"])
        assert coef < 1.0  # clipping is active
        oracle.adamw(P, M, V, G, pb.counts, pb.no_decay, HP, t, coef)
    assert _eq(pb.flat(pb.master).numpy(), P) and _eq(pb.flat(pb.v).numpy(), V)
    assert np.array_equal(u16(pb.flat(pb.w)), oracle.bf16_rne(P))


def test_pointer_lists_are_checked():
    plan = z.Plan([64, 8], [0, 1], 1, 0)
    good = [torch.zeros(64, device="cuda"), torch.zeros(8, device="cuda")]
    with pytest.raises(ValueError):
        z.PointerLists(plan, [good[0], torch.zeros(9, device="cuda")], torch.float32)   # wrong length
    with pytest.raises(TypeError):
        z.PointerLists(plan, [good[0], good[1].to(torch.bfloat16)], torch.float32)     # wrong dtype
    with pytest.raises(ValueError):
        z.PointerLists(plan, [good[0]], torch.float32)                                   # wrong count
    with pytest.raises(ValueError):
        z.PointerLists(plan, [good[0], torch.zeros(16, device="cuda")[::2]], torch.float32)  # not contiguous
    pl = z.PointerLists(plan, good, torch.float32)
    assert pl.dev.cpu().tolist()[:2] == [good[0].data_ptr(), good[1].data_ptr()]
    # each call checks its lists against the plan's shard sizes, their dtype and list count, and
    # that the run table is the plan's own, before anything is launched
    other = z.Plan([64, 16], [0, 1], 1, 0)
    table, ws, nout = plan.list_table(), plan.new_list_workspace(), z.new_norm_out()
    foreign = z.PointerLists(other, [torch.zeros(64, device="cuda"), torch.zeros(16, device="cuda")], torch.float32)
    bf = z.PointerLists(plan, [t.to(torch.bfloat16) for t in good], torch.bfloat16)
    two = z.PointerLists(plan, [good, good], torch.float32)
    with pytest.raises(ValueError):
        z.list_grad_norm(plan, table, foreign, ws, nout)            # another plan's shard sizes
    with pytest.raises(TypeError):
        z.list_grad_norm(plan, table, bf, ws, nout)                 # bf16 shards as gradients
    with pytest.raises(ValueError):
        z.list_grad_norm(plan, other.list_table(), pl, ws, nout)    # another plan's run table
    with pytest.raises(ValueError):
        z.list_grad_norm(plan, table, pl, ws, nout[:16])            # short norm record
    with pytest.raises(ValueError):
        z.list_step(plan, table, two, pl, pl, pl, None, z.Hparams(), 1)   # two lists as the master
    with pytest.raises(TypeError):
        z.list_accumulate(plan, table, pl, pl)                      # fp32 shards as micro-batches
    z.list_grad_norm(plan, table, pl, ws, nout)                     # the right arguments pass
    assert z.read_norm(nout)["sumsq"] == 0.0


def test_llama8b_full_size_list_equals_arena():
    """The 1.0B-element Llama-3.1-8B dp8 rank-0 shard (291 tensors), one step through the
    arena calls and through the list calls on one allocation per tensor shard, then a second
    through both one-micro-batch pairs (the bench's K = 1 path): every element of every state
    buffer identical after each, the norms within 1e-12."""
    from zero_sharded_mixed_local_gb300.workloads import InputGenerator, Layout, get_workload
    dev = torch.device("cuda")
    w = get_workload("llama8b")
    plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank)
    L = plan.layout()
    gen = InputGenerator(w, Layout(L.counts, L.offsets, L.no_decay, L.arena_numel), dev, seed=w.seed)
    master = gen.master()
    m, v, grad, wbf = gen.zeros(), gen.zeros(), gen.zeros(), gen.zeros(torch.bfloat16)
    micro = gen.micro_grads()[0]
    split = lambda buf: [t.clone() for t in plan.shard_views(buf)]  # noqa: E731
    lm, lmm, lv, lg, lw, lmic = split(master), split(m), split(v), split(grad), split(wbf), split(micro)
    hp = z.Hparams(**w.hp)
    ws, nout = plan.new_workspace(dev), z.new_norm_out(dev)
    z.accumulate_norm(plan, grad, micro, ws, nout)
    z.step(plan, master, m, v, grad, wbf, hp, 1, nout)
    a_norm = z.read_norm(nout)
    del micro
    lists = [z.PointerLists(plan, x, torch.float32) for x in (lm, lmm, lv, lg)]
    wl, ml = z.PointerLists(plan, lw, torch.bfloat16), z.PointerLists(plan, lmic, torch.bfloat16)
    table, lws, lnout = plan.list_table(), plan.new_list_workspace(), z.new_norm_out()
    z.list_accumulate_norm(plan, table, lists[3], ml, lws, lnout)
    z.list_step(plan, table, *lists, wl, hp, 1, lnout)
    l_norm = z.read_norm(lnout)
    assert abs(a_norm["sumsq"] - l_norm["sumsq"]) <= 1e-12 * a_norm["sumsq"]
    for arena, shards in ((grad, lg), (master, lm), (m, lmm), (v, lv), (wbf, lw)):
        for i, (a, b) in enumerate(zip(plan.shard_views(arena), shards)):
            assert torch.equal(a, b), i
    # step 2 as the bench runs K = 1: the micro-batch norm, then the step that writes the gradient
    micro = gen.micro_grads()[0]
    lmic2 = split(micro)
    ml2 = z.PointerLists(plan, lmic2, torch.bfloat16)
    z.micro_norm(plan, micro, ws, nout)
    z.step_accumulate(plan, master, m, v, grad, micro, wbf, hp, 2, nout)
    a_norm = z.read_norm(nout)
    z.list_micro_norm(plan, table, ml2, lws, lnout)
    z.list_step_accumulate(plan, table, *lists, ml2, wl, hp, 2, lnout)
    l_norm = z.read_norm(lnout)
    assert abs(a_norm["sumsq"] - l_norm["sumsq"]) <= 1e-12 * a_norm["sumsq"]
    for arena, shards in ((grad, lg), (master, lm), (m, lmm), (v, lv), (wbf, lw)):
        for i, (a, b) in enumerate(zip(plan.shard_views(arena), shards)):
            assert torch.equal(a, b), ("micro pair", i)


@pytest.mark.parametrize("guard", [64, 65])
def test_list_calls_write_nothing_outside_the_shards(guard):
    """Every shard buffer sits between guard zones filled with a pattern (64 elements keeps the
    shards 16-byte aligned, 65 forces the element-wise path); after every list call has run,
    the guards are unchanged.  Sizes cover partial last vectors and runs."""
    numels = [1000, 7, 16384 + 9, 33, 2, 16384 * 2 + 24]
    nd = [0, 1, 0, 1, 1, 0]
    plan = z.Plan(numels, nd, 3, 1)
    counts = [int(c) for c in plan.layout().counts]
    G = guard
    g = torch.Generator(device="cuda").manual_seed(17)
    bufs = {}

    def guarded(name, dtype, fill=None):
        out = []
        for i, c in enumerate(counts):
            buf = torch.empty(c + 2 * G, dtype=dtype, device="cuda")
            buf.view(torch.uint8).fill_(0xA5)
            mid = buf[G:G + c]
            if fill is None:
                mid.zero_()
            else:
                mid.copy_(fill(c))
            out.append((buf, mid))
        bufs[name] = out
        return [mid for _, mid in out]

    rnd = lambda s: (lambda c: torch.randn(c, device="cuda", generator=g) * s)  # noqa: E731
    grad = guarded("grad", torch.float32)
    master = guarded("master", torch.float32, rnd(0.02))
    m, v = guarded("m", torch.float32), guarded("v", torch.float32)
    w = guarded("w", torch.bfloat16)
    mb = guarded("mb", torch.bfloat16, rnd(0.1))
    mb2 = guarded("mb2", torch.bfloat16, rnd(0.1))
    L = {k: z.PointerLists(plan, x, torch.float32) for k, x in (("grad", grad), ("master", master), ("m", m), ("v", v))}
    wl = z.PointerLists(plan, w, torch.bfloat16)
    one, two = z.PointerLists(plan, mb, torch.bfloat16), z.PointerLists(plan, [mb, mb2], torch.bfloat16)
    table, ws, nout = plan.list_table(), plan.new_list_workspace(), z.new_norm_out()
    z.list_accumulate(plan, table, L["grad"], one)
    z.list_accumulate(plan, table, L["grad"], two, overwrite_first=False)
    z.list_accumulate(plan, table, L["grad"], two, overwrite_first=True)
    z.list_accumulate_norm(plan, table, L["grad"], one, ws, nout, overwrite_first=False, divisor=3.0)
    z.list_accumulate_norm(plan, table, L["grad"], one, ws, nout, overwrite_first=True)
    z.list_grad_norm(plan, table, L["grad"], ws, nout)
    z.list_step(plan, table, L["master"], L["m"], L["v"], L["grad"], wl, z.Hparams(), 1, nout)
    z.list_step(plan, table, L["master"], L["m"], L["v"], L["grad"], None, z.Hparams(), 2, nout)
    torch.cuda.synchronize()
    assert z.read_norm(nout)["status"] == 0
    for name, lst in bufs.items():
        for i, (buf, mid) in enumerate(lst):
            raw = buf.view(torch.uint8)
            eb = buf.element_size()
            head, tail = raw[:G * eb], raw[(G + mid.numel()) * eb:]
            assert bool((head == 0xA5).all()) and bool((tail == 0xA5).all()), (name, i)


@pytest.mark.parametrize("K", [2, 3, 5, 8, 9])
@pytest.mark.parametrize("misaligned", [False, True])
def test_k_way_list_pass_matches_the_oracle(K, misaligned):
    """All K micro-batch lists in one list_accumulate_norm call (the K-specialised kernels for
    K <= 8, the general one above), and in one list_accumulate call, aligned and misaligned."""
    pb = ListProblem(NUMELS, NO_DECAY, misaligned=misaligned, seed=20 + K, sigma=0.3)
    micros = [pb.micro_like(pb.micro()) for _ in range(K)]
    G = np.zeros(int(pb.counts.sum()), np.float32)
    for k, mb in enumerate(micros):
        oracle.accumulate(G, u16(pb.flat(mb)), overwrite=(k == 0))
    pl = z.PointerLists(pb.opt.plan, micros, torch.bfloat16)
    gl = pb.opt.pointer_lists["grad"]
    z.list_accumulate_norm(pb.opt.plan, pb.opt.table, gl, pl, pb.opt.workspace, pb.opt.norm_out, overwrite_first=True,
                           divisor=2.0)
    got = pb.opt.read_norm()
    Gd = G.copy()
    oracle.divide(Gd, 2.0)
    assert _eq(pb.flat(pb.grad).numpy(), Gd)
    ref = oracle.sumsq(Gd)
    assert abs(got["sumsq"] - ref) <= 1e-12 * ref
    z.list_accumulate(pb.opt.plan, pb.opt.table, gl, pl, overwrite_first=True)
    assert _eq(pb.flat(pb.grad).numpy(), G)


def test_list_tensor_beyond_2_to_32_elements():
    """Maximum size through the list calls: one shard of 2^32 + 2^20 + 5 elements (run offsets
    past 2^32) plus a 3-element excluded one, gradients all 2^-8, so the sum of squares is
    N * 2^-16 exactly; elements around 2^31, 2^32 and the tail are stepped by the oracle.  Through
    the two-pass list calls, then through the list micro-batch pair on the same buffers."""
    n0 = (1 << 32) + (1 << 20) + 5
    plan = z.Plan([n0, 3], [0, 1], 1, 0)
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(4)
    master = [torch.empty(n0, device=dev).normal_(0.0, 0.02, generator=g), torch.ones(3, device=dev)]
    m = [torch.zeros(n0, device=dev), torch.zeros(3, device=dev)]
    v = [torch.zeros(n0, device=dev), torch.zeros(3, device=dev)]
    grad = [torch.empty(n0, device=dev), torch.empty(3, device=dev)]
    w = [torch.zeros(n0, dtype=torch.bfloat16, device=dev), torch.zeros(3, dtype=torch.bfloat16, device=dev)]
    mb = [torch.full((n0,), 2.0 ** -8, dtype=torch.bfloat16, device=dev),
          torch.full((3,), 2.0 ** -8, dtype=torch.bfloat16, device=dev)]
    idx = np.unique(np.concatenate([np.arange(e, e + 24) for e in ((1 << 31) - 12, (1 << 32) - 12, n0 - 24)] +
                                   [np.random.default_rng(1).integers(0, n0, 100000)]))
    it = torch.from_numpy(idx).to(dev)
    P0 = np.concatenate([master[0][it].cpu().numpy(), master[1].cpu().numpy()])
    L = [z.PointerLists(plan, x, torch.float32) for x in (master, m, v, grad)]
    wl, ml = z.PointerLists(plan, w, torch.bfloat16), z.PointerLists(plan, mb, torch.bfloat16)
    table, ws, nout = plan.list_table(), plan.new_list_workspace(), z.new_norm_out()
    z.list_accumulate_norm(plan, table, L[3], ml, ws, nout)
    z.list_step(plan, table, *L, wl, z.Hparams(**HP), 1, nout)
    got = z.read_norm(nout)
    N = n0 + 3
    assert got["status"] == 0 and got["sumsq"] == N * 2.0 ** -16, got
    G = np.concatenate([grad[0][it].cpu().numpy(), grad[1].cpu().numpy()])
    assert np.all(G == np.float32(2.0 ** -8))
    _, _, coef = oracle.clip_coef(N * 2.0 ** -16, HP["clip_grad"])
    P, M, V = P0.copy(), np.zeros_like(P0), np.zeros_like(P0)
    oracle.adamw(P, M, V, G, [idx.size, 3], [0, 1], HP, 1, coef)
    for name, lst, ref in (("master", master, P), ("m", m, M), ("v", v, V)):
        gotv = np.concatenate([lst[0][it].cpu().numpy(), lst[1].cpu().numpy()])
        assert np.array_equal(gotv.view(np.uint32), ref.view(np.uint32)), name
    wv = torch.cat([w[0][it], w[1]])
    assert np.array_equal(u16(wv), oracle.bf16_rne(P))
    # the same step through the list micro-batch pair, on the same buffers restored to the initial state
    g = torch.Generator(device=dev).manual_seed(4)
    master[0].normal_(0.0, 0.02, generator=g)
    master[1].fill_(1.0)
    assert np.array_equal(np.concatenate([master[0][it].cpu().numpy(), master[1].cpu().numpy()]), P0)
    for x in m + v + w:
        x.zero_()
    for x in grad:
        x.fill_(float("nan"))
    z.list_micro_norm(plan, table, ml, ws, nout)
    z.list_step_accumulate(plan, table, *L, ml, wl, z.Hparams(**HP), 1, nout)
    got = z.read_norm(nout)
    assert got["status"] == 0 and got["sumsq"] == N * 2.0 ** -16, got
    assert np.all(np.concatenate([grad[0][it].cpu().numpy(), grad[1].cpu().numpy()]) == np.float32(2.0 ** -8))
    for name, lst, ref in (("master", master, P), ("m", m, M), ("v", v, V)):
        gotv = np.concatenate([lst[0][it].cpu().numpy(), lst[1].cpu().numpy()])
        assert np.array_equal(gotv.view(np.uint32), ref.view(np.uint32)), name
    assert np.array_equal(u16(torch.cat([w[0][it], w[1]])), oracle.bf16_rne(P))
    del master, m, v, grad, w, mb, L, wl, ml
    torch.cuda.empty_cache()


def test_ragged_full_size_list_equals_arena():
    """The 20,000-tensor ragged list (dp2 rank 1, 2.74e9 elements), one step (two micro-batches)
    through the arena calls and through the list calls on one allocation per shard: every
    element of every state buffer identical, the norms within 1e-12 (clipping active)."""
    from zero_sharded_mixed_local_gb300.workloads import InputGenerator, Layout, get_workload
    dev = torch.device("cuda")
    w = get_workload("ragged")
    w.micro_batches = 2
    plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank)
    L = plan.layout()
    gen = InputGenerator(w, Layout(L.counts, L.offsets, L.no_decay, L.arena_numel), dev, seed=w.seed)
    master = gen.master()
    m, v, grad, wbf = gen.zeros(), gen.zeros(), gen.zeros(), gen.zeros(torch.bfloat16)
    micros = gen.micro_grads()
    split = lambda buf: [t.clone() for t in plan.shard_views(buf)]  # noqa: E731
    lm, lmm, lv, lg, lw = split(master), split(m), split(v), split(grad), split(wbf)
    lmic = [split(mb) for mb in micros]
    hp = z.Hparams(**w.hp)
    ws, nout = plan.new_workspace(dev), z.new_norm_out(dev)
    z.accumulate(plan, grad, micros[0])
    z.accumulate_norm(plan, grad, micros[1], ws, nout, overwrite_first=False)
    z.step(plan, master, m, v, grad, wbf, hp, 1, nout)
    a_norm = z.read_norm(nout)
    del micros
    lists = [z.PointerLists(plan, x, torch.float32) for x in (lm, lmm, lv, lg)]
    wl = z.PointerLists(plan, lw, torch.bfloat16)
    ml = [z.PointerLists(plan, x, torch.bfloat16) for x in lmic]
    table, lws, lnout = plan.list_table(), plan.new_list_workspace(), z.new_norm_out()
    z.list_accumulate(plan, table, lists[3], ml[0])
    z.list_accumulate_norm(plan, table, lists[3], ml[1], lws, lnout, overwrite_first=False)
    z.list_step(plan, table, *lists, wl, hp, 1, lnout)
    l_norm = z.read_norm(lnout)
    assert a_norm["norm"] > 1.0  # clipping active
    assert abs(a_norm["sumsq"] - l_norm["sumsq"]) <= 1e-12 * a_norm["sumsq"]
    for arena, shards in ((grad, lg), (master, lm), (m, lmm), (v, lv), (wbf, lw)):
        flat_a = torch.cat([x for x in plan.shard_views(arena) if x.numel()])
        flat_l = torch.cat([x for x in shards if x.numel()])
        assert torch.equal(flat_a, flat_l)
        del flat_a, flat_l
    del master, m, v, grad, wbf, lm, lmm, lv, lg, lw, lmic, lists, wl, ml
    torch.cuda.empty_cache()


def test_random_list_configurations_match_the_oracle():
    """Thirty seeded random lists through ShardListAdamW, with buffers aligned or one element off a
    16-byte boundary. Each has 1-10 tensors of 0 to 50,000 elements (a fifth under 20), a random
    no-decay set, dp 1-8 at a random rank, 1-5 micro-batches, random hyper-parameters and gradient
    scales. Over two steps, the gradient, the norm, master, m, v and the bf16 copy are checked against
    the oracle fed the shards concatenated in model order. Half of the one-micro-batch draws take
    ShardListAdamW.step_from (the micro-batch norm and the list step that writes the gradient)."""
    rng = np.random.default_rng(77)
    n_micro_pair = 0
    for case in range(30):
        nt = int(rng.integers(1, 11))
        small = rng.random(nt) < 0.2
        numels = [int(x) for x in np.where(small, rng.integers(0, 20, nt), rng.integers(0, 50000, nt))]
        dp = int(rng.integers(1, 9))
        numels[0] += 1000 * dp  # at least one shard on every rank
        rank = int(rng.integers(0, dp))
        no_decay = [int(x) for x in rng.random(nt) < 0.3]
        hp = dict(lr=float(10 ** rng.uniform(-5, -2)), beta1=float(rng.uniform(0.8, 0.99)),
                  beta2=float(rng.uniform(0.9, 0.9999)), eps=float(10 ** rng.uniform(-10, -6)),
                  weight_decay=float(rng.uniform(0.0, 0.2)), clip_grad=float(rng.choice([0.0, 0.5, 1.0, 5.0])))
        pb = ListProblem(numels, no_decay, dp=dp, rank=rank, misaligned=bool(rng.random() < 0.5), hp=hp, seed=case,
                         sigma=float(10 ** rng.uniform(-4, -1)))
        K = int(rng.integers(1, 6))
        P, M, V = _oracle_state(pb)
        micro_pair = K == 1 and case % 2 == 0
        n_micro_pair += micro_pair
        for t in (1, 2):
            micros = [pb.micro_like(pb.micro()) for _ in range(K)]
            if micro_pair:  # the micro-batch's norm, then the list step that writes the gradient
                pb.opt.step_from(micros[0])
            else:
                for k, mb in enumerate(micros):
                    pb.opt.accumulate(mb, last=(k == K - 1))
                pb.opt.step()
            got = pb.opt.read_norm()
            G = np.zeros(P.size, np.float32)
            for k, mb in enumerate(micros):
                oracle.accumulate(G, u16(pb.flat(mb)), overwrite=(k == 0))
            assert _eq(pb.flat(pb.grad).numpy(), G), (case, t)
            ref = oracle.sumsq(G)
            assert got["status"] == 0 and abs(got["sumsq"] - ref) <= 1e-12 * ref, (case, t, got["sumsq"], ref)
            ok, _, coef = oracle.clip_coef(ref, hp["clip_grad"])
            assert ok
            oracle.adamw(P, M, V, G, pb.counts, pb.no_decay, hp, t, coef)
        for name, lst, ref in (("master", pb.master, P), ("m", pb.m, M), ("v", pb.v, V)):
            assert _eq(pb.flat(lst).numpy(), ref), (case, name)
        assert np.array_equal(u16(pb.flat(pb.w)), oracle.bf16_rne(P)), case
    assert n_micro_pair >= 2, n_micro_pair  # draws that take the one-micro-batch list pair


@pytest.mark.parametrize("misaligned", [False, True])
def test_list_micro_pair_equals_accumulate_norm_and_step(misaligned):
    """One micro-batch over the tensor lists: list_micro_norm + list_step_accumulate (the norm from
    the micro-batch, then the step that writes the gradients) against list_accumulate_norm +
    list_step, bit for bit: every gradient, master, m, v and bf16 shard and the norm record, over
    three steps with clipping active, with the divisor on the last; the element-wise path when every
    buffer sits one element off a 16-byte boundary."""
    a = ListProblem(NUMELS, NO_DECAY, misaligned=misaligned, seed=11, sigma=0.05)
    b = ListProblem(NUMELS, NO_DECAY, misaligned=misaligned, seed=11, sigma=0.05)
    hp = z.Hparams(**HP)
    for t in (1, 2, 3):
        div = 2.0 if t == 3 else 1.0
        mb = a.micro()
        ap, bp = a.opt.plan, b.opt.plan  # the plans whose run tables the optimizers uploaded
        pa = z.PointerLists(ap, a.micro_like(mb), torch.bfloat16)
        pb = z.PointerLists(bp, b.micro_like(mb), torch.bfloat16)
        La, Lb = a.opt.pointer_lists, b.opt.pointer_lists
        z.list_micro_norm(ap, a.opt.table, pa, a.opt.workspace, a.opt.norm_out, divisor=div)
        z.list_step_accumulate(ap, a.opt.table, La["master"], La["exp_avg"], La["exp_avg_sq"], La["grad"], pa,
                               La["weight_bf16"], hp, t, a.opt.norm_out, divisor=div)
        z.list_accumulate_norm(bp, b.opt.table, Lb["grad"], pb, b.opt.workspace, b.opt.norm_out, divisor=div)
        z.list_step(bp, b.opt.table, Lb["master"], Lb["exp_avg"], Lb["exp_avg_sq"], Lb["grad"], Lb["weight_bf16"],
                    hp, t, b.opt.norm_out)
        torch.cuda.synchronize()
        assert bytes(a.opt.norm_out[:24].cpu().numpy()) == bytes(b.opt.norm_out[:24].cpu().numpy())
        assert z.read_norm(a.opt.norm_out)["norm"] > 1.0
    for name in ("grad", "master", "m", "v"):
        for x, y in zip(getattr(a, name), getattr(b, name)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), name
    for x, y in zip(a.w, b.w):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("kind", ["exact", "outside", "zeros", "large", "inf"])
@pytest.mark.parametrize("divisor", [1.0, 3.0])
def test_list_micro_norm_record_equals_the_accumulating_pass_on_any_bf16_values(kind, divisor):
    """The list micro-batch norm (exact-square form on full runs without a divisor) gives the record
    of list_accumulate_norm's one-micro-batch pass, bit for bit, whatever mix of exact and inexact
    squares the runs hold."""
    from parity import bf16_norm_pattern
    a = ListProblem(NUMELS, NO_DECAY, seed=13, sigma=0.05)
    gen = torch.Generator(device="cuda").manual_seed(14)
    mb = [bf16_norm_pattern(t, kind, gen) for t in a.micro()]
    pl = a.opt.plan
    pm = z.PointerLists(pl, mb, torch.bfloat16)
    L = a.opt.pointer_lists
    other = z.new_norm_out()
    z.list_micro_norm(pl, a.opt.table, pm, a.opt.workspace, a.opt.norm_out, divisor=divisor)
    torch.cuda.synchronize()
    z.list_accumulate_norm(pl, a.opt.table, L["grad"], pm, a.opt.workspace, other, divisor=divisor)
    torch.cuda.synchronize()
    assert bytes(a.opt.norm_out[:24].cpu().numpy()) == bytes(other[:24].cpu().numpy())
    rec = z.read_norm(other)
    assert (rec["status"] == z.ZERO1_ENONFINITE) == (kind in ("large", "inf"))


def test_list_micro_pair_skips_on_a_nonfinite_gradient_and_still_writes_it():
    a = ListProblem(NUMELS, NO_DECAY, seed=12)
    mb = a.micro()
    mb[3][2] = float("nan")
    before = [t.clone() for t in a.master]
    assert a.opt.step_from(mb, check_finite=True) is False and a.opt.t == 0
    for x, y in zip(a.master, before):
        assert torch.equal(x, y)
    for g, m in zip(a.grad, mb):
        assert torch.equal(g.view(torch.int32), m.float().view(torch.int32))  # NaN included


def test_step_from_equals_accumulate_then_step_and_the_arena_form():
    """ShardListAdamW.step_from (one micro-batch, then three) against accumulate(last=True) + step()
    and, for one micro-batch, against the arena pair on the same values."""
    a = ListProblem(NUMELS, NO_DECAY, seed=13, sigma=0.05)
    b = ListProblem(NUMELS, NO_DECAY, seed=13, sigma=0.05)
    arena = z.LocalShardAdamW(NUMELS, a.no_decay, 3, 1, hparams=a.hp)
    for t0, o0 in zip(a.master, a.plan.shard_views(arena.master)):
        o0.copy_(t0)
    for t in (1, 2):
        mb = a.micro()
        a.opt.step_from(mb)
        b.opt.accumulate(mb, last=True)
        b.opt.step()
        am = a.plan.new_arena(torch.bfloat16)
        for o, x in zip(a.plan.shard_views(am), mb):
            o.copy_(x)
        arena.step_from(am)
    mbs = [a.micro() for _ in range(3)]
    a.opt.step_from(mbs)
    b.opt.accumulate(mbs, last=True)
    b.opt.step()
    for name in ("grad", "master", "m", "v"):
        for x, y in zip(getattr(a, name), getattr(b, name)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), name
    a2 = ListProblem(NUMELS, NO_DECAY, seed=13, sigma=0.05)  # the arena after the two one-micro-batch steps
    for t in (1, 2):
        a2.opt.step_from(a2.micro())
    for x, y in zip(a2.master, a.plan.shard_views(arena.master)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
