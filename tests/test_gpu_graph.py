"""The local step captured as CUDA graphs (StepGraph over zero1_step_dev, and over
zero1_list_step_dev for the tensor-list path): the same results, bit for bit, as
the eager calls, while the step count and the learning rate change between
replays."""
import pytest
import torch

import zero_sharded_mixed_local_gb300 as z
from zero_sharded_mixed_local_gb300.workloads import get_workload

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _opt(w, seed):
    opt = z.LocalShardAdamW(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank, hparams=w.hp)
    g = torch.Generator(device="cuda").manual_seed(seed)
    L = opt.plan.layout()
    for o, c in zip(L.offsets, L.counts):
        opt.master[int(o):int(o) + int(c)].normal_(0.0, 0.02, generator=g)
    return opt


def test_step_dev_equals_step():
    w = get_workload("toy")
    outs = []
    for dev_scalars in (False, True):
        opt = _opt(w, 1)
        g = torch.Generator(device="cuda").manual_seed(2)
        mb = (torch.randn(opt.plan.arena_numel, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
        L = opt.plan.layout()
        pad = torch.ones(opt.plan.arena_numel, dtype=torch.bool, device="cuda")
        for o, c in zip(L.offsets, L.counts):
            pad[int(o):int(o) + int(c)] = False
        mb[pad] = 0
        z.accumulate_norm(opt.plan, opt.grad, mb, opt.workspace, opt.norm_out)
        hp = z.Hparams(**w.hp)
        for t in (1, 2, 7):
            if dev_scalars:
                sc = torch.frombuffer(bytearray(z.step_scalars(opt.plan, hp, t)), dtype=torch.uint8).cuda()
                z.step_dev(opt.plan, opt.master, opt.exp_avg, opt.exp_avg_sq, opt.grad, opt.weight_bf16, sc,
                           opt.norm_out)
            else:
                z.step(opt.plan, opt.master, opt.exp_avg, opt.exp_avg_sq, opt.grad, opt.weight_bf16, hp, t,
                       opt.norm_out)
        outs.append([opt.master.clone(), opt.exp_avg.clone(), opt.exp_avg_sq.clone(), opt.weight_bf16.clone()])
    for a, b in zip(*outs):
        assert torch.equal(_bits(a), _bits(b))


@pytest.mark.parametrize("K", [1, 3])
def test_step_graph_replays_equal_eager_steps(K):
    w = get_workload("toy")
    eager, graphed = _opt(w, 5), _opt(w, 5)
    n = eager.plan.arena_numel
    L = eager.plan.layout()
    pad = torch.ones(n, dtype=torch.bool, device="cuda")
    for o, c in zip(L.offsets, L.counts):
        pad[int(o):int(o) + int(c)] = False
    buffers = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(K)]
    sg = z.StepGraph(graphed, buffers)
    gen = torch.Generator(device="cuda").manual_seed(6)
    for t in range(1, 7):
        lr = z.lr_at(t, 3e-3, 3, 10, 3e-4)
        micros = []
        for _ in range(K):
            mb = (torch.randn(n, device="cuda", generator=gen) * 0.05).to(torch.bfloat16)
            mb[pad] = 0
            micros.append(mb)
        for k, mb in enumerate(micros):
            eager.accumulate(mb, last=(k == K - 1))
        eager.step(lr=lr)
        for buf, mb in zip(buffers, micros):
            buf.copy_(mb)
        sg.replay(lr=lr)
        assert graphed.t == eager.t == t
    torch.cuda.synchronize()
    for a, b in ((graphed.master, eager.master), (graphed.exp_avg, eager.exp_avg),
                 (graphed.exp_avg_sq, eager.exp_avg_sq), (graphed.weight_bf16, eager.weight_bf16),
                 (graphed.grad, eager.grad)):
        assert torch.equal(_bits(a), _bits(b))
    assert graphed.read_norm() == eager.read_norm()


@pytest.mark.parametrize("K", [1, 3])
def test_step_graph_replays_the_tensor_list_path(K):
    """StepGraph over a ShardListAdamW (zero1_list_step_dev): replays equal the eager list
    calls bit for bit, with the learning rate changing every step."""
    numels = [1000, 7, 4096, 33, 16385, 40000]
    nd = [0, 1, 0, 1, 0, 0]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)

    def make():
        opt = z.ShardListAdamW(numels, nd, dp_size=3, dp_rank=1, hparams=hp)
        g = torch.Generator(device="cuda").manual_seed(11)
        for t in opt.master:
            t.normal_(0.0, 0.02, generator=g)
        return opt

    eager, graphed = make(), make()
    counts = eager.plan.layout().counts
    micro = [[torch.zeros(int(c), dtype=torch.bfloat16, device="cuda") for c in counts] for _ in range(K)]
    sg = z.StepGraph(graphed, micro)
    g = torch.Generator(device="cuda").manual_seed(12)
    for step in range(4):
        for mb in micro:
            for t in mb:
                t.copy_(torch.randn(t.numel(), device="cuda", generator=g) * 0.05)
        lr = 1e-3 * (step + 1)
        for k, mb in enumerate(micro):
            eager.accumulate(mb, last=(k == K - 1))
        eager.step(lr=lr)
        sg.replay(lr=lr)
    torch.cuda.synchronize()
    assert graphed.t == eager.t == 4
    for name in ("master", "exp_avg", "exp_avg_sq", "weight_bf16", "grad"):
        for a, b in zip(getattr(eager, name), getattr(graphed, name)):
            assert torch.equal(_bits(a), _bits(b)), name
