"""The library in a training loop: a small bf16 MLP trained on synthetic data.

Each step's bf16 parameter gradients are laid out in model layout, moved into
a LocalShardAdamW's arena with shard_gather, stepped (fused accumulate + norm,
clip, AdamW, bf16 copy), and the bf16 weights are scattered back into the
model.  A twin model trained by torch.optim.AdamW on fp32 master weights with
torch's clip_grad_norm_ must follow the same trajectory up to rounding-order
noise: losses within 2%, weights within 0.5% in L2 per tensor and 95% of them
within two bf16 ulps (the two AdamW implementations differ only in rounding
order, which the bf16 forward passes then amplify).
"""
import pytest
import torch

import zero_sharded_mixed_local_gb300 as z

pytestmark = pytest.mark.gpu


def _model(seed):
    torch.manual_seed(seed)
    return torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(), torch.nn.LayerNorm(256),
                               torch.nn.Linear(256, 16)).cuda()


def test_training_loop_tracks_torch_adamw():
    hp = dict(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)
    base = _model(0)
    ours, ref = _model(0), _model(0)
    for m in (ours, ref):
        m.load_state_dict(base.state_dict())
    params_o = list(ours.parameters())
    params_r = list(ref.parameters())
    # fp32 masters: ours in the optimizer's arena, the reference's in torch parameters
    master_r = [p.detach().clone().float().requires_grad_(True) for p in params_r]
    for m in (ours, ref):
        m.to(torch.bfloat16)
    names = [n for n, _ in ours.named_parameters()]
    no_decay = [1 if (n.endswith("bias") or n.startswith("2.")) else 0 for n in names]  # biases, LayerNorm
    numels = [p.numel() for p in params_o]
    opt = z.LocalShardAdamW(numels, no_decay, hparams=hp)
    z.shard_gather(opt.plan, torch.cat([p.detach().float().reshape(-1) for p in base.parameters()]), opt.master)
    decay = [p for p, nd in zip(master_r, no_decay) if not nd]
    nodecay = [p for p, nd in zip(master_r, no_decay) if nd]
    topt = torch.optim.AdamW([{"params": decay, "weight_decay": hp["weight_decay"]},
                              {"params": nodecay, "weight_decay": 0.0}], lr=hp["lr"],
                             betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"], foreach=False, fused=False)

    g = torch.Generator(device="cuda").manual_seed(1)
    w_true = torch.randn(64, 16, device="cuda", generator=g)
    mb_arena = opt.plan.new_arena(torch.bfloat16)
    full_w = torch.zeros(opt.plan.total_numel, dtype=torch.bfloat16, device="cuda")
    losses = []
    for step in range(25):
        x = torch.randn(128, 64, device="cuda", generator=g)
        y = x @ w_true
        lo = torch.nn.functional.mse_loss(ours(x.bfloat16()).float(), y)
        lr_ = torch.nn.functional.mse_loss(ref(x.bfloat16()).float(), y)
        for m in (ours, ref):
            m.zero_grad(set_to_none=True)
        lo.backward()
        lr_.backward()
        losses.append((lo.item(), lr_.item()))
        # ours: model-layout bf16 gradient -> arena -> step -> bf16 weights -> model
        full_g = torch.cat([p.grad.reshape(-1) for p in params_o])
        z.shard_gather(opt.plan, full_g, mb_arena)
        opt.accumulate(mb_arena, last=True)
        opt.step()
        z.shard_scatter(opt.plan, opt.weight_bf16, full_w)
        with torch.no_grad():
            off = 0
            for p in params_o:
                p.copy_(full_w[off:off + p.numel()].view_as(p))
                off += p.numel()
        # reference: fp32 masters, torch's clipping, AdamW, then the bf16 copy
        for mp, p in zip(master_r, params_r):
            mp.grad = p.grad.float()
        torch.nn.utils.clip_grad_norm_(master_r, hp["clip_grad"])
        topt.step()
        with torch.no_grad():
            for mp, p in zip(master_r, params_r):
                p.copy_(mp.to(torch.bfloat16))
    assert losses[-1][0] < 0.5 * losses[0][0]  # it trains
    for (a, b) in losses:
        assert abs(a - b) <= 2e-2 * max(abs(b), 1e-6), (a, b)
    for po, pr in zip(params_o, params_r):
        po, pr = po.detach(), pr.detach()
        diff = (po.float() - pr.float()).abs()
        # rounding-order noise between the two AdamW implementations compounds through the bf16 forward
        # passes, most where weights pass near zero; the trajectories must still agree closely
        assert float(diff.norm() / pr.float().norm()) < 5e-3
        ulp = torch.finfo(torch.bfloat16).eps * pr.float().abs().clamp_min(1e-3)
        assert float((diff <= 2 * ulp).float().mean()) > 0.95


def test_module_optimizer_tracks_torch_adamw():
    """Zero1AdamW over model.named_parameters(): gradients read from p.grad and bf16
    weights written into the parameters in place, no copies in between; the same
    trajectory as torch's AdamW on fp32 masters."""
    hp = dict(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)
    base = _model(0)
    ours, ref = _model(0), _model(0)
    for m in (ours, ref):
        m.load_state_dict(base.state_dict())
    params_r = list(ref.parameters())
    master_r = [p.detach().clone().float().requires_grad_(True) for p in params_r]
    for m in (ours, ref):
        m.to(torch.bfloat16)
    nd = lambda n, p: n.endswith("bias") or n.startswith("2.")  # noqa: E731  biases, LayerNorm
    opt = z.Zero1AdamW(ours.named_parameters(), hparams=hp, no_decay=nd)
    storage = [p.data_ptr() for p in ours.parameters()]
    decay = [p for (n, _), p in zip(ref.named_parameters(), master_r) if not nd(n, p)]
    nodecay = [p for (n, _), p in zip(ref.named_parameters(), master_r) if nd(n, p)]
    topt = torch.optim.AdamW([{"params": decay, "weight_decay": hp["weight_decay"]},
                              {"params": nodecay, "weight_decay": 0.0}], lr=hp["lr"],
                             betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"], foreach=False, fused=False)
    g = torch.Generator(device="cuda").manual_seed(1)
    w_true = torch.randn(64, 16, device="cuda", generator=g)
    losses = []
    for step in range(25):
        acc_r = [torch.zeros_like(mp) for mp in master_r]
        lo = lr_ = 0.0
        for micro in range(2):  # two micro-batches, each gradient added in fp32 on both sides
            for m in (ours, ref):
                m.zero_grad(set_to_none=False)
            x = torch.randn(64, 64, device="cuda", generator=g)
            y = x @ w_true
            l1 = torch.nn.functional.mse_loss(ours(x.bfloat16()).float(), y)
            l2 = torch.nn.functional.mse_loss(ref(x.bfloat16()).float(), y)
            l1.backward()
            l2.backward()
            opt.accumulate(last=(micro == 1))  # reads p.grad; the last call also takes the norm
            for a, p in zip(acc_r, params_r):
                a += p.grad.float()
            lo, lr_ = lo + l1.item(), lr_ + l2.item()
        losses.append((lo, lr_))
        opt.step()
        for mp, a in zip(master_r, acc_r):
            mp.grad = a
        torch.nn.utils.clip_grad_norm_(master_r, hp["clip_grad"])
        topt.step()
        with torch.no_grad():
            for mp, p in zip(master_r, params_r):
                p.copy_(mp.to(torch.bfloat16))
    assert [p.data_ptr() for p in ours.parameters()] == storage  # updated in place
    assert opt.t == 25
    assert losses[-1][0] < 0.7 * losses[0][0]  # it trains
    for (a, b) in losses:
        assert abs(a - b) <= 2e-2 * max(abs(b), 1e-6), (a, b)
    for po, pr in zip(ours.parameters(), ref.parameters()):
        po, pr = po.detach().float(), pr.detach().float()
        assert float((po - pr).norm() / pr.norm()) < 1e-2


def test_module_optimizer_steps_only_its_slice():
    """dp 2, rank 1: only rank 1's slice of every parameter changes, by the oracle's step on
    that slice (its own sum of squares: no group given)."""
    import numpy as np

    import oracle
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)
    model = _model(3).to(torch.bfloat16)
    before = [p.detach().clone() for p in model.parameters()]
    opt = z.Zero1AdamW(model.named_parameters(), hparams=hp, dp_size=2, dp_rank=1)
    x = torch.randn(32, 64, device="cuda", generator=torch.Generator(device="cuda").manual_seed(5))
    model(x.bfloat16()).float().pow(2).mean().backward()
    grads = [p.grad.detach().clone() for p in model.parameters()]
    opt.step()
    torch.cuda.synchronize()
    sl = opt._slices
    P = np.concatenate([b.view(-1)[s:s + c].float().cpu().numpy() for b, (s, c) in zip(before, sl)])
    G = np.concatenate([g.view(-1)[s:s + c].float().cpu().numpy() for g, (s, c) in zip(grads, sl)])
    M, V = np.zeros_like(P), np.zeros_like(P)
    _, _, coef = oracle.clip_coef(oracle.sumsq(G), hp["clip_grad"])
    oracle.adamw(P, M, V, G, [c for _, c in sl], opt.no_decay, hp, 1, coef)
    got = np.concatenate([p.detach().view(-1)[s:s + c].view(torch.int16).cpu().numpy().view(np.uint16)
                          for p, (s, c) in zip(model.parameters(), sl)])
    assert np.array_equal(got, oracle.bf16_rne(P))
    for p, b, (s, c) in zip(model.parameters(), before, sl):
        rest = torch.cat([p.detach().view(-1)[:s], p.detach().view(-1)[s + c:]])
        rest_b = torch.cat([b.view(-1)[:s], b.view(-1)[s + c:]])
        assert torch.equal(rest, rest_b)


def test_module_optimizer_follows_reallocated_gradients():
    """zero_grad(set_to_none=True) makes autograd allocate new gradient tensors every step;
    the optimizer must read the new ones (its cached pointer lists are keyed on them), and
    give the same parameters as a run that keeps the gradient buffers."""
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)
    runs = []
    for set_to_none in (False, True):
        model = _model(4).to(torch.bfloat16)
        opt = z.Zero1AdamW(model.named_parameters(), hparams=hp)
        g = torch.Generator(device="cuda").manual_seed(9)
        for step in range(4):
            model.zero_grad(set_to_none=set_to_none)
            x = torch.randn(32, 64, device="cuda", generator=g)
            model(x.bfloat16()).float().pow(2).mean().backward()
            opt.step()
        runs.append([p.detach().clone() for p in model.parameters()])
    for a, b in zip(*runs):
        assert torch.equal(a, b)


def test_module_optimizer_on_a_side_stream_equals_the_current_stream():
    """Zero1AdamW.accumulate / step given a stream that is not the current one: the gradient pointer
    lists are uploaded on that stream, and the parameters equal those of the same steps on the current
    stream, with one micro-batch (no accumulate call) and with two."""
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, clip_grad=1.0)
    for n_micro in (1, 2):
        runs = []
        for use_side in (False, True):
            side = torch.cuda.Stream() if use_side else None
            model = _model(6).to(torch.bfloat16)
            opt = z.Zero1AdamW(model.named_parameters(), hparams=hp)
            g = torch.Generator(device="cuda").manual_seed(11)
            for step in range(3):
                for micro in range(n_micro):
                    model.zero_grad(set_to_none=True)  # new gradient tensors: new pointer lists every call
                    x = torch.randn(32, 64, device="cuda", generator=g)
                    model(x.bfloat16()).float().pow(2).mean().backward()
                    if side is not None:
                        side.wait_stream(torch.cuda.current_stream())
                    if n_micro > 1:
                        opt.accumulate(last=(micro == n_micro - 1), stream=side)
                        if side is not None:  # the gradients it read are freed on the current stream next
                            torch.cuda.current_stream().wait_stream(side)
                if side is not None:
                    side.wait_stream(torch.cuda.current_stream())
                opt.step(stream=side)
                if side is not None:
                    torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            runs.append([p.detach().clone() for p in model.parameters()])
        for a, b in zip(*runs):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), n_micro
