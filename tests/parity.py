"""GPU-vs-oracle parity harness (test infrastructure).

Runs the CUDA path through the C ABI and the CPU oracle on the same seeded
inputs and compares them element by element:
  - fp32 grad arena: bit-exact (same IEEE additions in the same order)
  - sum of squares / norm: within 1e-5 relative
  - master, m, v: within 4 fp32 ulp after all steps
  - bf16 copy: bit-exact against round-to-nearest-even of the GPU master
The oracle accumulates over the whole arena in host chunks (padding is zero
and stays zero under every operation, which the comparison checks too) and
steps either every arena element or, for the full-size workloads, sampled
arena indices.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import zero_sharded_mixed_local_gb300 as z
from zero_sharded_mixed_local_gb300.workloads import InputGenerator, Layout, Workload, get_workload

SUMSQ_RTOL = 1e-5     # the stated bar for the gradient norm
SUMSQ_TIGHT = 1e-12   # both sides sum the exact squares with compensation; they agree far closer
MAX_ULP = 4


def ordered_int(x):
    i = np.asarray(x, np.float32).view(np.int32).astype(np.int64)
    return np.where(i < 0, -(i & 0x7FFFFFFF), i)


def ulp_diff(a, b):
    return np.abs(ordered_int(a) - ordered_int(b))


def u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def rne_of(master_cpu):
    return master_cpu.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


class Problem:
    """One workload on the GPU: plan, arenas, generator."""

    def __init__(self, workload, device="cuda", seed=None):
        self.w = workload if isinstance(workload, Workload) else get_workload(workload)
        self.dev = torch.device(device)
        p = self.w.params
        self.plan = z.Plan(p.numels, dp_size=self.w.dp_size, dp_rank=self.w.dp_rank, **self.w.plan_kwargs())
        L = self.plan.layout()
        self.layout = Layout(L.counts, L.offsets, L.no_decay, L.arena_numel)
        self.gen = InputGenerator(self.w, self.layout, self.dev, seed)
        self.n = self.plan.arena_numel
        self.group1 = self.plan.group_range(1)[0]
        self.hp = z.Hparams(**self.w.hp)
        self.master = self.gen.master()
        self.m = self.gen.zeros()
        self.v = self.gen.zeros()
        self.grad = self.gen.zeros()
        self.wbf = self.gen.zeros(torch.bfloat16)
        self.ws = self.plan.new_workspace(self.dev)
        self.nout = z.new_norm_out(self.dev)

    def gpu_step(self, micros, t, extra_sumsq=0.0, fused=True, micro_step=False):
        """One step as bench.py runs it: the last micro-batch's accumulation takes the norm
        (fused=True), or separate accumulate and grad_norm calls (fused=False); with one
        micro-batch and micro_step, its norm from the micro-batch and the step that writes the
        gradient (micro_norm + step_accumulate, the bench's path for K = 1)."""
        if micro_step:
            assert len(micros) == 1
            z.micro_norm(self.plan, micros[0], self.ws, self.nout, extra_sumsq=extra_sumsq)
            z.step_accumulate(self.plan, self.master, self.m, self.v, self.grad, micros[0], self.wbf, self.hp, t,
                              self.nout)
            return z.read_norm(self.nout)
        last = len(micros) - 1
        for k, mb in enumerate(micros[:last] if fused else micros):
            z.accumulate(self.plan, self.grad, mb, overwrite_first=(k == 0))
        if fused:
            z.accumulate_norm(self.plan, self.grad, micros[last], self.ws, self.nout, overwrite_first=(last == 0),
                              extra_sumsq=extra_sumsq)
        else:
            z.grad_norm(self.plan, self.grad, self.ws, self.nout, extra_sumsq)
        z.step(self.plan, self.master, self.m, self.v, self.grad, self.wbf, self.hp, t, self.nout)
        return z.read_norm(self.nout)


def oracle_grad(n, micros_u16):
    g = np.zeros(n, np.float32)
    oracle.accumulate_all(g, micros_u16)
    return g


def group_counts(idx, plan):
    """Number of the sorted arena indices idx in each parameter group's arena range."""
    bounds = [plan.group_range(g)[0] for g in range(1, z.MAX_GROUPS)]
    cuts = np.searchsorted(idx, bounds)
    return np.diff(np.concatenate([[0], cuts, [len(idx)]])).astype(np.int64)


CHUNK = 1 << 26  # elements per host pass: bounds host memory on the full-size workloads
ORACLE_THREADS = max(1, min(8, os.cpu_count() or 1))  # chunks in flight (ctypes releases the GIL)


def _oracle_chunk(micros, gpu_grad, c0, c1):
    g = np.zeros(c1 - c0, np.float32)
    for k, mb in enumerate(micros):
        oracle.accumulate(g, u16(mb[c0:c1]), overwrite=(k == 0))
    gg = gpu_grad[c0:c1].cpu().numpy()
    bad = None
    if not np.array_equal(gg.view(np.uint32), g.view(np.uint32)):
        bad = int(np.nonzero(gg.view(np.uint32) != g.view(np.uint32))[0][0]) + c0
    return g, bad, oracle.sumsq(g)


def oracle_pass(micros, gpu_grad, idx):
    """Oracle accumulation over the whole arena, chunk by chunk: checks the GPU grad
    arena bit for bit, returns (oracle grad at idx, oracle sum of squares).  Chunks run
    on a few host threads; their sums of squares are added in chunk order."""
    n = gpu_grad.numel()
    s = 0.0
    g_idx = np.empty(idx.size, np.float32)
    bounds = [(c0, min(n, c0 + CHUNK)) for c0 in range(0, n, CHUNK)]
    with ThreadPoolExecutor(max_workers=ORACLE_THREADS) as ex:
        futures = [ex.submit(_oracle_chunk, micros, gpu_grad, c0, c1) for c0, c1 in bounds]
        for j, (c0, c1) in enumerate(bounds):
            g, bad, part = futures[j].result()
            futures[j] = None  # the chunk's host arrays go as soon as they are read
            if bad is not None:
                raise AssertionError("grad arena differs from the oracle at element %d" % bad)
            s += part
            lo, hi = np.searchsorted(idx, [c0, c1])
            g_idx[lo:hi] = g[idx[lo:hi] - c0]
    return g_idx, s


def run_parity(workload, steps=None, fresh_grads=True, sample=None, device="cuda", seed=None, fused=True,
               micro_step=False):
    """Run `steps` steps on GPU and oracle; assert parity.  `sample`: None compares every
    arena element (padding included), "sampled" the tensor edges, the padding and a
    million random elements; the grad arena and the bf16 copy are checked in full."""
    pb = Problem(workload, device, seed)
    w = pb.w
    steps = w.steps if steps is None else steps
    n = pb.n
    idx = np.arange(n, dtype=np.int64) if sample is None else sample_indices(pb.layout)
    idx_t = torch.from_numpy(idx).to(pb.dev)
    counts = group_counts(idx, pb.plan)
    lr_scale, wd_scale = w.group_scales()  # from the workload's own definition
    P = pb.master[idx_t].cpu().numpy().copy()
    M = np.zeros(idx.size, np.float32)
    V = np.zeros(idx.size, np.float32)

    micros = None
    report = []
    for t in range(1, steps + 1):
        new_grads = micros is None or fresh_grads
        if new_grads:  # refill the same buffers: one set of micro-batch arenas at a time
            micros = pb.gen.micro_grads(out=micros)
        got = pb.gpu_step(micros, t, fused=fused, micro_step=micro_step)
        if new_grads:
            g_idx, ref_sumsq = oracle_pass(micros, pb.grad, idx)
        assert got["status"] == 0
        assert abs(got["sumsq"] - ref_sumsq) <= SUMSQ_RTOL * ref_sumsq, (t, got["sumsq"], ref_sumsq)
        assert abs(got["sumsq"] - ref_sumsq) <= SUMSQ_TIGHT * ref_sumsq, (t, got["sumsq"], ref_sumsq)
        ok, norm, coef = oracle.clip_coef(ref_sumsq, w.hp["clip_grad"])
        assert ok
        oracle.adamw_scaled(P, M, V, g_idx, counts, lr_scale, wd_scale, w.hp, t, coef)
        report.append((t, got["norm"], norm, float(coef)))

    res = {}
    for name, dev_t, ref in (("master", pb.master, P), ("m", pb.m, M), ("v", pb.v, V)):
        a = dev_t[idx_t].cpu().numpy()
        d = ulp_diff(a, ref)
        res[name] = int(d.max()) if d.size else 0
        assert res[name] <= MAX_ULP, (name, res[name], int(idx[int(np.argmax(d))]))
    # bf16 copy: bit-exact round-to-nearest-even of the GPU master (torch's cast), in full
    for c0 in range(0, n, CHUNK):
        c1 = min(n, c0 + CHUNK)
        assert torch.equal(pb.wbf[c0:c1].view(torch.int16), pb.master[c0:c1].to(torch.bfloat16).view(torch.int16)), \
            "bf16 copy is not the RNE of the GPU master in [%d, %d)" % (c0, c1)
    res["norms"] = report
    res["local_numel"] = pb.plan.local_numel
    res["compared"] = int(idx.size)
    return res


def sample_indices(layout, per_tensor_edge=2048, n_random=1_000_000, seed=0):
    """First and last `per_tensor_edge` local elements of every tensor, plus random ones."""
    parts = []
    for o, c in zip(layout.offsets, layout.counts):
        o, c = int(o), int(c)
        if c == 0:
            continue
        e = min(c, per_tensor_edge)
        parts.append(np.arange(o, o + e, dtype=np.int64))
        parts.append(np.arange(o + c - e, o + c, dtype=np.int64))
        # the padding after the shard (zero, and it must stay zero)
        parts.append(np.arange(o + c, (o + c + 7) // 8 * 8, dtype=np.int64))
    rng = np.random.default_rng(seed)
    parts.append(rng.integers(0, layout.arena_numel, size=min(n_random, layout.arena_numel), dtype=np.int64))
    return np.unique(np.concatenate(parts))


def bf16_norm_pattern(x, kind, gen):
    """Overwrite some of a flat bf16 CUDA tensor's elements, in place, with values that steer the
    norm kernels between their exact-square form and the general one:
    "exact" leaves gradient-sized values (every square exact); "outside" scatters bf16 subnormals and
    values just below the exact range (and its lower end) among them; "zeros" makes 30% of the values
    and every 37th whole vector zero, with some -0; "large" scatters values near 2^63 and 2^64, whose
    squares overflow the sums; "inf" places one infinity."""
    n = x.numel()
    if n == 0 or kind == "exact":
        return x
    b = x.view(torch.int16)

    def put(every, values):
        k = max(1, n // every)
        idx = torch.randint(0, n, (k,), generator=gen, device=x.device)
        vals = torch.tensor(np.array(values, np.uint16).view(np.int16), device=x.device)
        b[idx] = vals[torch.randint(0, len(values), (k,), generator=gen, device=x.device)]

    if kind == "outside":
        put(500, [0x0001, 0x0040, 0x807F, 0x1D80, 0x9DFF, 0x1D82, 0x1E00, 0x9E01])
    elif kind == "zeros":
        b[torch.rand(n, generator=gen, device=x.device) < 0.3] = 0
        b[:n - n % 8].view(-1, 8)[::37] = 0
        put(1000, [0x8000])
    elif kind == "large":
        put(5000, [0x5F00, 0xDF7F, 0x5F80])
    elif kind == "inf":
        b[n // 2] = 0x7F80
    else:
        raise ValueError(kind)
    return x
