"""The host-fed loop the bench's end-to-end figure runs (``HostFedSteps``), checked.

Every step's micro-batch gradients start in pinned host memory and are copied
on a side stream into one of two staging sets; the step stream waits for its
copy (an event), runs accumulate / accumulate_norm / step as programmatic
dependent launches, and copies the norm record back, read one step behind.
This is the only place on the path where cross-stream event waits meet
programmatic stream serialisation, so the test runs exactly that loop, with
fresh gradients every step, and requires:
  - master, m, v and the bf16 copy equal, bit for bit, to the same steps run
    synchronously from device-resident gradients;
  - every step's norm record equal to the synchronous step's;
  - master, m and v within 4 fp32 ulp of the oracle (every element of the toy
    shard; the usual sample of the full-size SmolLM-135M list and of the
    1.0B-element Llama-3.1-8B shard the bench's e2e figure runs), the gradient
    of every synchronous step bit-exact against the oracle in full, and the
    bf16 copy the RNE of the master, in full.
The loop runs in two calls (the bench's warm-up and timed calls, the second
gated on an event), so the alternating slots carry over between calls.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_local_gb300 as z

from parity import MAX_ULP, Problem, group_counts, oracle_pass, sample_indices, ulp_diff

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _sync_step(pb, micros, t, k_way):
    """The synchronous step from device-resident gradients, as the bench's timed step runs it."""
    if not k_way:
        return pb.gpu_step(micros, t)
    z.accumulate_norm(pb.plan, pb.grad, micros, pb.ws, pb.nout, overwrite_first=True)
    z.step(pb.plan, pb.master, pb.m, pb.v, pb.grad, pb.wbf, pb.hp, t, pb.nout)
    return z.read_norm(pb.nout)


def _host_fed_vs_sync_and_oracle(workload, steps, sampled, k_way=False, first_call=2):
    sync, pipe = Problem(workload), Problem(workload)
    assert torch.equal(_bits(sync.master), _bits(pipe.master))  # same seed, same draw
    w, n = sync.w, sync.n
    idx = sample_indices(sync.layout) if sampled else np.arange(n, dtype=np.int64)
    idx_t = torch.from_numpy(idx).to(sync.dev)
    counts = group_counts(idx, sync.plan)
    lr_scale, wd_scale = w.group_scales()
    P = sync.master[idx_t].cpu().numpy().copy()
    M, V = np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32)

    host, sync_records = [], []
    for t in range(1, steps + 1):
        micros = sync.gen.micro_grads()  # fresh gradients every step
        host.append([mb.cpu().pin_memory() for mb in micros])
        sync_records.append(_sync_step(sync, micros, t, k_way))
        g_idx, ref_sumsq = oracle_pass(micros, sync.grad, idx)  # the gradient, bit for bit, in full
        ok, norm, coef = oracle.clip_coef(ref_sumsq, w.hp["clip_grad"])
        assert ok and sync_records[-1]["status"] == 0
        oracle.adamw_scaled(P, M, V, g_idx, counts, lr_scale, wd_scale, w.hp, t, coef)
        del micros

    loop = z.HostFedSteps(pipe.plan, pipe.master, pipe.m, pipe.v, pipe.wbf, pipe.hp, w.micro_batches, k_way=k_way)
    records = loop.run(lambda i: host[i], first_call)
    gate = torch.cuda.Event()
    gate.record(loop.stream)
    records += loop.run(lambda i: host[first_call + i], steps - first_call, first_event=gate, time_copies=True)
    torch.cuda.synchronize()
    assert loop.t == steps and len(records) == steps
    assert records == sync_records

    for name, a, b in (("master", pipe.master, sync.master), ("m", pipe.m, sync.m), ("v", pipe.v, sync.v),
                       ("bf16", pipe.wbf, sync.wbf)):
        assert torch.equal(_bits(a), _bits(b)), name
    for name, dev_t, ref in (("master", pipe.master, P), ("m", pipe.m, M), ("v", pipe.v, V)):
        d = ulp_diff(dev_t[idx_t].cpu().numpy(), ref)
        assert int(d.max()) <= MAX_ULP, (name, int(d.max()), int(idx[int(np.argmax(d))]))
    assert torch.equal(_bits(pipe.wbf), _bits(pipe.master.to(torch.bfloat16)))
    return records


def test_host_fed_toy_every_element():
    recs = _host_fed_vs_sync_and_oracle("toy", steps=8, sampled=False)
    assert len({r["sumsq"] for r in recs}) == 8  # a new gradient every step


def test_host_fed_toy_k_way():
    _host_fed_vs_sync_and_oracle("toy", steps=5, sampled=False, k_way=True, first_call=1)


def test_host_fed_smollm135m_sampled():
    recs = _host_fed_vs_sync_and_oracle("smollm135m", steps=4, sampled=True)
    assert len({r["sumsq"] for r in recs}) == 4


def test_host_fed_llama8b_sampled():
    """The bench's own workload for its e2e figure: the 1.0B-element Llama-3.1-8B shard, K = 1."""
    recs = _host_fed_vs_sync_and_oracle("llama8b", steps=3, sampled=True)
    assert len({r["sumsq"] for r in recs}) == 3


def test_host_fed_on_a_stream_that_is_not_the_current_one():
    """Every copy and kernel of the loop runs on the stream it was given, not on torch's current
    stream: the same results as the synchronous steps while the current stream stays idle."""
    sync, pipe = Problem("toy"), Problem("toy")
    host = []
    for t in range(1, 5):
        micros = sync.gen.micro_grads()
        host.append([mb.cpu().pin_memory() for mb in micros])
        sync.gpu_step(micros, t)
    own = torch.cuda.Stream()
    loop = z.HostFedSteps(pipe.plan, pipe.master, pipe.m, pipe.v, pipe.wbf, pipe.hp, pipe.w.micro_batches,
                          stream=own)
    records = loop.run(lambda i: host[i], 4)
    own.synchronize()
    assert records[-1] == z.read_norm(sync.nout)
    for a, b in ((pipe.master, sync.master), (pipe.m, sync.m), (pipe.v, sync.v), (pipe.wbf, sync.wbf)):
        assert torch.equal(_bits(a), _bits(b))


def test_host_fed_rejects_pageable_host_gradients():
    pb = Problem("toy")
    loop = z.HostFedSteps(pb.plan, pb.master, pb.m, pb.v, pb.wbf, pb.hp, pb.w.micro_batches)
    pageable = [torch.zeros(pb.n, dtype=torch.bfloat16) for _ in range(pb.w.micro_batches)]
    with pytest.raises(ValueError, match="pinned"):
        loop.run(pageable, 1)
    assert loop.t == 0
