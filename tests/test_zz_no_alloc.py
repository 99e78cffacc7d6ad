"""zero1_grad_norm_static, the norm call that allocates nothing.

It serves callers that cannot provide device scratch (a plain C program with
no device allocator, a process whose framework allocator holds nearly all of
the GPU's memory, a step that must not call cudaMalloc).  Through the C ABI it
must give the same norm record as zero1_grad_norm with a caller workspace,
call after call: the second of two calls in a row runs on a different
gradient (and a smaller plan), with the first call's partial sums still in
the shared array.

This file is named to be collected last; it passes alone in a fresh process
and after the other tests.
"""
import ctypes

import pytest
import torch

import zero_sharded_mixed_local_gb300 as z
from zero_sharded_mixed_local_gb300.binding import _NormOut

pytestmark = pytest.mark.gpu

TIGHT = 1e-12  # the relative agreement the parity tests require of two sums of squares


def _c_norm(lib, nout, stream):
    out = _NormOut()
    assert lib.zero1_read_norm(ctypes.c_void_p(nout.data_ptr()), stream, ctypes.byref(out)) == z.ZERO1_OK
    return out


def _case(numels, no_decay, sigma, seed):
    plan = z.Plan(numels, no_decay, 1, 0)
    g = torch.Generator(device="cuda").manual_seed(seed)
    grad = plan.new_arena()
    L = plan.layout()
    for o, c in zip(L.offsets, L.counts):
        grad[int(o):int(o) + int(c)] = torch.randn(int(c), device="cuda", generator=g) * sigma
    return plan, grad


def test_static_norm_matches_workspace_norm_on_two_calls_in_a_row():
    assert torch.cuda.is_available()
    lib = z.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [
        _case([16384 * 40 + 8 * 5 + 3, 1000, 77], [0, 1, 0], 0.01, 1),  # 42 tiles, ragged tail
        _case([5000, 12, 1], [0, 0, 1], 3.0, 2),                         # 1 tile, smaller than before
    ]
    for extra in (0.0, 1.25):
        for plan, grad in cases:
            ws = plan.new_workspace()
            ref_out, got_out = z.new_norm_out(), z.new_norm_out()
            gp = ctypes.c_void_p(grad.data_ptr())
            rc = lib.zero1_grad_norm(plan.handle, gp, ctypes.c_double(extra), ctypes.c_void_p(ws.data_ptr()),
                                     ctypes.c_size_t(ws.numel()), ctypes.c_void_p(ref_out.data_ptr()), stream)
            assert rc == z.ZERO1_OK
            rc = lib.zero1_grad_norm_static(plan.handle, gp, ctypes.c_double(extra),
                                            ctypes.c_void_p(got_out.data_ptr()), stream)
            assert rc == z.ZERO1_OK, lib.zero1_strerror(rc)
            ref, got = _c_norm(lib, ref_out, stream), _c_norm(lib, got_out, stream)
            assert got.status == ref.status == z.ZERO1_OK
            assert got.n_partials == ref.n_partials
            assert abs(got.sumsq - ref.sumsq) <= TIGHT * ref.sumsq
            assert abs(got.norm - ref.norm) <= TIGHT * ref.norm


def test_static_norm_feeds_the_step_like_the_workspace_norm():
    plan, grad = _case([20000, 64], [0, 1], 0.05, 3)
    outs = []
    for use_static in (False, True):
        nout = z.new_norm_out()
        if use_static:
            z.grad_norm_static(plan, grad, nout)
        else:
            z.grad_norm(plan, grad, plan.new_workspace(), nout)
        master = torch.linspace(-0.1, 0.1, plan.arena_numel, device="cuda")
        m, v, w = plan.new_arena(), plan.new_arena(), plan.new_arena(torch.bfloat16)
        z.step(plan, master, m, v, grad, w, z.Hparams(), 1, nout)
        outs.append((master, m, v, w))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_static_norm_rejects_plans_beyond_its_limit():
    lib = z.load_library()
    big = z.Plan([z.binding.STATIC_NORM_MAX_NUMEL + 8], [0], 1, 0)  # host-only plan, nothing allocated
    fake = ctypes.c_void_p(1 << 20)  # never used: the size check comes first
    rc = lib.zero1_grad_norm_static(big.handle, fake, ctypes.c_double(0.0), fake, None)
    assert rc == z.ZERO1_ETOOBIG
    assert "static" in lib.zero1_strerror(rc).decode()
    with pytest.raises(ValueError, match="static norm scratch limit"):
        z.grad_norm_static(big, torch.zeros(16, device="cuda"), z.new_norm_out())
