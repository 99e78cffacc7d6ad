"""zero1_grad_norm_static, the norm call that allocates nothing.

It serves callers that cannot provide device scratch (a plain C program with
no device allocator, a process whose framework allocator holds nearly all of
the GPU's memory, a step that must not call cudaMalloc).  Through the C ABI it
must give the same norm record as zero1_grad_norm with a caller workspace,
field for field and bit for bit (the same kernels over the same tiles), call
after call: consecutive calls change the plan, the gradient and the number of
tiles, up and down, with the earlier calls' partial sums still in the shared
array.  A plan of exactly the largest size it serves is accepted; one
8-element vector more is refused before anything is launched.

This file is named to be collected last; it passes alone in a fresh process
and after the other tests.
"""
import ctypes

import pytest
import torch

import zero_sharded_mixed_local_gb300 as z
from zero_sharded_mixed_local_gb300.binding import _NormOut

pytestmark = pytest.mark.gpu


def _c_norm(lib, nout, stream):
    out = _NormOut()
    assert lib.zero1_read_norm(ctypes.c_void_p(nout.data_ptr()), stream, ctypes.byref(out)) == z.ZERO1_OK
    return out


def _fields(rec):
    return (rec.sumsq, rec.norm, rec.status, rec.n_partials)


def _case(numels, no_decay, sigma, seed):
    plan = z.Plan(numels, no_decay, 1, 0)
    g = torch.Generator(device="cuda").manual_seed(seed)
    grad = plan.new_arena()
    L = plan.layout()
    for o, c in zip(L.offsets, L.counts):
        grad[int(o):int(o) + int(c)] = torch.randn(int(c), device="cuda", generator=g) * sigma
    return plan, grad


def _both(lib, plan, grad, extra, stream):
    """(workspace record, static record) of one gradient, each through the C ABI."""
    ws = plan.new_workspace()
    ref_out, got_out = z.new_norm_out(), z.new_norm_out()
    gp = ctypes.c_void_p(grad.data_ptr())
    rc = lib.zero1_grad_norm(plan.handle, gp, ctypes.c_double(extra), ctypes.c_void_p(ws.data_ptr()),
                             ctypes.c_size_t(ws.numel()), ctypes.c_void_p(ref_out.data_ptr()), stream)
    assert rc == z.ZERO1_OK
    rc = lib.zero1_grad_norm_static(plan.handle, gp, ctypes.c_double(extra), ctypes.c_void_p(got_out.data_ptr()),
                                    stream)
    assert rc == z.ZERO1_OK, lib.zero1_strerror(rc)
    return _c_norm(lib, ref_out, stream), _c_norm(lib, got_out, stream)


def test_static_norm_matches_workspace_norm_on_calls_in_a_row():
    assert torch.cuda.is_available()
    lib = z.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    small = _case([5000, 12, 1], [0, 0, 1], 3.0, 2)                          # 1 tile
    large = _case([16384 * 40 + 8 * 5 + 3, 1000, 77], [0, 1, 0], 0.01, 1)   # 42 tiles, ragged tail
    # one tile, then 42 (the second call reads 41 partials the first never wrote), then one again
    for extra in (0.0, 1.25):
        for plan, grad in (small, large, small):
            ref, got = _both(lib, plan, grad, extra, stream)
            assert got.status == z.ZERO1_OK
            assert _fields(got) == _fields(ref)


def test_static_norm_at_its_size_limit_and_one_vector_beyond():
    """A 2^32-element arena (the whole 2 MiB array, 262,144 tiles) after a one-tile call:
    every element 2^-8, so the sum of squares is 2^32 * 2^-16 = 65536 exactly and both
    calls must say so.  One more 8-element vector is refused before any launch."""
    lib = z.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    plan, grad = _case([100], [0], 1.0, 5)
    ref, got = _both(lib, plan, grad, 0.0, stream)
    assert _fields(got) == _fields(ref) and ref.n_partials == 1
    del grad

    limit = z.binding.STATIC_NORM_MAX_NUMEL
    big = z.Plan([limit], [0], 1, 0)
    assert big.arena_numel == limit
    grad = torch.full((limit,), 2.0 ** -8, dtype=torch.float32, device="cuda")  # 16 GiB
    ref, got = _both(lib, big, grad, 0.0, stream)
    assert _fields(got) == _fields(ref)
    assert got.sumsq == 65536.0 and got.norm == 256.0
    assert got.n_partials == z.binding.STATIC_NORM_MAX_NUMEL // 16384
    del grad
    torch.cuda.empty_cache()

    over = z.Plan([limit + 8], [0], 1, 0)  # host-only plan, nothing allocated
    fake = ctypes.c_void_p(1 << 20)  # never used: the size check comes before anything else
    rc = lib.zero1_grad_norm_static(over.handle, fake, ctypes.c_double(0.0), fake, None)
    assert rc == z.ZERO1_ETOOBIG
    assert "static" in lib.zero1_strerror(rc).decode()


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


def test_static_norm_binding_refuses_plans_beyond_its_limit():
    big = z.Plan([z.binding.STATIC_NORM_MAX_NUMEL + 8], [0], 1, 0)
    with pytest.raises(ValueError, match="static norm scratch limit"):
        z.grad_norm_static(big, torch.zeros(16, device="cuda"), z.new_norm_out())
