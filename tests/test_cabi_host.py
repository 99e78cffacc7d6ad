"""Host-side checks of the C ABI (no GPU): the library loads, exports every
declared entry point, and its plan (shard split, arena layout, byte
accounting) agrees with the oracle.  Only calls that never touch CUDA are
made; argument errors return before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from zero_sharded_mixed_local_gb300 import build as zbuild
from zero_sharded_mixed_local_gb300.workloads import WORKLOADS, get_workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def z():
    zbuild.build_library()
    import zero_sharded_mixed_local_gb300 as z
    z.load_library()
    return z


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(zero1_\w+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_symbol(z):
    names = declared_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(zbuild.LIB)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_exported_symbols_are_all_declared(z):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", zbuild.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (zero1_\w+)", out))
    assert exported == set(declared_functions())


@pytest.mark.parametrize("name", WORKLOADS)
def test_plan_matches_oracle_for_every_workload(z, name):
    w = get_workload(name)
    plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank)
    start, count, local = oracle.plan(w.params.numels, w.dp_size, w.dp_rank)
    L = plan.layout()
    assert np.array_equal(L.shard_start, start) and np.array_equal(L.counts, count)
    assert plan.local_numel == local and plan.total_numel == w.params.total
    assert plan.num_tensors == len(w.params)
    _check_layout(plan, w.params.no_decay)
    for gb in (2, 4):
        assert plan.bytes(gb) == oracle.zero1_bytes(w.params.total, local, gb)


def _check_layout(plan, no_decay):
    L = plan.layout()
    assert plan.arena_numel % 8 == 0
    assert np.all(L.offsets % 8 == 0)
    b0, e0 = plan.group_range(0)
    b1, e1 = plan.group_range(1)
    assert b0 == 0 and e0 == b1 and e1 == plan.arena_numel
    nd = np.asarray(no_decay, bool)
    # each group holds exactly its tensors, in model order, without overlap
    for g, (b, e) in enumerate(((b0, e0), (b1, e1))):
        sel = np.nonzero(nd == bool(g))[0]
        offs, cnts = L.offsets[sel], L.counts[sel]
        assert np.all(offs >= b) and np.all(offs + cnts <= e)
        assert np.all(np.diff(offs) >= 0)
        ends = offs + cnts
        assert np.all(ends[:-1] <= offs[1:])
        assert (np.sum((cnts + 7) // 8 * 8) == e - b)


def test_plan_matches_oracle_on_random_shape_lists(z):
    """Two hundred seeded draws: 1-40 tensors of 0-70,000 elements (a fifth under the dp size),
    random no-decay flags, dp 1-16 and every rank of a few of them.  Shard split, counts, local size
    and byte accounting as the oracle gives them; arena layout as _check_layout requires; and the
    ranks' shards tile every tensor exactly."""
    rng = np.random.default_rng(2024)
    for draw in range(200):
        n = int(rng.integers(1, 41))
        dp = int(rng.integers(1, 17))
        small = rng.random(n) < 0.2
        numels = np.where(small, rng.integers(0, dp + 1, n), rng.integers(0, 70001, n)).astype(np.int64)
        nd = (rng.random(n) < 0.3).astype(np.uint8)
        ranks = range(dp) if draw % 20 == 0 else [int(rng.integers(0, dp))]
        covered = np.zeros(n, np.int64)
        for r in ranks:
            plan = z.Plan(numels.tolist(), nd.tolist(), dp, r)
            start, count, local = oracle.plan(numels.tolist(), dp, r)
            L = plan.layout()
            assert np.array_equal(L.shard_start, start) and np.array_equal(L.counts, count), (draw, r)
            assert plan.local_numel == local and plan.total_numel == int(numels.sum())
            _check_layout(plan, nd)
            assert plan.bytes(2) == oracle.zero1_bytes(int(numels.sum()), local, 2)
            covered += L.counts
        if draw % 20 == 0:
            assert np.array_equal(covered, numels), draw


def test_small_plan_worked_example(z):
    # numels 10, 3, 8 over dp=3; tensor 1 is a norm weight
    plans = [z.Plan([10, 3, 8], [0, 1, 0], 3, r) for r in range(3)]
    assert [p.layout().counts.tolist() for p in plans] == [[4, 1, 3], [3, 1, 3], [3, 1, 2]]
    assert [p.layout().shard_start.tolist() for p in plans] == [[0, 0, 0], [4, 1, 3], [7, 2, 6]]
    # arena of rank 0: tensor 0 at 0 (4 -> pad 8), tensor 2 at 8 (3 -> 8), norm group at 16
    assert plans[0].layout().offsets.tolist() == [0, 16, 8]
    assert plans[0].arena_numel == 24 and plans[0].group_range(1) == (16, 24)
    assert plans[0].workspace_bytes == 8


def test_plan_rejects_bad_arguments(z):
    lib = z.load_library()
    h = ctypes.c_void_p()
    n = np.array([4, 4], np.int64)
    nd = np.array([0, 1], np.uint8)
    bad_nd = np.array([0, 2], np.uint8)
    neg = np.array([4, -1], np.int64)
    huge = np.array([1 << 55, (1 << 55) + 1], np.int64)   # adds up to 2^56 + 1 elements
    cases = [                  # (numels, no_decay, n_tensors, dp_size, dp_rank)
        (n, nd, 2, 2, 2),      # rank == dp
        (n, nd, 2, 2, -1),     # negative rank
        (n, nd, -1, 1, 0),     # negative tensor count
        (n, nd, 2, -3, 0),     # dp < 1
        (n, nd, 2, 0, 0),      # dp == 0
        (n, bad_nd, 2, 1, 0),  # no_decay not 0/1
        (neg, nd, 2, 1, 0),    # negative numel
        (huge, nd, 2, 1, 0),   # more than ZERO1_MAX_TOTAL_NUMEL in all
    ]
    for numels, flags, count, dp, rank in cases:
        rc = lib.zero1_plan_create(numels.ctypes.data, flags.ctypes.data, count, dp, rank, ctypes.byref(h))
        assert rc == z.ZERO1_EINVAL, (count, dp, rank)
        assert not h.value
    assert lib.zero1_plan_create(n.ctypes.data, nd.ctypes.data, 2, 1, 0, None) == z.ZERO1_EINVAL
    assert lib.zero1_plan_create(None, None, 2, 1, 0, ctypes.byref(h)) == z.ZERO1_EINVAL
    assert lib.zero1_plan_create(None, None, 0, 1, 0, ctypes.byref(h)) == z.ZERO1_OK
    lib.zero1_plan_destroy(h)
    lib.zero1_plan_destroy(None)
    assert lib.zero1_plan_arena_numel(None) == -1
    assert lib.zero1_plan_tensor(None, 0, None, None, None) == z.ZERO1_EINVAL


def test_compute_calls_reject_bad_arguments_before_any_launch(z):
    lib = z.load_library()
    plan = z.Plan([100, 8], [0, 1], 1, 0)
    h = plan.handle
    fake = ctypes.c_void_p(0x10000)      # never dereferenced: every case fails its checks first
    odd = ctypes.c_void_p(0x10008)
    arr = (ctypes.c_void_p * 1)(0x20000)
    arr_odd = (ctypes.c_void_p * 1)(0x20002)
    assert lib.zero1_accumulate(h, fake, arr, 0, 1, None) == z.ZERO1_EINVAL
    assert lib.zero1_accumulate(h, fake, arr, 17, 1, None) == z.ZERO1_EINVAL
    assert lib.zero1_accumulate(h, None, arr, 1, 1, None) == z.ZERO1_EINVAL
    assert lib.zero1_accumulate(h, fake, arr_odd, 1, 1, None) == z.ZERO1_EALIGN
    assert lib.zero1_accumulate(h, odd, arr, 1, 1, None) == z.ZERO1_EALIGN
    assert plan.workspace_bytes == 8
    assert lib.zero1_grad_norm(h, fake, 0.0, fake, 4, fake, None) == z.ZERO1_EINVAL  # workspace too small
    assert lib.zero1_grad_norm(h, fake, 0.0, odd, 64, fake, None) == z.ZERO1_EALIGN
    assert lib.zero1_grad_norm(h, fake, -1.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_grad_norm(None, fake, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    hp = z.binding._Hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 1.0)
    args = [h, fake, fake, fake, fake, fake]
    assert lib.zero1_step(*args, ctypes.byref(hp), 0, None, None) == z.ZERO1_EINVAL  # t < 1
    assert lib.zero1_step(h, fake, fake, fake, odd, fake, ctypes.byref(hp), 1, None, None) == z.ZERO1_EALIGN
    assert lib.zero1_step(h, fake, fake, fake, fake, odd, ctypes.byref(hp), 1, None, None) == z.ZERO1_EALIGN
    bad = z.binding._Hparams(3e-4, 1.0, 0.95, 1e-8, 0.1, 1.0)
    assert lib.zero1_step(*args, ctypes.byref(bad), 1, None, None) == z.ZERO1_EINVAL
    bad = z.binding._Hparams(float("nan"), 0.9, 0.95, 1e-8, 0.1, 1.0)
    assert lib.zero1_step(*args, ctypes.byref(bad), 1, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_read_norm(None, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_strerror(z.ZERO1_ENONFINITE).decode().startswith("gradient norm")
    assert lib.zero1_last_cuda_error().decode() == ""


def test_one_micro_batch_calls_reject_bad_arguments_before_any_launch(z):
    """zero1_micro_norm, zero1_step_accumulate and their tensor-list forms: every case below fails
    a check that comes before any CUDA call (the addresses are never dereferenced)."""
    lib = z.load_library()
    plan = z.Plan([100, 8], [0, 1], 1, 0)
    h = plan.handle
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    nan = float("nan")
    hp = z.binding._Hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 1.0)
    # the arena pair
    assert lib.zero1_micro_norm(None, fake, 1.0, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_micro_norm(h, fake, 0.0, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL    # divisor
    assert lib.zero1_micro_norm(h, fake, nan, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_micro_norm(h, fake, 1.0, -1.0, fake, 64, fake, None) == z.ZERO1_EINVAL   # extra_sumsq
    assert lib.zero1_micro_norm(h, fake, 1.0, 0.0, fake, 64, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_micro_norm(h, fake, 1.0, 0.0, fake, 64, odd, None) == z.ZERO1_EALIGN
    assert lib.zero1_micro_norm(h, None, 1.0, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_micro_norm(h, fake, 1.0, 0.0, fake, 4, fake, None) == z.ZERO1_EINVAL    # workspace
    assert lib.zero1_micro_norm(h, odd, 1.0, 0.0, fake, 64, fake, None) == z.ZERO1_EALIGN
    st = [h, fake, fake, fake, fake]
    assert lib.zero1_step_accumulate(*st, fake, 1.0, fake, None, 1, None, None) == z.ZERO1_EINVAL   # no hparams
    assert lib.zero1_step_accumulate(*st, fake, 1.0, fake, ctypes.byref(hp), 0, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_step_accumulate(*st, fake, nan, fake, ctypes.byref(hp), 1, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_step_accumulate(*st, odd, 1.0, fake, ctypes.byref(hp), 1, None, None) == z.ZERO1_EALIGN
    # the tensor-list pair
    assert lib.zero1_list_micro_norm(None, fake, fake, 1.0, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_micro_norm(h, fake, fake, 0.0, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_micro_norm(h, fake, fake, 1.0, nan, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_micro_norm(h, fake, fake, 1.0, 0.0, fake, 64, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_micro_norm(h, fake, fake, 1.0, 0.0, fake, 64, odd, None) == z.ZERO1_EALIGN
    assert lib.zero1_list_micro_norm(h, None, fake, 1.0, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL  # table
    assert lib.zero1_list_micro_norm(h, fake, None, 1.0, 0.0, fake, 64, fake, None) == z.ZERO1_EINVAL  # lists
    assert lib.zero1_list_micro_norm(h, fake, odd, 1.0, 0.0, fake, 64, fake, None) == z.ZERO1_EALIGN
    assert lib.zero1_list_micro_norm(h, fake, fake, 1.0, 0.0, fake, 4, fake, None) == z.ZERO1_EINVAL  # workspace
    lt = [h, fake, fake, fake, fake, fake]
    assert lib.zero1_list_step_accumulate(*lt, fake, 1.0, fake, None, 1, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_step_accumulate(*lt, fake, 1.0, fake, ctypes.byref(hp), 0, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_step_accumulate(*lt, None, 1.0, fake, ctypes.byref(hp), 1, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_step_accumulate(*lt, fake, nan, fake, ctypes.byref(hp), 1, None, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_step_accumulate(*lt, odd, 1.0, fake, ctypes.byref(hp), 1, None, None) == z.ZERO1_EALIGN
    assert lib.zero1_list_step_accumulate(h, fake, None, fake, fake, fake, fake, 1.0, fake, ctypes.byref(hp), 1,
                                          None, None) == z.ZERO1_EINVAL   # no master list
    assert lib.zero1_last_cuda_error().decode() == ""


def test_binding_refuses_cpu_tensors(z):
    import torch
    plan = z.Plan([64], [0], 1, 0)
    with pytest.raises(ValueError):
        z.accumulate(plan, torch.zeros(64), torch.zeros(64, dtype=torch.bfloat16))


def test_grouped_plan_layout_and_scales(z):
    numels = [10, 20, 30, 40, 50]
    groups = [4, 0, 4, 2, 0]
    lr = [1.0, 2.0, 0.5, 1.0, 0.25, 1.0, 1.0, 1.0]
    wd = [1.0, 1.0, 0.0, 1.0, 0.5, 1.0, 1.0, 1.0]
    plan = z.Plan(numels, groups=groups, lr_scale=lr, wd_scale=wd)
    L = plan.layout()
    # arena order: group 0 (tensors 1, 4: 20 -> 24, 50 -> 56), group 2 (tensor 3: 40),
    # group 4 (tensors 0, 2: 10 -> 16, 30 -> 32); every shard padded to a multiple of 8
    assert L.offsets.tolist() == [120, 0, 136, 80, 24]
    assert plan.group_range(0) == (0, 80) and plan.group_range(2) == (80, 120) and plan.group_range(4) == (120, 168)
    assert plan.group_range(1) == (80, 80) and plan.group_range(7) == (168, 168)
    for g in range(8):
        assert plan.group_scales(g) == (lr[g], wd[g])
    # defaults: lr 1 everywhere, no decay only in group 1
    d = z.Plan(numels, groups=groups)
    assert [d.group_scales(g) for g in range(3)] == [(1.0, 1.0), (1.0, 0.0), (1.0, 1.0)]
    assert z.Plan(numels, [0, 1, 0, 1, 0]).layout().no_decay.tolist() == [0, 1, 0, 1, 0]


def test_grouped_plan_rejects_bad_groups_and_scales(z):
    with pytest.raises(z.Zero1Error):
        z.Plan([4, 4], groups=[0, 8])
    with pytest.raises(z.Zero1Error):
        z.Plan([4, 4], groups=[0, 1], lr_scale=[1.0] * 7 + [-1.0])
    with pytest.raises(z.Zero1Error):
        z.Plan([4, 4], groups=[0, 1], wd_scale=[float("nan")] + [1.0] * 7)
    with pytest.raises(ValueError):
        z.Plan([4, 4], no_decay=[0, 1], groups=[0, 1])


def test_lr_schedule_closed_forms(z):
    lr, wu, dec, mn = 3e-3, 2000, 100000, 3e-4  # the Nanotron guide's scheduler settings
    assert z.lr_at(1, lr, wu, dec, mn) == lr / wu
    assert z.lr_at(wu, lr, wu, dec, mn) == lr
    assert abs(z.lr_at(wu + dec // 2, lr, wu, dec, mn) - (lr + mn) / 2) < 1e-15
    assert z.lr_at(wu + dec, lr, wu, dec, mn) == mn and z.lr_at(wu + dec + 5, lr, wu, dec, mn) == mn
    assert abs(z.lr_at(wu + dec // 4, lr, wu, dec, mn, "linear") - (mn + 0.75 * (lr - mn))) < 1e-15
    assert z.lr_at(wu + 7, lr, wu, dec, mn, "constant") == lr
    vals = [z.lr_at(t, lr, wu, dec, mn) for t in range(wu, wu + dec + 1, 997)]
    assert all(a >= b for a, b in zip(vals, vals[1:]))
    with pytest.raises(ValueError):
        z.lr_at(0, lr, wu, dec, mn)
    with pytest.raises(ValueError):  # an unknown curve is refused even where it would not be used
        z.lr_at(1, lr, wu, 0, mn, "exponential")


def test_mup_groups_follow_the_hidden_width_rule(z):
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    names = get_workload("smollm135m").params.names
    groups, lr_scale, wd_scale = z.mup_groups(names, d_model=576)
    kinds = dict(zip(names, groups))
    assert kinds["embed_tokens.weight"] == 2 and kinds["norm.weight"] == 1
    assert kinds["layers.3.mlp.up_proj.weight"] == 0 and kinds["layers.0.input_layernorm.weight"] == 1
    assert lr_scale[0] == 1 / 576 and lr_scale[1] == lr_scale[2] == 1.0  # eta_hidden = eta_0 / d_model
    assert wd_scale[1] == 0.0 and wd_scale[0] == wd_scale[2] == 1.0
    assert z.mup_groups(names, d_model=576, base_d_model=64)[1][0] == 64 / 576


@pytest.mark.parametrize("name", ["toy", "llama8b", "ragged"])
def test_layout_table_covers_the_shard_in_16k_runs(z, name):
    w = get_workload(name)
    plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank)
    _, count, _ = oracle.plan(w.params.numels, w.dp_size, w.dp_rank)
    runs = int(np.sum((count + 16383) // 16384))
    assert z.load_library().zero1_layout_table_bytes(plan.handle) == 24 * runs


def test_layout_calls_reject_bad_arguments_before_any_launch(z):
    lib = z.load_library()
    plan = z.Plan([100, 8], [0, 1], 1, 0)
    fake = ctypes.c_void_p(0x10000)
    assert lib.zero1_shard_gather(plan.handle, fake, fake, fake, 3, None) == z.ZERO1_EINVAL      # elem_bytes
    assert lib.zero1_shard_gather(plan.handle, None, fake, fake, 4, None) == z.ZERO1_EINVAL      # no table
    assert lib.zero1_shard_gather(plan.handle, fake, fake, ctypes.c_void_p(0x10004), 4, None) == z.ZERO1_EALIGN
    assert lib.zero1_shard_scatter(plan.handle, fake, fake, ctypes.c_void_p(0x10001), 2, None) == z.ZERO1_EALIGN
    assert lib.zero1_layout_table_upload(plan.handle, fake, 8, None) == z.ZERO1_EINVAL           # too small
    empty = z.Plan([0], [0], 1, 0)
    assert lib.zero1_layout_table_bytes(empty.handle) == 0
    assert lib.zero1_shard_gather(empty.handle, None, None, None, 4, None) == z.ZERO1_OK


def test_step_scalars_on_the_host(z):
    import struct
    plan = z.Plan([100, 8], groups=[0, 3], lr_scale=[1, 1, 1, 0.5, 1, 1, 1, 1], wd_scale=[1, 1, 1, 0, 1, 1, 1, 1])
    v = struct.unpack("<16f6fd", z.step_scalars(plan, z.Hparams(lr=1e-3, beta1=0.9, beta2=0.99, eps=1e-8,
                                                                weight_decay=0.1, clip_grad=2.0), 1))
    stepsize, dfac, rest, clip = v[:8], v[8:16], v[16:22], v[22]
    f32 = lambda x: struct.unpack("<f", struct.pack("<f", x))[0]  # noqa: E731
    assert stepsize[0] == f32(1e-3 / (1 - 0.9)) and stepsize[3] == f32(0.5e-3 / (1 - 0.9))
    assert dfac[0] == f32(1 - 1e-3 * 0.1) and dfac[3] == 1.0
    assert rest == (f32(0.9), f32(0.99), f32(1 - 0.9), f32(1 - 0.99), f32(1e-8), f32((1 - 0.99) ** 0.5))
    assert clip == 2.0
    with pytest.raises(z.Zero1Error):
        z.step_scalars(plan, z.Hparams(beta1=1.0), 1)
    with pytest.raises(z.Zero1Error):
        z.step_scalars(plan, z.Hparams(), 0)


def test_fused_pass_rejects_a_bad_divisor_before_any_launch(z):
    lib = z.load_library()
    plan = z.Plan([100, 8], [0, 1], 1, 0)
    fake = ctypes.c_void_p(0x10000)
    arr = (ctypes.c_void_p * 1)(0x20000)
    for d in (0.0, -2.0, float("nan"), float("inf"), 1e300, 1e-300):  # the last two leave fp32
        rc = lib.zero1_accumulate_norm(plan.handle, fake, arr, 1, 1, d, 0.0, fake, 64, fake, None)
        assert rc == z.ZERO1_EINVAL, d


@pytest.mark.parametrize("name", ["toy", "llama8b", "ragged"])
def test_list_table_has_one_16_byte_entry_per_run(z, name):
    w = get_workload(name)
    plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank)
    _, count, _ = oracle.plan(w.params.numels, w.dp_size, w.dp_rank)
    runs = int(np.sum((count + 16383) // 16384))
    lib = z.load_library()
    assert lib.zero1_list_table_bytes(plan.handle) == 16 * runs
    assert lib.zero1_list_workspace_bytes(plan.handle) == 8 * runs == plan.list_workspace_bytes


def test_list_calls_reject_bad_arguments_before_any_launch(z):
    lib = z.load_library()
    plan = z.Plan([100, 8, 0], [0, 1, 0], 1, 0)
    h = plan.handle
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    # pointer-list upload: entries of non-empty shards must be non-NULL and naturally aligned
    ok = (ctypes.c_void_p * 3)(0x20000, 0x30000, None)        # the empty tensor's entry may be NULL
    null = (ctypes.c_void_p * 3)(0x20000, None, None)
    odd4 = (ctypes.c_void_p * 3)(0x20000, 0x30002, None)
    assert lib.zero1_list_ptrs_upload(h, null, 1, 4, fake, 64, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_ptrs_upload(h, odd4, 1, 4, fake, 64, None) == z.ZERO1_EALIGN
    assert lib.zero1_list_ptrs_upload(h, odd4, 1, 3, fake, 64, None) == z.ZERO1_EINVAL    # elem_bytes
    assert lib.zero1_list_ptrs_upload(h, ok, 0, 4, fake, 64, None) == z.ZERO1_EINVAL       # n_lists
    assert lib.zero1_list_ptrs_upload(h, ok, 17, 4, fake, 64, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_ptrs_upload(h, ok, 1, 4, fake, 16, None) == z.ZERO1_EINVAL       # too small
    assert lib.zero1_list_ptrs_upload(h, ok, 1, 4, odd, 64, None) == z.ZERO1_EALIGN
    assert lib.zero1_list_ptrs_upload(h, None, 1, 4, fake, 64, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_table_upload(h, fake, 8, None) == z.ZERO1_EINVAL                 # too small
    assert lib.zero1_list_table_upload(h, odd, 64, None) == z.ZERO1_EALIGN
    # compute calls
    assert lib.zero1_list_accumulate(h, fake, fake, fake, 0, 1, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_accumulate(h, fake, fake, fake, 17, 1, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_accumulate(h, None, fake, fake, 1, 1, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_accumulate(h, fake, odd, fake, 1, 1, None) == z.ZERO1_EALIGN
    assert lib.zero1_list_accumulate(h, fake, fake, None, 1, 1, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_workspace_bytes(h) == 16
    for d in (0.0, -1.0, float("nan"), float("inf"), 1e300, 1e-300):
        assert lib.zero1_list_accumulate_norm(h, fake, fake, fake, 1, 1, d, 0.0, fake, 64, fake, None) == \
            z.ZERO1_EINVAL
    assert lib.zero1_list_accumulate_norm(h, fake, fake, fake, 1, 1, 1.0, 0.0, fake, 8, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_grad_norm(h, fake, fake, 0.0, fake, 8, fake, None) == z.ZERO1_EINVAL  # workspace
    assert lib.zero1_list_grad_norm(h, fake, fake, -1.0, fake, 64, fake, None) == z.ZERO1_EINVAL
    assert lib.zero1_list_grad_norm(h, fake, fake, 0.0, odd, 64, fake, None) == z.ZERO1_EALIGN
    assert lib.zero1_list_grad_norm(h, fake, fake, 0.0, fake, 64, None, None) == z.ZERO1_EINVAL
    hp = z.binding._Hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, 1.0)
    five = [fake] * 5
    assert lib.zero1_list_step(h, fake, *five, ctypes.byref(hp), 0, None, None) == z.ZERO1_EINVAL  # t < 1
    assert lib.zero1_list_step(h, fake, fake, fake, fake, odd, fake, ctypes.byref(hp), 1, None, None) == \
        z.ZERO1_EALIGN
    assert lib.zero1_list_step(h, fake, fake, fake, None, fake, fake, ctypes.byref(hp), 1, None, None) == \
        z.ZERO1_EINVAL
    bad = z.binding._Hparams(3e-4, 0.9, 1.0, 1e-8, 0.1, 1.0)
    assert lib.zero1_list_step(h, fake, *five, ctypes.byref(bad), 1, None, None) == z.ZERO1_EINVAL
    # an all-empty plan: nothing to do, NULL lists accepted
    empty = z.Plan([0, 0], [0, 1], 1, 0)
    assert lib.zero1_list_table_bytes(empty.handle) == 0
    assert lib.zero1_list_table_upload(empty.handle, None, 0, None) == z.ZERO1_OK
    assert lib.zero1_list_accumulate(empty.handle, None, None, None, 1, 1, None) == z.ZERO1_OK
    assert lib.zero1_list_step(empty.handle, None, None, None, None, None, None, ctypes.byref(hp), 1, None,
                               None) == z.ZERO1_OK
    none = (ctypes.c_void_p * 2)(None, None)
    assert lib.zero1_list_ptrs_upload(empty.handle, none, 1, 4, None, 0, None) == z.ZERO1_EINVAL  # no destination


def test_binding_signatures_match_the_header(z):
    """Every declared entry point has ctypes argument types of the header's kinds and count
    (pointer, int32, int64, size_t, double), so no argument is passed at the wrong width."""
    src = ""
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src += open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)

    def c_kind(a):
        if "*" in a or "[" in a:
            return "ptr"
        for key, k in (("size_t", "size"), ("int64_t", "i64"), ("double", "f64"), ("int32_t", "i32")):
            if key in a:
                return k
        return "i32" if re.match(r"(const\s+)?int\b", a) else a

    def py_kind(t):
        if t is ctypes.c_void_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
            return "ptr"
        return {ctypes.c_int32: "i32", ctypes.c_int64: "i64", ctypes.c_size_t: "size", ctypes.c_double: "f64"}.get(t, t)

    lib = z.load_library()
    checked = 0
    for m in re.finditer(r"\b(zero1_\w+)\s*\(([^;]*?)\)\s*;", src, re.S):
        name, args = m.group(1), m.group(2).strip()
        args = [] if args in ("", "void") else [a.strip() for a in args.split(",")]
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None, name
        assert [c_kind(a) for a in args] == [py_kind(t) for t in argtypes], name
        checked += 1
    assert checked == len(declared_functions())


def test_plan_sizes_are_the_librarys(z):
    """The Python Plan reads its sizes once at creation; they must be the library's own answers."""
    lib = z.load_library()
    w = get_workload("ragged")
    plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank)
    h = plan.handle
    assert plan.num_tensors == lib.zero1_plan_num_tensors(h) == len(w.params.numels)
    assert plan.total_numel == lib.zero1_plan_total_numel(h)
    assert plan.local_numel == lib.zero1_plan_local_numel(h)
    assert plan.arena_numel == lib.zero1_plan_arena_numel(h)
    assert plan.workspace_bytes == lib.zero1_workspace_bytes(h)
    assert plan.list_workspace_bytes == lib.zero1_list_workspace_bytes(h)


def test_plan_for_rank_is_the_same_list_sharded_for_another_rank():
    """DataParallelStep builds the other ranks' plans with Plan.for_rank: the same tensors,
    groups and scales, each rank's own shard (equal to a plan made directly for that rank)."""
    import zero_sharded_mixed_local_gb300 as z
    numels = [5000, 17, 64, 3, 999, 1]
    for kw in ({"no_decay": [0, 1, 0, 1, 0, 0]},
               {"groups": [3, 0, 3, 1, 2, 0], "lr_scale": [1.0, 0.5, 2.0] + [1.0] * 5,
                "wd_scale": [1.0, 0.0, 0.25] + [1.0] * 5}):
        base = z.Plan(numels, dp_size=4, dp_rank=1, **kw)
        for r in range(4):
            a, b = base.for_rank(r), z.Plan(numels, dp_size=4, dp_rank=r, **kw)
            assert (a.dp_size, a.dp_rank, a.local_numel, a.arena_numel) == (4, r, b.local_numel, b.arena_numel)
            la, lb = a.layout(), b.layout()
            for f in ("shard_start", "counts", "offsets", "no_decay"):
                assert np.array_equal(getattr(la, f), getattr(lb, f)), (r, f)
            assert [a.group_scales(g) for g in range(8)] == [b.group_scales(g) for g in range(8)]
