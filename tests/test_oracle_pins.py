"""Pins for the CPU oracle: each test checks it against something other than
itself -- a library routine, a closed form of the mathematics, a value the
pages print, or brute force -- so that a dropped term, a wrong sign or index,
or a swapped operand anywhere in the oracle fails at least one of them.

All CPU, no GPU (run under -m "not gpu").
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def f32_bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def ulp_diff(a, b):
    """Distance in fp32 ulps (ordered-integer metric), elementwise."""
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


# --------------------------------------------------------------------------
# Shard split: brute force against numpy.array_split, which implements the
# same "first n mod dp ranks get one more" rule independently.
# --------------------------------------------------------------------------
def test_shard_split_matches_array_split_bruteforce(oracle_mod):
    for n in range(0, 65):
        idx = np.arange(n)
        for dp in range(1, 10):
            parts = np.array_split(idx, dp)
            covered = []
            for r in range(dp):
                s, c = oracle_mod.shard_range(n, dp, r)
                assert c == len(parts[r]), (n, dp, r)
                if c:
                    assert s == parts[r][0], (n, dp, r)
                covered.extend(range(s, s + c))
            assert covered == list(range(n))


def test_shard_split_large_counts(oracle_mod):
    n = 8_030_261_248 // 7 * 7 + 5
    for dp in (2, 7, 8, 64):
        tot = 0
        prev_end = 0
        for r in range(dp):
            s, c = oracle_mod.shard_range(n, dp, r)
            assert s == prev_end
            assert c in (n // dp, n // dp + 1)
            prev_end = s + c
            tot += c
        assert tot == n and prev_end == n


def test_plan_sums_shards(oracle_mod):
    numels = [1, 2, 3, 7, 8, 9, 1000, 4097]
    for dp in (1, 2, 3, 4, 8):
        per_rank = []
        for r in range(dp):
            start, count, local = oracle_mod.plan(numels, dp, r)
            assert local == int(count.sum())
            per_rank.append(count)
        np.testing.assert_array_equal(np.sum(per_rank, axis=0), numels)


# --------------------------------------------------------------------------
# Memory accounting: the figures the pages print.
# --------------------------------------------------------------------------
def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_memory_accounting_matches_printed_figures(oracle_mod):
    rows = _golden_rows("zero1_memory_accounting.txt")
    assert len(rows) >= 8
    for params, dp, gb, field, expected, rounding, src in rows:
        params, dp, gb, expected = int(params), int(dp), int(gb), int(expected)
        _, _, local = oracle_mod.plan([params], dp, 0)
        got = oracle_mod.zero1_bytes(params, local, gb)[field]
        if rounding == "exact":
            assert got == expected, (src, field, got, expected)
        else:
            unit = int(rounding)
            assert abs(got - expected) < unit, (src, field, got, expected)


def test_memory_accounting_optimizer_share_and_18_byte_variant(oracle_mod):
    b = oracle_mod.zero1_bytes(1000, 1000, 2)
    assert b["optimizer"] / b["total"] == 0.75  # 12 of 16 bytes
    # the itemised 2+4+4+4+4 list of the Nanotron guide (fp32 gradient) sums to 18
    assert oracle_mod.zero1_bytes(1, 1, 4)["total"] == 18


# --------------------------------------------------------------------------
# bf16 conversions.
# --------------------------------------------------------------------------
def test_bf16_widening_exhaustive_vs_torch(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = np.array([oracle_mod.bf16_to_f32(int(b)) for b in bits[::37]], np.float32)
    r = ref[::37]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(f32_bits(got[~nan]), f32_bits(r[~nan]))


def test_bf16_rne_golden_cases(oracle_mod):
    for f_hex, b_hex, *_ in _golden_rows("bf16_rne_cases.txt"):
        x = np.array([int(f_hex, 16)], np.uint32).view(np.float32)
        got = int(oracle_mod.bf16_rne(x)[0])
        assert got == int(b_hex, 16), (f_hex, hex(got), b_hex)


def test_bf16_rne_vs_torch_random(oracle_mod):
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[~np.isnan(x)]
    got = oracle_mod.bf16_rne(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rne_nan_stays_nan(oracle_mod):
    for pat in (0x7FC00000, 0x7F800001, 0xFF800001, 0x7FFFFFFF):
        x = np.array([pat], np.uint32).view(np.float32)
        b = int(oracle_mod.bf16_rne(x)[0])
        assert (b & 0x7F80) == 0x7F80 and (b & 0x007F) != 0 and (b >> 15) == (pat >> 31)


# --------------------------------------------------------------------------
# Gradient accumulation.
# --------------------------------------------------------------------------
def _to_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_accumulate_integer_values_exact(oracle_mod):
    rng = np.random.default_rng(2)
    K, n = 8, 4099
    ints = rng.integers(-256, 257, size=(K, n))
    micros = [_to_bf16_bits(ints[k]) for k in range(K)]
    grad = np.full(n, 123.0, np.float32)  # overwritten by the first micro-batch
    oracle_mod.accumulate_all(grad, micros)
    np.testing.assert_array_equal(grad, ints.sum(axis=0).astype(np.float32))


def test_accumulate_matches_sequential_numpy_float32(oracle_mod):
    rng = np.random.default_rng(3)
    K, n = 5, 10007
    micros = [_to_bf16_bits(rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 3, n)) for _ in range(K)]
    widened = [np.asarray(m, np.uint32).__lshift__(16).view(np.float32) for m in micros]
    ref = widened[0].copy()
    for k in range(1, K):
        ref = ref + widened[k]  # numpy float32 add: one IEEE rounding per element
    grad = np.zeros(n, np.float32)
    oracle_mod.accumulate_all(grad, micros)
    assert np.array_equal(f32_bits(grad), f32_bits(ref))


def test_accumulate_overwrite_keeps_negative_zero(oracle_mod):
    grad = np.ones(3, np.float32)
    oracle_mod.accumulate(grad, np.array([0x8000, 0x0000, 0xBF80], np.uint16), overwrite=True)
    assert f32_bits(grad).tolist() == [0x80000000, 0, 0xBF800000]
    oracle_mod.accumulate(grad, np.array([0x3F80, 0x3F80, 0x3F80], np.uint16), overwrite=False)
    assert grad.tolist() == [1.0, 1.0, 0.0]


# --------------------------------------------------------------------------
# Norm and clipping.
# --------------------------------------------------------------------------
def test_sumsq_closed_forms(oracle_mod):
    assert oracle_mod.sumsq(np.ones(1_000_003, np.float32)) == 1_000_003.0
    assert oracle_mod.sumsq(np.zeros(0, np.float32)) == 0.0
    x = np.arange(1, 1001, dtype=np.float32)
    assert oracle_mod.sumsq(x) == 1000 * 1001 * 2001 // 6


def test_sumsq_vs_exactly_rounded_fsum(oracle_mod):
    """math.fsum gives the correctly rounded sum of the (exact) squares; the oracle
    must be within a few double ulps of it, at any length and scale mix."""
    rng = np.random.default_rng(4)
    for n, spread in ((200_000, 6), (1_000_003, 2), (3, 30)):
        x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-spread / 2, spread / 2, n)).astype(np.float32)
        exact = math.fsum(float(v) * float(v) for v in x)
        got = oracle_mod.sumsq(x)
        assert abs(got - exact) <= 4 * math.ulp(exact), (n, got, exact)
    assert abs(math.sqrt(got) - float(np.linalg.norm(x.astype(np.float64)))) <= 1e-12 * math.sqrt(exact)


def test_sumsq_no_drift_on_bf16_structured_squares(oracle_mod):
    """Squares of sums of bf16 values have structured low bits; summing millions of them
    must not drift (a plain running sum does, by ~1e-7 relative in fp32)."""
    rng = np.random.default_rng(12)
    n = 2_000_000
    a = _to_bf16_bits(rng.standard_normal(n) * 1e-3).astype(np.uint32) << 16
    b = _to_bf16_bits(rng.standard_normal(n) * 1e-3).astype(np.uint32) << 16
    g = (a.view(np.float32) + b.view(np.float32)).astype(np.float32)
    exact = math.fsum((g.astype(np.float64) ** 2).tolist())
    assert abs(oracle_mod.sumsq(g) - exact) <= 4 * math.ulp(exact)


def test_clip_coef_vs_torch_clip_grad_norm(oracle_mod):
    for norm_target in (0.3, 0.999, 1.0, 1.5, 4.0, 1e3):
        g = torch.full((16,), norm_target / 4.0, dtype=torch.float64)
        total = float((g * g).sum())
        p = torch.nn.Parameter(torch.zeros(16, dtype=torch.float64))
        p.grad = g.clone()
        tn = torch.nn.utils.clip_grad_norm_([p], max_norm=1.0)
        applied = float(p.grad[0] / g[0])
        ok, norm, coef = oracle_mod.clip_coef(total, 1.0)
        assert ok
        assert abs(norm - float(tn)) <= 1e-15 * norm
        assert np.float32(applied) == coef or abs(float(coef) - applied) <= 6e-8 * applied


def test_clip_inactive_and_disabled(oracle_mod):
    ok, norm, coef = oracle_mod.clip_coef(0.25, 1.0)
    assert ok and norm == 0.5 and coef == np.float32(1.0)
    ok, norm, coef = oracle_mod.clip_coef(100.0, 0.0)  # clip <= 0 disables clipping
    assert ok and coef == np.float32(1.0)
    ok, norm, coef = oracle_mod.clip_coef(100.0, 1.0)
    assert ok and coef == np.float32(1.0 / (10.0 + 1e-6))


def test_clip_nonfinite(oracle_mod):
    for bad in (float("inf"), float("nan")):
        ok, norm, coef = oracle_mod.clip_coef(bad, 1.0)
        assert not ok


# --------------------------------------------------------------------------
# AdamW: closed forms.
# --------------------------------------------------------------------------
def _one_tensor(n, no_decay=0):
    return np.array([n], np.int64), np.array([no_decay], np.uint8)


def test_adamw_step1_closed_form(oracle_mod):
    """From m = v = 0 the first bias-corrected update is lr*g/(|g|+eps)."""
    g = np.array([1e-3, -2.0, 5e-6, 1e-8, -3e-8, 0.7], np.float32)
    n = g.size
    p0 = np.linspace(-0.05, 0.05, n).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    hp = dict(HP, weight_decay=0.0)
    oracle_mod.adamw(p, m, v, g.copy(), *_one_tensor(n), hp, 1, np.float32(1.0))
    g64 = g.astype(np.float64)
    expect = p0.astype(np.float64) - hp["lr"] * g64 / (np.abs(g64) + hp["eps"])
    assert np.all(np.abs(p - expect) <= 2e-6 * hp["lr"] + 4 * np.spacing(np.abs(p0)))
    # |g| >> eps: the step size is lr, whatever the gradient's scale
    big = np.abs(g) > 1e-4
    np.testing.assert_allclose(np.abs(p0 - p)[big], hp["lr"], rtol=1e-4)
    # in general the step is lr*|g|/(|g|+eps)
    np.testing.assert_allclose(np.abs(p0 - p)[:3], hp["lr"] * np.abs(g64[:3]) / (np.abs(g64[:3]) + hp["eps"]),
                               rtol=1e-4)
    # |g| = eps gives half a step: eps sits outside the square root
    assert abs(abs(float(p0[3] - p[3])) - hp["lr"] / 2) < 1e-3 * hp["lr"]
    np.testing.assert_allclose(m, (1 - hp["beta1"]) * g64, rtol=1e-6)
    np.testing.assert_allclose(v, (1 - hp["beta2"]) * g64 * g64, rtol=1e-6)


def test_adamw_constant_gradient_every_step_same_size(oracle_mod):
    """With constant g and no decay, bias correction makes every step lr*g/(|g|+eps)."""
    n, T = 7, 25
    g = np.array([0.5, -0.1, 3.0, -7e-3, 1e-4, 2.0, -1.0], np.float32)
    p = np.zeros(n, np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    hp = dict(HP, weight_decay=0.0)
    for t in range(1, T + 1):
        before = p.copy()
        oracle_mod.adamw(p, m, v, g.copy(), *_one_tensor(n), hp, t, np.float32(1.0))
        step = (before - p).astype(np.float64)
        np.testing.assert_allclose(step, hp["lr"] * np.sign(g), rtol=2e-4)
    np.testing.assert_allclose(p, -T * hp["lr"] * np.sign(g), rtol=2e-4)


def test_adamw_alternating_gradient_second_step(oracle_mod):
    """g then -g from zero state: the second update is +lr*(1-b1)/(1+b1)*sign(g)
    (m2 = -(1-b1)^2 g, v2 = (1-b2)(1+b2) g^2 and their corrections)."""
    g = np.array([0.25, -4.0, 1.0], np.float32)
    n = g.size
    p, m, v = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    hp = dict(HP, weight_decay=0.0)
    oracle_mod.adamw(p, m, v, g.copy(), *_one_tensor(n), hp, 1, np.float32(1.0))
    p1 = p.copy()
    oracle_mod.adamw(p, m, v, (-g).copy(), *_one_tensor(n), hp, 2, np.float32(1.0))
    b1, b2 = hp["beta1"], hp["beta2"]
    expect = hp["lr"] * (1 - b1) / (1 + b1) * np.sign(g)
    np.testing.assert_allclose((p - p1).astype(np.float64), expect, rtol=1e-4)
    np.testing.assert_allclose(m, -(1 - b1) ** 2 * g.astype(np.float64), rtol=1e-6)
    np.testing.assert_allclose(v, (1 - b2) * (1 + b2) * g.astype(np.float64) ** 2, rtol=1e-6)


def test_adamw_zero_grad_is_pure_decay_bit_exact(oracle_mod):
    rng = np.random.default_rng(5)
    counts = np.array([5, 3, 8], np.int64)
    no_decay = np.array([0, 1, 0], np.uint8)
    n = int(counts.sum())
    p0 = rng.standard_normal(n).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle_mod.adamw(p, m, v, np.zeros(n, np.float32), counts, no_decay, HP, 1, np.float32(1.0))
    dfac = np.float32(1.0 - HP["lr"] * HP["weight_decay"])
    expect = p0.copy()
    expect[:5] = p0[:5] * dfac
    expect[8:] = p0[8:] * dfac
    assert np.array_equal(f32_bits(p), f32_bits(expect))
    assert not m.any() and not v.any()
    # ten decays multiply out to (1 - lr*wd)^10 up to rounding
    for t in range(2, 11):
        oracle_mod.adamw(p, m, v, np.zeros(n, np.float32), counts, no_decay, HP, t, np.float32(1.0))
    np.testing.assert_allclose(p[:5], p0[:5].astype(np.float64) * (1 - 3e-5) ** 10, rtol=1e-6)
    assert np.array_equal(p[5:8], p0[5:8])


def test_adamw_writes_bf16_rne_of_master(oracle_mod):
    rng = np.random.default_rng(6)
    n = 5000
    p = rng.standard_normal(n).astype(np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    w = np.zeros(n, np.uint16)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    oracle_mod.adamw(p, m, v, g, *_one_tensor(n), HP, 1, np.float32(1.0), w=w)
    ref = torch.from_numpy(p.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(w, ref)


# --------------------------------------------------------------------------
# AdamW: independent library implementation (torch.optim.AdamW, single-tensor
# CPU path).  It differs only in rounding order (lerp, addcmul), so agreement
# is to a few ulp of the master weights and a small relative error of m, v.
# --------------------------------------------------------------------------
def test_adamw_vs_torch_optim_adamw(oracle_mod):
    rng = np.random.default_rng(7)
    counts = np.array([300, 17, 129, 64], np.int64)
    no_decay = np.array([0, 1, 0, 1], np.uint8)
    n = int(counts.sum())
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    splits = np.cumsum(counts)[:-1]
    tparams = [torch.nn.Parameter(torch.from_numpy(x.copy())) for x in np.split(p0, splits)]
    groups = [
        {"params": [tp for tp, nd in zip(tparams, no_decay) if not nd], "weight_decay": HP["weight_decay"]},
        {"params": [tp for tp, nd in zip(tparams, no_decay) if nd], "weight_decay": 0.0},
    ]
    opt = torch.optim.AdamW(groups, lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            foreach=False, fused=False)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    gmax = np.zeros(n)
    for t in range(1, 11):
        g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-4, -1, n)).astype(np.float32)
        gmax = np.maximum(gmax, np.abs(g))
        for tp, gg in zip(tparams, np.split(g, splits)):
            tp.grad = torch.from_numpy(gg.copy())
        opt.step()
        oracle_mod.adamw(p, m, v, g, counts, no_decay, HP, t, np.float32(1.0))
    tp_all = np.concatenate([tp.detach().numpy() for tp in tparams])
    tm = np.concatenate([opt.state[tp]["exp_avg"].numpy() for tp in tparams])
    tv = np.concatenate([opt.state[tp]["exp_avg_sq"].numpy() for tp in tparams])
    # master: a few ulp of p, plus a 1e-5 relative share of the ten lr-sized updates (where |p| is
    # near lr the rounding differences of m and v dominate the ulp of p)
    bound = 4 * np.spacing(np.abs(tp_all)) + 1e-5 * HP["lr"] * 10
    assert np.all(np.abs(p - tp_all) <= bound)
    assert np.median(ulp_diff(p, tp_all)) <= 1
    # m, v: rounding differences of a few ulp of the largest gradient term that fed the element
    # (a relative bound on m fails where sign changes cancel it)
    assert np.all(np.abs(m - tm) <= 8 * 2.0**-24 * gmax)
    assert np.all(np.abs(v - tv) <= 8 * 2.0**-24 * gmax * gmax)


# --------------------------------------------------------------------------
# The whole step.
# --------------------------------------------------------------------------
def _rand_problem(rng, counts, K, sigma):
    n = int(sum(counts))
    micros = [_to_bf16_bits(rng.standard_normal(n) * sigma) for _ in range(K)]
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    return n, micros, p


def test_full_step_clip_below_threshold_is_identity(oracle_mod):
    rng = np.random.default_rng(8)
    counts = np.array([100, 28, 1000], np.int64)
    nd = np.array([0, 1, 0], np.uint8)
    n, micros, p0 = _rand_problem(rng, counts, 3, 1e-3)
    res = []
    for clip in (1.0, 0.0):
        p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        w = np.zeros(n, np.uint16)
        info = oracle_mod.full_step(p, m, v, micros, counts, nd, HP, 1, clip, w=w)
        assert info["norm"] < 1.0 and info["coef"] == 1.0
        res.append((p, m, v, w))
    for a, b in zip(*res):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_full_step_clip_active_scales_to_threshold(oracle_mod):
    """Above the threshold the gradient the update sees has norm clip*norm/(norm+1e-6):
    after a step from zero state, m = (1-b1)*g_clipped."""
    rng = np.random.default_rng(9)
    counts = np.array([4096, 64, 999], np.int64)
    nd = np.array([0, 1, 0], np.uint8)
    n, micros, p0 = _rand_problem(rng, counts, 4, 0.05)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    info = oracle_mod.full_step(p, m, v, micros, counts, nd, HP, 1, 1.0)
    assert info["norm"] > 2.0 and info["coef"] < 1.0
    g_seen = m.astype(np.float64) / (1 - HP["beta1"])
    clipped_norm = float(np.linalg.norm(g_seen))
    assert abs(clipped_norm - 1.0 * info["norm"] / (info["norm"] + 1e-6)) < 1e-5


def test_full_step_nonfinite_grad_skips_update(oracle_mod):
    rng = np.random.default_rng(10)
    counts = np.array([50, 50], np.int64)
    nd = np.array([0, 0], np.uint8)
    n, micros, p0 = _rand_problem(rng, counts, 2, 1e-3)
    micros[1][17] = 0x7FC0  # NaN
    p, m, v = p0.copy(), np.ones(n, np.float32), np.ones(n, np.float32)
    w = np.full(n, 7, np.uint16)
    info = oracle_mod.full_step(p, m, v, micros, counts, nd, HP, 1, 1.0, w=w)
    assert not info["applied"]
    assert np.array_equal(p, p0) and (m == 1).all() and (v == 1).all() and (w == 7).all()


def test_shard_concatenation_invariant(oracle_mod):
    """Stepping each rank's shard with the global sum of squares gives exactly
    the unsharded step, tensor by tensor (the step is element-wise given the norm)."""
    rng = np.random.default_rng(11)
    numels = [1, 3, 8, 17, 64, 1000, 2, 513]
    nd = np.array([0, 1, 0, 0, 1, 0, 0, 0], np.uint8)
    full_counts = np.array(numels, np.int64)
    N, K = int(sum(numels)), 3
    full_micros = [_to_bf16_bits(rng.standard_normal(N) * 0.3) for _ in range(K)]  # clip active
    p0 = (rng.standard_normal(N) * 0.02).astype(np.float32)
    tstart = np.concatenate([[0], np.cumsum(numels)[:-1]])

    p, m, v, w = p0.copy(), np.zeros(N, np.float32), np.zeros(N, np.float32), np.zeros(N, np.uint16)
    ref = oracle_mod.full_step(p, m, v, full_micros, full_counts, nd, HP, 1, 1.0, w=w)
    assert ref["coef"] < 1.0

    for dp in (2, 3, 4, 8):
        shards = []
        for r in range(dp):
            start, count, local = oracle_mod.plan(numels, dp, r)
            idx = np.concatenate([np.arange(tstart[i] + start[i], tstart[i] + start[i] + count[i])
                                  for i in range(len(numels))]).astype(np.int64)
            shards.append((count, idx))
        sums = []
        for count, idx in shards:
            g = np.zeros(idx.size, np.float32)
            oracle_mod.accumulate_all(g, [mb[idx] for mb in full_micros])
            sums.append(oracle_mod.sumsq(g))
        P, M, V, W = [np.zeros(N, dt) for dt in (np.float32, np.float32, np.float32, np.uint16)]
        for r, (count, idx) in enumerate(shards):
            extra = sum(s for q, s in enumerate(sums) if q != r)
            pp, mm, vv, ww = p0[idx].copy(), np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32), \
                np.zeros(idx.size, np.uint16)
            info = oracle_mod.full_step(pp, mm, vv, [mb[idx] for mb in full_micros], count, nd, HP, 1, 1.0,
                                        extra_sumsq=extra, w=ww)
            assert info["coef"] == ref["coef"]
            P[idx], M[idx], V[idx], W[idx] = pp, mm, vv, ww
        for a, b in ((P, p), (M, m), (V, v), (W, w)):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), dp


# --------------------------------------------------------------------------
# Per-tensor learning-rate / weight-decay multipliers.
# --------------------------------------------------------------------------
def test_adamw_scaled_step1_moves_each_tensor_by_its_own_lr(oracle_mod):
    """From zero state, step 1 moves every element by lr_i*g/(|g|+eps) after decay by 1-lr_i*wd_i."""
    counts = np.array([5, 4, 3], np.int64)
    lr_scale = np.array([1.0, 1.0 / 64, 4.0])
    wd_scale = np.array([1.0, 0.0, 0.5])
    g = np.array([0.3, -0.2, 1.0, 2e-3, -4.0, 0.7, 0.1, 1e-2, -1e-3, 3.0, -0.5, 0.25], np.float32)
    p0 = np.linspace(-0.03, 0.03, g.size).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(g.size, np.float32), np.zeros(g.size, np.float32)
    oracle_mod.adamw_scaled(p, m, v, g.copy(), counts, lr_scale, wd_scale, HP, 1, np.float32(1.0))
    lr_i = np.repeat(HP["lr"] * lr_scale, counts)
    wd_i = np.repeat(HP["weight_decay"] * wd_scale, counts)
    g64 = g.astype(np.float64)
    expect = p0 * (1 - lr_i * wd_i) - lr_i * g64 / (np.abs(g64) + HP["eps"])
    np.testing.assert_allclose(p, expect, rtol=0, atol=1e-6 * lr_i.max())
    np.testing.assert_allclose(np.abs((p0 * (1 - lr_i * wd_i)) - p) / lr_i, 1.0, rtol=1e-4)


def test_adamw_scaled_reduces_to_no_decay_flags(oracle_mod):
    rng = np.random.default_rng(13)
    counts = np.array([100, 7, 64, 1], np.int64)
    nd = np.array([0, 1, 0, 1], np.uint8)
    n = int(counts.sum())
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    outs = []
    for scaled in (False, True):
        p, m, v, w = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
        for t in (1, 2, 3):
            if scaled:
                oracle_mod.adamw_scaled(p, m, v, g.copy(), counts, np.ones(4), 1.0 - nd, HP, t, np.float32(0.5), w=w)
            else:
                oracle_mod.adamw(p, m, v, g.copy(), counts, nd, HP, t, np.float32(0.5), w=w)
        outs.append((p, m, v, w))
    for a, b in zip(*outs):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_adamw_scaled_vs_torch_param_groups(oracle_mod):
    """torch.optim.AdamW with one param group per (lr, weight decay) pair."""
    rng = np.random.default_rng(14)
    counts = np.array([200, 33, 128], np.int64)
    lr_scale = np.array([1.0, 0.125, 2.0])
    wd_scale = np.array([1.0, 0.0, 0.25])
    n = int(counts.sum())
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    splits = np.cumsum(counts)[:-1]
    tparams = [torch.nn.Parameter(torch.from_numpy(x.copy())) for x in np.split(p0, splits)]
    groups = [{"params": [tp], "lr": HP["lr"] * ls, "weight_decay": HP["weight_decay"] * ws}
              for tp, ls, ws in zip(tparams, lr_scale, wd_scale)]
    opt = torch.optim.AdamW(groups, lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            foreach=False, fused=False)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    lr_el = np.repeat(HP["lr"] * lr_scale, counts)
    for t in range(1, 8):
        g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-4, -1, n)).astype(np.float32)
        for tp, gg in zip(tparams, np.split(g, splits)):
            tp.grad = torch.from_numpy(gg.copy())
        opt.step()
        oracle_mod.adamw_scaled(p, m, v, g, counts, lr_scale, wd_scale, HP, t, np.float32(1.0))
    tp_all = np.concatenate([tp.detach().numpy() for tp in tparams])
    bound = 4 * np.spacing(np.abs(tp_all)) + 1e-5 * lr_el * 7
    assert np.all(np.abs(p - tp_all) <= bound)


# --------------------------------------------------------------------------
# Division of the reduced gradient by the world size.
# --------------------------------------------------------------------------
def test_divide_matches_numpy_float32_division(oracle_mod):
    rng = np.random.default_rng(15)
    g = (rng.standard_normal(100_003) * 10.0 ** rng.uniform(-30, 30, 100_003)).astype(np.float32)
    for d in (1.0, 2.0, 3.0, 7.0, 8.0, 64.0, 1.5):
        x = g.copy()
        oracle_mod.divide(x, d)
        assert np.array_equal(f32_bits(x), f32_bits(g / np.float32(d))), d
    x = g.copy()
    oracle_mod.divide(x, 1.0)
    assert np.array_equal(f32_bits(x), f32_bits(g))
    x = np.array([3.0, -9.0, 0.75], np.float32)
    oracle_mod.divide(x, 3.0)
    assert x.tolist() == [1.0, -3.0, 0.25]


# A four-element case worked by hand ("ZeRO-1 风格的 Distributed Optimizer", section 6.6 hyper-parameters
# beta1 0.9, beta2 0.95, eps 1e-8, weight decay 0.1, clip_grad 1.0; lr 0.1 for round numbers).  Tensor A
# (decayed) holds elements 0-1, tensor B (a norm weight, no decay) elements 2-3; bf16-exact gradients.
#   step 1: g = [0.375, -0.5, 0, 1.5]; sum of squares 0.140625 + 0.25 + 2.25 = 2.640625, norm 1.625,
#           clipped by c = 1/(1.625 + 1e-6).  From m = v = 0 the bias-corrected update is g/|g| (eps is
#           ~1e-8 of |cg| and vanishes in fp32): +1, -1, 0, +1; A decays by 1 - 0.1*0.1 = 0.99, B does not:
#           p = [0.5*0.99 - 0.1, -0.25*0.99 + 0.1, 1.0, 1.0 - 0.1] = [0.395, -0.1475, 1.0, 0.9].
#   step 2: g = [0.375, 0.5, 0, -1.5] (norm 1.625 again, same c).  Element 0 repeats its gradient, so
#           m^ = c*0.375 and sqrt(v^) = c*0.375: update 1, p = 0.395*0.99 - 0.1 = 0.29105.  Elements 1 and 3
#           flip sign: m2 = c*(0.09*g1 + 0.1*g2) = 0.01*c*g2, m^ = m2/0.19; v2 = 0.05*c^2*(0.95 + 1)*g^2,
#           v^ = v2/0.0975 = c^2*g^2: update = (0.01/0.19)*sign(g2) = 0.0526315789*sign(g2), so
#           p1 = -0.1475*0.99 - 0.1*0.0526315789 = -0.1512881579 and p3 = 0.9 + 0.00526315789 = 0.9052631579.
#           Element 2 (g = 0 twice) stays 1.0.
FOUR_HP = dict(lr=0.1, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
FOUR_P0 = [0.5, -0.25, 1.0, 1.0]
FOUR_G = ([0.375, -0.5, 0.0, 1.5], [0.375, 0.5, 0.0, -1.5])
FOUR_P = ([0.395, -0.1475, 1.0, 0.9], [0.29105, -0.1512881579, 1.0, 0.9052631579])


def test_four_element_two_step_worked_example(oracle_mod):
    p = np.array(FOUR_P0, np.float32)
    m, v = np.zeros(4, np.float32), np.zeros(4, np.float32)
    for t, (g, expect) in enumerate(zip(FOUR_G, FOUR_P), start=1):
        micro = oracle_mod.bf16_rne(np.array(g, np.float32))
        info = oracle_mod.full_step(p, m, v, [micro], [2, 2], [0, 1], FOUR_HP, t, 1.0)
        assert info["sumsq"] == 2.640625 and info["norm"] == 1.625
        assert info["coef"] == np.float32(1.0 / (1.625 + 1e-6))
        np.testing.assert_allclose(p, expect, rtol=0, atol=2.5e-7)
    # m2 = c*(0.09*g1 + 0.1*g2): 0.375*0.19 = 0.07125, 0.09*(-0.5) + 0.05 = 0.005, 0.135 - 0.15 = -0.015
    c = 1.0 / 1.625
    np.testing.assert_allclose(m[[0, 1, 3]], [c * 0.07125, c * 0.005, -c * 0.015], rtol=1e-5)
