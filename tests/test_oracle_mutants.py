"""The oracle's pins must catch plausible mistakes.

Each mutant below is one small textual change to a temporary copy of the
oracle's C source (a swapped beta, a dropped term, a flipped sign, an
off-by-one index...).  The copy is compiled on the CPU and the whole pin
suite (test_oracle_pins.py) is run against it in a subprocess; every mutant
must make at least one pin fail.  The committed oracle is never modified.
"""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero1_oracle.c")

MUTANTS = {
    "beta1_to_beta2_in_m": ("float mj = b1 * m[j] + omb1 * g;", "float mj = b2 * m[j] + omb1 * g;"),
    "beta2_to_beta1_in_v": ("float vj = b2 * v[j] + omb2 * gg;", "float vj = b1 * v[j] + omb2 * gg;"),
    "g_not_squared_in_v": ("float vj = b2 * v[j] + omb2 * gg;", "float vj = b2 * v[j] + omb2 * g;"),
    "eps_inside_sqrt": ("float d = sqrtf(vj) / sqrtbc2 + eps;", "float d = sqrtf(vj + eps) / sqrtbc2;"),
    "no_bias_correction_2": ("float d = sqrtf(vj) / sqrtbc2 + eps;", "float d = sqrtf(vj) + eps;"),
    "no_bias_correction_1": ("const float stepsize = (float)(hp->lr / bc1);",
                             "const float stepsize = (float)(hp->lr);"),
    "bias_corrections_swapped": ("double bc1 = 1.0 - pow(hp->beta1, (double)t);",
                                 "double bc1 = 1.0 - pow(hp->beta2, (double)t);"),
    "update_sign_flipped": ("pj = pj - stepsize * upd;", "pj = pj + stepsize * upd;"),
    "stale_m_in_update": ("float upd = mj / d;", "float upd = m[j] / d;"),
    "decay_dropped": ("float pj = p[j] * dfac;", "float pj = p[j];"),
    "decay_set_inverted": ("const float dfac = no_decay[i] ? 1.0f : dfac_decay;",
                           "const float dfac = no_decay[i] ? dfac_decay : 1.0f;"),
    "decay_not_scaled_by_lr": ("(float)(1.0 - hp->lr * hp->weight_decay)", "(float)(1.0 - hp->weight_decay)"),
    "clip_dropped": ("float g = grad[j] * coef;", "float g = grad[j];"),
    "clip_no_eps_guard_squared": ("double q = clip / (norm + 1e-6);", "double q = clip / (norm * norm + 1e-6);"),
    "clip_when_below_threshold": ("if (q < 1.0)", "if (q > 0.0)"),
    "nonfinite_not_detected": ("if (!isfinite(norm))\n        return 0;", "if (norm < 0)\n        return 0;"),
    "shard_remainder_off_by_one": ("*count = q + ((r < rem) ? 1 : 0);", "*count = q + ((r <= rem) ? 1 : 0);"),
    "shard_start_ignores_remainder": ("*start = (int64_t)r * q + extra_before;", "*start = (int64_t)r * q;"),
    "sumsq_not_squared": ("double sq = x * x;", "double sq = fabs(x);"),
    "sumsq_compensation_sign": ("comp += (s - t) + sq;", "comp -= (s - t) + sq;"),
    "accumulate_subtracts": ("grad[j] = overwrite ? g : grad[j] + g;", "grad[j] = overwrite ? g : grad[j] - g;"),
    "accumulate_overwrite_adds_zero": ("grad[j] = overwrite ? g : grad[j] + g;",
                                       "grad[j] = overwrite ? 0.0f + g : grad[j] + g;"),
    "rne_rounds_half_up": ("u += 0x7fffu + kept_lsb;", "u += 0x8000u;"),
    "rne_truncates": ("u += 0x7fffu + kept_lsb;", "u += 0u;"),
    "nan_not_quieted": ("return (uint16_t)((u >> 16) | 0x0040u);", "return (uint16_t)(u >> 16);"),
    "optimizer_bytes_not_sharded": ("out[2] = 12 * local_numel;", "out[2] = 12 * total_numel;"),
    "weights_bytes_fp32": ("out[0] = 2 * total_numel;", "out[0] = 4 * total_numel;"),
    "divide_is_multiply": ("grad[j] = grad[j] / divisor;", "grad[j] = grad[j] * divisor;"),
    "divide_by_reciprocal": ("grad[j] = grad[j] / divisor;", "grad[j] = grad[j] * (1.0f / divisor);"),
    "scaled_lr_ignored": ("const double lr_i = hp->lr * lr_scale[i];", "const double lr_i = hp->lr;"),
    "scaled_wd_ignored": ("const double wd_i = hp->weight_decay * wd_scale[i];",
                          "const double wd_i = hp->weight_decay;"),
    "scaled_decay_uses_base_lr": ("const float dfac = (float)(1.0 - lr_i * wd_i);",
                                  "const float dfac = (float)(1.0 - hp->lr * wd_i);"),
}


def _run_mutant(name, old, new, tmpdir):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, "mutation anchor not found for %s" % name
    mutated = src.replace(old, new, 1)
    c_path = os.path.join(tmpdir, name + ".c")
    so_path = os.path.join(tmpdir, name + ".so")
    with open(c_path, "w", encoding="utf-8") as f:
        f.write(mutated)
    sys.path.insert(0, ROOT)
    from oracle.build import CFLAGS
    subprocess.run(["gcc", *CFLAGS, c_path, "-o", so_path, "-lm"], check=True)
    env = dict(os.environ, ZERO1_ORACLE_LIB=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_mutant_is_caught_by_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            futs = [ex.submit(_run_mutant, n, o, w, tmp) for n, (o, w) in MUTANTS.items()]
            results = [f.result() for f in futs]
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, "mutants not caught by any pin: %s" % [n for n, _ in survivors]
    # a crash of the test run is not a catch; a failing assertion is
    for n, rc, out in results:
        assert rc == 1, (n, rc, out)
