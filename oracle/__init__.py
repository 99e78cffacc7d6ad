"""Scalar CPU oracle for the ZeRO-1 local-shard optimizer step.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product path (the CUDA
library and its Python binding) never imports it.

Thin ctypes wrapper over ``zero1_oracle.c``; all arithmetic lives in the C
file, which cites the passage each function follows.  Arrays are numpy,
in the local shard list's plan order, without padding.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)


class _HP(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in ("lr", "beta1", "beta2", "eps", "weight_decay")]


def _load():
    global _lib
    if _lib is None:
        # ZERO1_ORACLE_LIB lets the mutation test load a deliberately broken copy of the oracle
        path = os.environ.get("ZERO1_ORACLE_LIB") or build_oracle()
        lib = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        lib.oracle_shard_range.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i64p, _i64p]
        lib.oracle_plan.argtypes = [vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp]
        lib.oracle_plan.restype = ctypes.c_int64
        lib.oracle_zero1_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, vp]
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne_array.argtypes = [vp, vp, ctypes.c_int64]
        lib.oracle_accumulate.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int32]
        lib.oracle_divide.argtypes = [vp, ctypes.c_int64, ctypes.c_float]
        lib.oracle_sumsq.argtypes = [vp, ctypes.c_int64]
        lib.oracle_sumsq.restype = ctypes.c_double
        lib.oracle_clip_coef.argtypes = [ctypes.c_double, ctypes.c_double,
                                         ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)]
        lib.oracle_clip_coef.restype = ctypes.c_int32
        lib.oracle_adamw.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32,
                                     ctypes.POINTER(_HP), ctypes.c_int64, ctypes.c_float]
        lib.oracle_adamw_scaled.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int32,
                                            ctypes.POINTER(_HP), ctypes.c_int64, ctypes.c_float]
        _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _check(a, dtype, name):
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError("%s must be a C-contiguous numpy %s array" % (name, np.dtype(dtype).name))


def shard_range(n, dp_size, dp_rank):
    s, c = ctypes.c_int64(), ctypes.c_int64()
    _load().oracle_shard_range(int(n), int(dp_size), int(dp_rank), ctypes.byref(s), ctypes.byref(c))
    return s.value, c.value


def plan(numels, dp_size, dp_rank):
    """Per-tensor (shard_start, shard_count) arrays and the local element count."""
    numels = np.ascontiguousarray(numels, dtype=np.int64)
    start = np.zeros(len(numels), np.int64)
    count = np.zeros(len(numels), np.int64)
    local = _load().oracle_plan(_ptr(numels), len(numels), int(dp_size), int(dp_rank),
                                _ptr(start), _ptr(count))
    return start, count, local


def zero1_bytes(total_numel, local_numel, grad_bytes=2):
    out = np.zeros(4, np.int64)
    _load().oracle_zero1_bytes(int(total_numel), int(local_numel), int(grad_bytes), _ptr(out))
    return {"weights": int(out[0]), "grads": int(out[1]), "optimizer": int(out[2]), "total": int(out[3])}


def bf16_to_f32(b):
    return _load().oracle_bf16_to_f32(int(b))


def bf16_rne(x):
    """binary32 -> bf16 bits (uint16), round to nearest even; scalar or array."""
    if np.isscalar(x):
        return _load().oracle_bf16_rne(float(np.float32(x)))
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_bf16_rne_array(_ptr(x), _ptr(out), x.size)
    return out


def accumulate(grad, micro_bf16, overwrite):
    """grad (float32, in place) = [grad +] float(micro) for one micro-batch."""
    _check(grad, np.float32, "grad")
    _check(micro_bf16, np.uint16, "micro_bf16")
    if grad.size != micro_bf16.size:
        raise ValueError("size mismatch")
    _load().oracle_accumulate(_ptr(grad), _ptr(micro_bf16), grad.size, 1 if overwrite else 0)


def accumulate_all(grad, micros):
    """Accumulate every micro-batch in order, the first one overwriting."""
    for k, mb in enumerate(micros):
        accumulate(grad, mb, overwrite=(k == 0))


def divide(grad, divisor):
    """grad (float32, in place) /= divisor (rounded to fp32), one IEEE division per element."""
    _check(grad, np.float32, "grad")
    _load().oracle_divide(_ptr(grad), grad.size, float(np.float32(divisor)))


def sumsq(grad):
    _check(grad, np.float32, "grad")
    return _load().oracle_sumsq(_ptr(grad), grad.size)


def clip_coef(sumsq_total, clip):
    """(finite, norm, coef): norm = sqrt(sumsq_total), coef the fp32 clip factor."""
    norm, coef = ctypes.c_double(), ctypes.c_float()
    ok = _load().oracle_clip_coef(float(sumsq_total), float(clip), ctypes.byref(norm), ctypes.byref(coef))
    return bool(ok), norm.value, np.float32(coef.value)


def adamw(p, m, v, grad, counts, no_decay, hp, t, coef, w=None):
    """One AdamW step in place on p/m/v (float32); writes bf16 bits into w if given.

    hp: dict with lr, beta1, beta2, eps, weight_decay.  counts/no_decay give the
    per-tensor shard sizes and weight-decay exclusion in plan order.
    """
    for a, nme in ((p, "p"), (m, "m"), (v, "v"), (grad, "grad")):
        _check(a, np.float32, nme)
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    no_decay = np.ascontiguousarray(no_decay, dtype=np.uint8)
    n = int(counts.sum())
    if not (p.size == m.size == v.size == grad.size == n) or len(no_decay) != len(counts):
        raise ValueError("size mismatch")
    if w is not None:
        _check(w, np.uint16, "w")
        if w.size != n:
            raise ValueError("size mismatch")
    if t < 1:
        raise ValueError("t starts at 1")
    h = _HP(*(float(hp[k]) for k in ("lr", "beta1", "beta2", "eps", "weight_decay")))
    _load().oracle_adamw(_ptr(p), _ptr(m), _ptr(v), _ptr(grad), _ptr(w), _ptr(counts), _ptr(no_decay),
                         len(counts), ctypes.byref(h), int(t), float(coef))


def adamw_scaled(p, m, v, grad, counts, lr_scale, wd_scale, hp, t, coef, w=None):
    """AdamW with a per-tensor lr multiplier and weight-decay multiplier (in place)."""
    for a, nme in ((p, "p"), (m, "m"), (v, "v"), (grad, "grad")):
        _check(a, np.float32, nme)
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    lr_scale = np.ascontiguousarray(lr_scale, dtype=np.float64)
    wd_scale = np.ascontiguousarray(wd_scale, dtype=np.float64)
    n = int(counts.sum())
    if not (p.size == m.size == v.size == grad.size == n) or not (len(lr_scale) == len(wd_scale) == len(counts)):
        raise ValueError("size mismatch")
    if w is not None:
        _check(w, np.uint16, "w")
        if w.size != n:
            raise ValueError("size mismatch")
    if t < 1:
        raise ValueError("t starts at 1")
    h = _HP(*(float(hp[k]) for k in ("lr", "beta1", "beta2", "eps", "weight_decay")))
    _load().oracle_adamw_scaled(_ptr(p), _ptr(m), _ptr(v), _ptr(grad), _ptr(w), _ptr(counts), _ptr(lr_scale),
                                _ptr(wd_scale), len(counts), ctypes.byref(h), int(t), float(coef))


def full_step(p, m, v, micros, counts, no_decay, hp, t, clip, extra_sumsq=0.0, w=None, grad=None):
    """The whole local-shard step: accumulate, norm + clip, AdamW, bf16 copy.

    Returns a dict with the accumulated grad, local sumsq, norm, coef and
    whether the update ran (a non-finite norm skips it).
    """
    n = p.size
    if grad is None:
        grad = np.zeros(n, np.float32)
    accumulate_all(grad, micros)
    local = sumsq(grad)
    finite, norm, coef = clip_coef(local + extra_sumsq, clip)
    if finite:
        adamw(p, m, v, grad, counts, no_decay, hp, t, coef, w=w)
    return {"grad": grad, "sumsq": local, "norm": norm, "coef": coef, "applied": finite}
