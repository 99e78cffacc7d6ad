"""ctypes binding of libzero1.so: argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module checks
tensors (device, dtype, size, contiguity, 16-byte alignment), turns them into
raw pointers and forwards the current CUDA stream.  It has no fallback: when
the library is missing or a call fails it raises.
"""
import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzero1.so")

ZERO1_OK = 0
ZERO1_EINVAL = -1
ZERO1_EALIGN = -2
ZERO1_ECUDA = -3
ZERO1_ENONFINITE = -4
ZERO1_ENOMEM = -5
ZERO1_ETOOBIG = -6
STATIC_NORM_MAX_NUMEL = 262144 * 16384
ARENA_ALIGN = 8
MAX_GROUPS = 8
MAX_MICRO = 16
NORM_OUT_BYTES = 24

_lib = None


class Zero1Error(RuntimeError):
    def __init__(self, code, where):
        lib = load_library()
        msg = "%s failed: %s" % (where, lib.zero1_strerror(code).decode())
        if code == ZERO1_ECUDA:
            msg += " (%s)" % lib.zero1_last_cuda_error().decode()
        super().__init__(msg)
        self.code = code


class _Hparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in ("lr", "beta1", "beta2", "eps", "weight_decay", "clip_grad")]


class _StepScalars(ctypes.Structure):
    _fields_ = [("stepsize", ctypes.c_float * 8), ("dfac", ctypes.c_float * 8)] + \
               [(n, ctypes.c_float) for n in ("b1", "b2", "omb1", "omb2", "eps", "sqrtbc2")] + \
               [("clip", ctypes.c_double)]


STEP_SCALARS_BYTES = 96


class _NormOut(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("norm", ctypes.c_double), ("status", ctypes.c_int32),
                ("n_partials", ctypes.c_int32)]


def load_library(path=None):
    """Load libzero1.so (built in-tree by ``build.build_library``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("libzero1.so is not built (%s); run __graft_entry__.build() first" % path)
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    i64p = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "zero1_plan_create": (ctypes.c_int, [vp, vp, i32, i32, i32, ctypes.POINTER(vp)]),
        "zero1_plan_create_grouped": (ctypes.c_int, [vp, vp, i32, vp, vp, i32, i32, ctypes.POINTER(vp)]),
        "zero1_plan_group_scales": (ctypes.c_int, [vp, i32, ctypes.POINTER(ctypes.c_double),
                                                   ctypes.POINTER(ctypes.c_double)]),
        "zero1_plan_destroy": (None, [vp]),
        "zero1_plan_num_tensors": (i32, [vp]),
        "zero1_plan_total_numel": (i64, [vp]),
        "zero1_plan_local_numel": (i64, [vp]),
        "zero1_plan_arena_numel": (i64, [vp]),
        "zero1_plan_tensor": (ctypes.c_int, [vp, i32, i64p, i64p, i64p]),
        "zero1_plan_group_range": (ctypes.c_int, [vp, i32, i64p, i64p]),
        "zero1_plan_bytes": (ctypes.c_int, [vp, i32, i64p]),
        "zero1_workspace_bytes": (ctypes.c_size_t, [vp]),
        "zero1_accumulate": (ctypes.c_int, [vp, vp, ctypes.POINTER(vp), i32, i32, vp]),
        "zero1_accumulate_norm": (ctypes.c_int, [vp, vp, ctypes.POINTER(vp), i32, i32, ctypes.c_double,
                                                 ctypes.c_double, vp, ctypes.c_size_t, vp, vp]),
        "zero1_grad_norm": (ctypes.c_int, [vp, vp, ctypes.c_double, vp, ctypes.c_size_t, vp, vp]),
        "zero1_grad_norm_static": (ctypes.c_int, [vp, vp, ctypes.c_double, vp, vp]),
        "zero1_step": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, ctypes.POINTER(_Hparams), i64, vp, vp]),
        "zero1_micro_norm": (ctypes.c_int, [vp, vp, ctypes.c_double, ctypes.c_double, vp, ctypes.c_size_t, vp, vp]),
        "zero1_step_accumulate": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, ctypes.c_double, vp,
                                                 ctypes.POINTER(_Hparams), i64, vp, vp]),
        "zero1_local_step": (ctypes.c_int, [vp, vp, ctypes.POINTER(vp), i32, ctypes.c_double, ctypes.c_double, vp,
                                            ctypes.c_size_t, vp, vp, vp, vp, vp, ctypes.POINTER(_Hparams), i64,
                                            vp]),
        "zero1_read_norm": (ctypes.c_int, [vp, vp, ctypes.POINTER(_NormOut)]),
        "zero1_step_scalars_fill": (ctypes.c_int, [vp, ctypes.POINTER(_Hparams), i64, ctypes.POINTER(_StepScalars)]),
        "zero1_step_dev": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "zero1_layout_table_bytes": (ctypes.c_size_t, [vp]),
        "zero1_layout_table_upload": (ctypes.c_int, [vp, vp, ctypes.c_size_t, vp]),
        "zero1_shard_gather": (ctypes.c_int, [vp, vp, vp, vp, i32, vp]),
        "zero1_shard_scatter": (ctypes.c_int, [vp, vp, vp, vp, i32, vp]),
        "zero1_list_table_bytes": (ctypes.c_size_t, [vp]),
        "zero1_list_table_upload": (ctypes.c_int, [vp, vp, ctypes.c_size_t, vp]),
        "zero1_list_workspace_bytes": (ctypes.c_size_t, [vp]),
        "zero1_list_ptrs_upload": (ctypes.c_int, [vp, ctypes.POINTER(vp), i32, i32, vp, ctypes.c_size_t, vp]),
        "zero1_list_accumulate": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, vp]),
        "zero1_list_accumulate_norm": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, ctypes.c_double, ctypes.c_double,
                                                      vp, ctypes.c_size_t, vp, vp]),
        "zero1_list_grad_norm": (ctypes.c_int, [vp, vp, vp, ctypes.c_double, vp, ctypes.c_size_t, vp, vp]),
        "zero1_list_micro_norm": (ctypes.c_int, [vp, vp, vp, ctypes.c_double, ctypes.c_double, vp, ctypes.c_size_t,
                                                 vp, vp]),
        "zero1_list_step_accumulate": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, ctypes.c_double, vp,
                                                      ctypes.POINTER(_Hparams), i64, vp, vp]),
        "zero1_list_step": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(_Hparams), i64, vp, vp]),
        "zero1_list_step_dev": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "zero1_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "zero1_last_cuda_error": (ctypes.c_char_p, []),
        "zero1_launch_count": (ctypes.c_uint64, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def launch_count():
    """zero1_launch_count: kernel launches the library has issued since it was loaded."""
    return int(load_library().zero1_launch_count())


def _check(code, where):
    if code != ZERO1_OK:
        raise Zero1Error(code, where)


# torch's own accessors of the current device and of its current stream's handle: what
# torch.cuda.current_device() and current_stream().cuda_stream return, without building a
# Stream object on every call
_current_device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
_current_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, device):
    """The stream a call launches on (a cudaStream_t as an int).  The library launches on the
    current CUDA device, so the tensors' device must be the current one (a kernel given another
    device's memory or stream would fail); say so here rather than through a CUDA error."""
    if not isinstance(device, torch.device):
        device = torch.device(device)
    index = device.index
    current = _current_device()
    if index is not None and device.type == "cuda" and index != current:
        raise ValueError("the buffers are on %s but the current CUDA device is cuda:%d; call inside "
                         "torch.cuda.device(%d)" % (device, current, index))
    if stream is None:
        if _current_raw_stream is not None:
            return _current_raw_stream(current)  # the current device's, checked above
        stream = torch.cuda.current_stream()
    elif index is not None and stream.device_index != index:
        raise ValueError("stream is on %s, the buffers on %s" % (stream.device, device))
    return stream.cuda_stream


def _ptr(t, dtype, numel, name, device=None, host_ok=False):
    """Raw pointer of a checked tensor.  With host_ok, a pinned CPU tensor is accepted too:
    kernels read it directly over the CPU-GPU link."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        if not (host_ok and t.device.type == "cpu" and t.is_pinned()):
            raise ValueError("%s must be on a CUDA device%s (got %s)" % (
                name, " or pinned host memory" if host_ok else "", t.device))
    elif device is not None and device.index is not None and t.get_device() != device.index:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if t.dtype != dtype:
        raise TypeError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if numel is not None and t.numel() != numel:
        raise ValueError("%s has %d elements, the plan's arena has %d" % (name, t.numel(), numel))
    ptr = t.data_ptr()
    if ptr % 16:
        raise ValueError("%s must start on a 16-byte boundary" % name)
    return ptr  # ctypes passes an int to a c_void_p parameter as the address


@dataclass
class Hparams:
    """AdamW settings of the ZeRO-1 optimizer (adam_w, betas 0.9/0.95, eps 1e-8,
    weight_decay 0.1, clip_grad 1.0 in nanotron's config)."""
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    clip_grad: float = 1.0

    def _c(self):
        """A fresh ctypes zero1_hparams for one call (never shared between calls)."""
        return _Hparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, self.clip_grad)


@dataclass
class ShardLayout:
    """Per-tensor shard placement of a plan (numpy arrays, model order)."""
    shard_start: np.ndarray
    counts: np.ndarray
    offsets: np.ndarray
    no_decay: np.ndarray   # 1 where the tensor's group has a weight-decay scale of 0
    arena_numel: int
    groups: np.ndarray = None


class Plan:
    """zero1_plan: every parameter tensor cut by numel into dp_size contiguous
    shards; this rank's shards laid out in one padded arena per quantity.

    Either ``no_decay`` flags (group 0 decays, group 1 does not) or ``groups``
    (0..MAX_GROUPS-1) with optional per-group ``lr_scale`` / ``wd_scale``
    (length MAX_GROUPS) multipliers of the step's lr and weight decay."""

    def __init__(self, numels, no_decay=None, dp_size=1, dp_rank=0, groups=None, lr_scale=None, wd_scale=None):
        lib = load_library()
        numels = np.ascontiguousarray(numels, dtype=np.int64)
        if (no_decay is None) == (groups is None):
            raise ValueError("give exactly one of no_decay and groups")
        grp = np.ascontiguousarray(no_decay if groups is None else groups, dtype=np.uint8)
        if numels.shape != grp.shape or numels.ndim != 1:
            raise ValueError("numels and no_decay/groups must be 1-D and the same length")
        h = ctypes.c_void_p()
        if groups is None:
            if lr_scale is not None or wd_scale is not None:
                raise ValueError("per-group scales need groups=")
            _check(lib.zero1_plan_create(numels.ctypes.data, grp.ctypes.data, len(numels), int(dp_size),
                                         int(dp_rank), ctypes.byref(h)), "zero1_plan_create")
        else:
            scales = []
            for sc in (lr_scale, wd_scale):
                if sc is None:
                    scales.append(None)
                else:
                    a = np.ascontiguousarray(sc, dtype=np.float64)
                    if a.shape != (MAX_GROUPS,):
                        raise ValueError("per-group scales need %d entries" % MAX_GROUPS)
                    scales.append(a)
            self._scales = scales
            _check(lib.zero1_plan_create_grouped(numels.ctypes.data, grp.ctypes.data, len(numels),
                                                 None if scales[0] is None else scales[0].ctypes.data,
                                                 None if scales[1] is None else scales[1].ctypes.data,
                                                 int(dp_size), int(dp_rank), ctypes.byref(h)),
                   "zero1_plan_create_grouped")
        self._h = h
        self._lib = lib
        self.dp_size, self.dp_rank = int(dp_size), int(dp_rank)
        # a plan never changes after creation: its sizes are read once, not on every call
        self._sizes = (lib.zero1_plan_num_tensors(h), lib.zero1_plan_total_numel(h), lib.zero1_plan_local_numel(h),
                       lib.zero1_plan_arena_numel(h), lib.zero1_workspace_bytes(h), lib.zero1_list_workspace_bytes(h))
        self._groups = grp.copy()
        self.numels = numels.copy()
        self._layout = None
        self._grouped = groups is not None

    def for_rank(self, dp_rank):
        """The same parameter list, groups and scales, sharded for another data-parallel rank."""
        if self._grouped:
            lr, wd = self._scales
            return Plan(self.numels, groups=self._groups, dp_size=self.dp_size, dp_rank=dp_rank, lr_scale=lr,
                        wd_scale=wd)
        return Plan(self.numels, self._groups, self.dp_size, dp_rank)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.zero1_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    @property
    def num_tensors(self):
        return self._sizes[0]

    @property
    def total_numel(self):
        return self._sizes[1]

    @property
    def local_numel(self):
        return self._sizes[2]

    @property
    def arena_numel(self):
        return self._sizes[3]

    @property
    def workspace_bytes(self):
        return self._sizes[4]

    def tensor(self, i):
        s, c, o = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.zero1_plan_tensor(self._h, int(i), ctypes.byref(s), ctypes.byref(c), ctypes.byref(o)),
               "zero1_plan_tensor")
        return s.value, c.value, o.value

    def group_range(self, g):
        b, e = ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.zero1_plan_group_range(self._h, int(g), ctypes.byref(b), ctypes.byref(e)),
               "zero1_plan_group_range")
        return b.value, e.value

    def group_scales(self, g):
        lr, wd = ctypes.c_double(), ctypes.c_double()
        _check(self._lib.zero1_plan_group_scales(self._h, int(g), ctypes.byref(lr), ctypes.byref(wd)),
               "zero1_plan_group_scales")
        return lr.value, wd.value

    def bytes(self, grad_bytes=2):
        out = (ctypes.c_int64 * 4)()
        _check(self._lib.zero1_plan_bytes(self._h, int(grad_bytes), out), "zero1_plan_bytes")
        return {"weights": out[0], "grads": out[1], "optimizer": out[2], "total": out[3]}

    def layout(self) -> ShardLayout:
        if self._layout is None:
            n = self.num_tensors
            st, ct, of = np.zeros(n, np.int64), np.zeros(n, np.int64), np.zeros(n, np.int64)
            for i in range(n):
                st[i], ct[i], of[i] = self.tensor(i)
            wd_zero = np.array([self.group_scales(g)[1] == 0.0 for g in range(MAX_GROUPS)])
            self._layout = ShardLayout(st, ct, of, wd_zero[self._groups].astype(np.uint8), self.arena_numel,
                                       self._groups.copy())
        return self._layout

    def layout_table(self, device="cuda", stream=None):
        """Device copy of this plan's model-layout <-> arena copy table (made once per device)."""
        device = torch.device(device)
        if device.index is None:
            device = torch.device("cuda", torch.cuda.current_device())
        cache = self.__dict__.setdefault("_tables", {})
        if device not in cache:
            nbytes = self._lib.zero1_layout_table_bytes(self._h)
            t = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
            _check(self._lib.zero1_layout_table_upload(self._h, ctypes.c_void_p(t.data_ptr()), t.numel(),
                                                       _stream_ptr(stream, device)), "zero1_layout_table_upload")
            cache[device] = t
        return cache[device]

    @property
    def list_workspace_bytes(self):
        return self._sizes[5]

    def list_table(self, device="cuda", stream=None):
        """Device copy of this plan's tensor-list run table (made once per device)."""
        device = torch.device(device)
        if device.index is None:
            device = torch.device("cuda", torch.cuda.current_device())
        cache = self.__dict__.setdefault("_list_tables", {})
        if device not in cache:
            nbytes = self._lib.zero1_list_table_bytes(self._h)
            t = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
            _check(self._lib.zero1_list_table_upload(self._h, ctypes.c_void_p(t.data_ptr()), t.numel(),
                                                     _stream_ptr(stream, device)), "zero1_list_table_upload")
            cache[device] = t
        return cache[device]

    def new_list_workspace(self, device="cuda"):
        return torch.empty(max(self.list_workspace_bytes, 16), dtype=torch.uint8, device=device)

    def new_shards(self, dtype=torch.float32, device="cuda"):
        """One zero-filled buffer per tensor shard (model order), for the tensor-list calls."""
        return [torch.zeros(int(c), dtype=dtype, device=device) for c in self.layout().counts]

    # -- buffers (the caller owns them; these are conveniences) --
    def new_arena(self, dtype=torch.float32, device="cuda"):
        """A zero-filled arena buffer (zero padding, as the layout contract requires)."""
        return torch.zeros(self.arena_numel, dtype=dtype, device=device)

    def new_workspace(self, device="cuda"):
        return torch.empty(max(self.workspace_bytes, 16), dtype=torch.uint8, device=device)

    def shard_views(self, arena):
        """Per-tensor views of an arena, in model order (empty shards give empty views)."""
        L = self.layout()
        return [arena[int(o):int(o) + int(c)] for o, c in zip(L.offsets, L.counts)]


def _norm_ptr(norm_out, name="norm_out", device=None):
    """Raw pointer of a norm-record buffer: a 16-byte aligned CUDA uint8 tensor of at least
    NORM_OUT_BYTES bytes."""
    p = _ptr(norm_out, torch.uint8, None, name, device)
    if norm_out.numel() < NORM_OUT_BYTES:
        raise ValueError("%s needs %d bytes (got %d)" % (name, NORM_OUT_BYTES, norm_out.numel()))
    return p


def new_norm_out(device="cuda"):
    """Device buffer for a zero1_norm_out (24 bytes, 16-byte aligned)."""
    return torch.zeros(32, dtype=torch.uint8, device=device)


def accumulate(plan, grad, micro, overwrite_first=True, stream=None):
    """zero1_accumulate: grad (fp32 arena) = [grad +] sum of the bf16 micro-batch arenas.

    A micro-batch arena may be a CUDA tensor or a pinned CPU tensor; the kernel reads a
    pinned one directly over the CPU-GPU link (no staging copy)."""
    lib = load_library()
    n = plan.arena_numel
    dev = grad.device
    gp = _ptr(grad, torch.float32, n, "grad")
    micro, arr = _micro_array(plan, micro, dev)
    _check(lib.zero1_accumulate(plan.handle, gp, arr, len(micro), 1 if overwrite_first else 0,
                                _stream_ptr(stream, dev)), "zero1_accumulate")


def _micro_array(plan, micro, dev):
    micro = [micro] if isinstance(micro, torch.Tensor) else list(micro)
    if not 1 <= len(micro) <= MAX_MICRO:
        raise ValueError("1..%d micro-batch gradients per call" % MAX_MICRO)
    return micro, (ctypes.c_void_p * len(micro))(*[_ptr(mb, torch.bfloat16, plan.arena_numel, "micro[%d]" % k, dev,
                                                        host_ok=True) for k, mb in enumerate(micro)])


def accumulate_norm(plan, grad, micro, workspace, norm_out, overwrite_first=True, extra_sumsq=0.0, divisor=1.0,
                    stream=None):
    """zero1_accumulate_norm: accumulate the last micro-batch(es) and take the norm in one pass.
    ``divisor`` (e.g. the data-parallel world size) divides the finished sum first."""
    lib = load_library()
    dev = grad.device
    gp = _ptr(grad, torch.float32, plan.arena_numel, "grad")
    micro, arr = _micro_array(plan, micro, dev)
    wp = _ptr(workspace, torch.uint8, None, "workspace", dev)
    if workspace.numel() < plan.workspace_bytes:
        raise ValueError("workspace has %d bytes, the plan needs %d" % (workspace.numel(), plan.workspace_bytes))
    op = _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_accumulate_norm(plan.handle, gp, arr, len(micro), 1 if overwrite_first else 0,
                                     float(divisor), float(extra_sumsq), wp, workspace.numel(), op,
                                     _stream_ptr(stream, dev)), "zero1_accumulate_norm")


def grad_norm(plan, grad, workspace, norm_out, extra_sumsq=0.0, stream=None):
    """zero1_grad_norm: device {sumsq, norm, status} of the fp32 grad arena (+ extra_sumsq)."""
    lib = load_library()
    dev = norm_out.device
    gp = _ptr(grad, torch.float32, plan.arena_numel, "grad", dev)
    wp = _ptr(workspace, torch.uint8, None, "workspace", dev)
    if workspace.numel() < plan.workspace_bytes:
        raise ValueError("workspace has %d bytes, the plan needs %d" % (workspace.numel(), plan.workspace_bytes))
    op = _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_grad_norm(plan.handle, gp, float(extra_sumsq), wp, workspace.numel(), op,
                               _stream_ptr(stream, dev)), "zero1_grad_norm")


def grad_norm_static(plan, grad, norm_out, extra_sumsq=0.0, stream=None):
    """zero1_grad_norm_static: the same norm record as grad_norm(), with no workspace.

    For callers that cannot allocate or supply device scratch: the partial
    sums go to a fixed 2 MiB array inside the library (arenas up to
    STATIC_NORM_MAX_NUMEL elements).  Calls that overlap on the GPU share that
    array and race; the first call on a device should precede any stream
    capture."""
    lib = load_library()
    if plan.arena_numel > STATIC_NORM_MAX_NUMEL:
        raise ValueError("arena of %d elements exceeds the static norm scratch limit of %d elements"
                         % (plan.arena_numel, STATIC_NORM_MAX_NUMEL))
    dev = norm_out.device
    gp = _ptr(grad, torch.float32, plan.arena_numel, "grad", dev)
    op = _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_grad_norm_static(plan.handle, gp, float(extra_sumsq), op, _stream_ptr(stream, dev)),
           "zero1_grad_norm_static")


def step(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, hparams, step_t, norm_out=None, stream=None):
    """zero1_step: fused clip + AdamW on the fp32 master/m/v arenas and the bf16 copy."""
    lib = load_library()
    n = plan.arena_numel
    dev = master.device
    ptrs = [_ptr(master, torch.float32, n, "master", dev), _ptr(exp_avg, torch.float32, n, "exp_avg", dev),
            _ptr(exp_avg_sq, torch.float32, n, "exp_avg_sq", dev), _ptr(grad, torch.float32, n, "grad", dev)]
    wp = None if weight_bf16 is None else _ptr(weight_bf16, torch.bfloat16, n, "weight_bf16", dev)
    npp = None if norm_out is None else _norm_ptr(norm_out, device=dev)
    hp = hparams._c() if isinstance(hparams, Hparams) else Hparams(**hparams)._c()
    _check(lib.zero1_step(plan.handle, *ptrs, wp, ctypes.byref(hp), int(step_t), npp, _stream_ptr(stream, dev)),
           "zero1_step")


def micro_norm(plan, micro, workspace, norm_out, extra_sumsq=0.0, divisor=1.0, stream=None):
    """zero1_micro_norm: the norm record of one micro-batch's gradient (float(micro) / divisor),
    without writing the gradient: the record accumulate_norm(overwrite_first=True) would write."""
    lib = load_library()
    dev = norm_out.device
    mp = _ptr(micro, torch.bfloat16, plan.arena_numel, "micro", dev, host_ok=True)
    wp = _ptr(workspace, torch.uint8, None, "workspace", dev)
    if workspace.numel() < plan.workspace_bytes:
        raise ValueError("workspace has %d bytes, the plan needs %d" % (workspace.numel(), plan.workspace_bytes))
    op = _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_micro_norm(plan.handle, mp, float(divisor), float(extra_sumsq), wp, workspace.numel(), op,
                                _stream_ptr(stream, dev)), "zero1_micro_norm")


def step_accumulate(plan, master, exp_avg, exp_avg_sq, grad, micro, weight_bf16, hparams, step_t, norm_out=None,
                    divisor=1.0, stream=None):
    """zero1_step_accumulate: the step for one micro-batch's gradient, written to ``grad`` in the
    same pass (the same results as accumulate_norm + step)."""
    lib = load_library()
    n = plan.arena_numel
    dev = master.device
    ptrs = [_ptr(master, torch.float32, n, "master", dev), _ptr(exp_avg, torch.float32, n, "exp_avg", dev),
            _ptr(exp_avg_sq, torch.float32, n, "exp_avg_sq", dev), _ptr(grad, torch.float32, n, "grad", dev),
            _ptr(micro, torch.bfloat16, n, "micro", dev, host_ok=True)]
    wp = None if weight_bf16 is None else _ptr(weight_bf16, torch.bfloat16, n, "weight_bf16", dev)
    npp = None if norm_out is None else _norm_ptr(norm_out, device=dev)
    hp = hparams._c() if isinstance(hparams, Hparams) else Hparams(**hparams)._c()
    _check(lib.zero1_step_accumulate(plan.handle, *ptrs, float(divisor), wp, ctypes.byref(hp), int(step_t), npp,
                                     _stream_ptr(stream, dev)), "zero1_step_accumulate")


def local_step(plan, grad, micro, workspace, norm_out, master, exp_avg, exp_avg_sq, weight_bf16, hparams, step_t,
               extra_sumsq=0.0, divisor=1.0, stream=None):
    """zero1_local_step: the whole local step in one call -- every micro-batch accumulated
    (the first overwriting ``grad``) with the norm in one pass, then clip + AdamW + the bf16
    copy (for one micro-batch, micro_norm then step_accumulate).  The same results as
    accumulate_norm(overwrite_first=True) then step()."""
    lib = load_library()
    n = plan.arena_numel
    dev = master.device
    micro, arr = _micro_array(plan, micro, dev)
    gp = _ptr(grad, torch.float32, n, "grad", dev)
    wp = _ptr(workspace, torch.uint8, None, "workspace", dev)
    if workspace.numel() < plan.workspace_bytes:
        raise ValueError("workspace has %d bytes, the plan needs %d" % (workspace.numel(), plan.workspace_bytes))
    op = _norm_ptr(norm_out, device=dev)
    ptrs = [_ptr(master, torch.float32, n, "master", dev), _ptr(exp_avg, torch.float32, n, "exp_avg", dev),
            _ptr(exp_avg_sq, torch.float32, n, "exp_avg_sq", dev)]
    bp = None if weight_bf16 is None else _ptr(weight_bf16, torch.bfloat16, n, "weight_bf16", dev)
    hp = hparams._c() if isinstance(hparams, Hparams) else Hparams(**hparams)._c()
    _check(lib.zero1_local_step(plan.handle, gp, arr, len(micro), float(divisor), float(extra_sumsq), wp,
                                workspace.numel(), op, *ptrs, bp, ctypes.byref(hp), int(step_t),
                                _stream_ptr(stream, dev)), "zero1_local_step")


def step_scalars(plan, hparams, step_t):
    """zero1_step_scalars_fill: the 96 bytes of fp32 step scalars for (plan, hparams, step_t)."""
    hp = hparams._c() if isinstance(hparams, Hparams) else Hparams(**hparams)._c()
    out = _StepScalars()
    _check(load_library().zero1_step_scalars_fill(plan.handle, ctypes.byref(hp), int(step_t), ctypes.byref(out)),
           "zero1_step_scalars_fill")
    return bytes(out)


def step_dev(plan, master, exp_avg, exp_avg_sq, grad, weight_bf16, d_scalars, norm_out=None, stream=None):
    """zero1_step_dev: the step with its scalars read from device memory (a uint8 tensor of at
    least 96 bytes holding step_scalars()), so the call can be captured in a CUDA graph."""
    lib = load_library()
    n = plan.arena_numel
    dev = master.device
    ptrs = [_ptr(master, torch.float32, n, "master", dev), _ptr(exp_avg, torch.float32, n, "exp_avg", dev),
            _ptr(exp_avg_sq, torch.float32, n, "exp_avg_sq", dev), _ptr(grad, torch.float32, n, "grad", dev)]
    wp = None if weight_bf16 is None else _ptr(weight_bf16, torch.bfloat16, n, "weight_bf16", dev)
    sp = _ptr(d_scalars, torch.uint8, None, "d_scalars", dev)
    if d_scalars.numel() < STEP_SCALARS_BYTES:
        raise ValueError("d_scalars needs %d bytes" % STEP_SCALARS_BYTES)
    npp = None if norm_out is None else _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_step_dev(plan.handle, *ptrs, wp, sp, npp, _stream_ptr(stream, dev)), "zero1_step_dev")


def read_norm(norm_out, stream=None):
    """zero1_read_norm: synchronise the stream and return the norm record as a dict."""
    lib = load_library()
    out = _NormOut()
    _check(lib.zero1_read_norm(_norm_ptr(norm_out),
                               _stream_ptr(stream, norm_out.device), ctypes.byref(out)), "zero1_read_norm")
    return {"sumsq": out.sumsq, "norm": out.norm, "status": out.status, "n_partials": out.n_partials}


_ELEM_BYTES = {torch.float32: 4, torch.int32: 4, torch.bfloat16: 2, torch.float16: 2, torch.int16: 2}


def _layout_args(plan, full, arena, name_full):
    if full.dtype != arena.dtype or full.dtype not in _ELEM_BYTES:
        raise TypeError("full and arena must share a 2- or 4-byte dtype")
    eb = _ELEM_BYTES[full.dtype]
    dev = arena.device
    ap = _ptr(arena, arena.dtype, plan.arena_numel, "arena", dev)
    if full.device != dev or not full.is_contiguous() or full.numel() != plan.total_numel:
        raise ValueError("%s must be a contiguous %d-element tensor on %s" % (name_full, plan.total_numel, dev))
    return eb, dev, ap, ctypes.c_void_p(full.data_ptr())


def shard_gather(plan, full, arena, stream=None):
    """zero1_shard_gather: this rank's shard of a model-layout tensor into its arena."""
    eb, dev, ap, fp = _layout_args(plan, full, arena, "full")
    tp = ctypes.c_void_p(plan.layout_table(dev).data_ptr())
    _check(load_library().zero1_shard_gather(plan.handle, tp, fp, ap, eb, _stream_ptr(stream, dev)),
           "zero1_shard_gather")


def shard_scatter(plan, arena, full, stream=None):
    """zero1_shard_scatter: an arena back into this rank's positions of a model-layout tensor."""
    eb, dev, ap, fp = _layout_args(plan, full, arena, "full")
    tp = ctypes.c_void_p(plan.layout_table(dev).data_ptr())
    _check(load_library().zero1_shard_scatter(plan.handle, tp, ap, fp, eb, _stream_ptr(stream, dev)),
           "zero1_shard_scatter")


def exchange_chunk_numel(plans):
    """Per-rank chunk length of a reduce-scatter / all-gather buffer: the largest arena."""
    return max(p.arena_numel for p in plans)


def pack_reduce_scatter(plans, full_grad, send, stream=None):
    """Lay a model-layout gradient out for a reduce-scatter: chunk r of ``send``
    (``len(plans)`` x ``exchange_chunk_numel(plans)`` elements) receives rank r's
    shard in rank r's arena layout, zero-padded."""
    chunk = exchange_chunk_numel(plans)
    if send.numel() != chunk * len(plans):
        raise ValueError("send must hold %d x %d elements" % (len(plans), chunk))
    if stream is None:
        send.zero_()
    else:
        with torch.cuda.stream(stream):  # the padding's fill in order before the gathers on that stream
            send.zero_()
    flat = send.view(-1)
    for r, pl in enumerate(plans):
        shard_gather(pl, full_grad, flat[r * chunk:r * chunk + pl.arena_numel], stream=stream)


def unpack_all_gather(plans, recv, full, stream=None):
    """Write every rank's arena (chunk r of an all-gather receive buffer) back into the
    model-layout tensor ``full``."""
    chunk = exchange_chunk_numel(plans)
    if recv.numel() != chunk * len(plans):
        raise ValueError("recv must hold %d x %d elements" % (len(plans), chunk))
    flat = recv.view(-1)
    for r, pl in enumerate(plans):
        shard_scatter(pl, flat[r * chunk:r * chunk + pl.arena_numel], full, stream=stream)


def allreduce_sumsq_(norm_out, group=None, stream=None):
    """Sum the ``sumsq`` field of a norm record across the ranks of ``group``, in place.

    This is the step's one exchange: each rank's zero1_grad_norm gives its
    local sum of squares, and after the all-reduce every rank's zero1_step
    clips with the same global norm (and skips if any rank saw inf/NaN).
    Works for a CUDA record with NCCL (or gloo) and a CPU record with gloo.
    A CUDA collective is ordered after the work of torch's current stream, so
    with ``stream`` (the torch.cuda.Stream the norm kernels ran on, and the step
    will run on) it is issued with that stream current.
    """
    import torch.distributed as dist

    rec = norm_out[:8].view(torch.float64)
    if stream is None or not norm_out.is_cuda:
        dist.all_reduce(rec, op=dist.ReduceOp.SUM, group=group)
        return
    with torch.cuda.stream(stream):
        dist.all_reduce(rec, op=dist.ReduceOp.SUM, group=group)


def decode_norm(norm_out_bytes):
    """Decode a zero1_norm_out already copied to the host (a uint8 tensor / bytes)."""
    b = bytes(norm_out_bytes.cpu().numpy().tobytes()) if isinstance(norm_out_bytes, torch.Tensor) else norm_out_bytes
    o = _NormOut.from_buffer_copy(b[:NORM_OUT_BYTES])
    return {"sumsq": o.sumsq, "norm": o.norm, "status": o.status, "n_partials": o.n_partials}


# ---- tensor lists: one buffer per tensor shard ----------------------------------------------

class PointerLists:
    """Device pointer lists for the tensor-list calls: ``n_lists`` lists of the plan's
    per-tensor shard buffers of one dtype (model order), checked and uploaded by
    zero1_list_ptrs_upload.  With ``keep`` (the default) it holds references to the
    tensors so their memory stays valid while the lists exist.  ``lists`` is one list
    of tensors or a list of them.  The upload is ordered on ``stream`` (a
    torch.cuda.Stream; the current stream by default): the calls that read the lists
    run on that stream, or on one that waits for it."""

    def __init__(self, plan, lists, dtype, device=None, stream=None, keep=True):
        lib = load_library()
        if device is not None:
            device = torch.device(device)
            if device.type == "cuda" and device.index is None:
                device = torch.device("cuda", torch.cuda.current_device())
        if len(lists) and (isinstance(lists[0], torch.Tensor) or lists[0] is None):
            lists = [lists]
        lists = [list(x) for x in lists]
        n = plan.num_tensors
        if not 1 <= len(lists) <= MAX_MICRO:
            raise ValueError("1..%d pointer lists per upload" % MAX_MICRO)
        counts = plan.layout().counts
        ptrs = []
        for k, lst in enumerate(lists):
            if len(lst) != n:
                raise ValueError("list %d has %d tensors, the plan has %d" % (k, len(lst), n))
            for i, t in enumerate(lst):
                if int(counts[i]) == 0 and t is None:
                    ptrs.append(None)
                    continue
                if not isinstance(t, torch.Tensor):
                    raise TypeError("entry %d of list %d must be a torch.Tensor" % (i, k))
                if t.device.type != "cuda":
                    raise ValueError("entry %d of list %d must be on a CUDA device (got %s)" % (i, k, t.device))
                if device is None:
                    device = t.device
                elif t.device != device:
                    raise ValueError("entry %d of list %d is on %s, expected %s" % (i, k, t.device, device))
                if t.dtype != dtype:
                    raise TypeError("entry %d of list %d must be %s (got %s)" % (i, k, dtype, t.dtype))
                if not t.is_contiguous() or t.numel() != int(counts[i]):
                    raise ValueError("entry %d of list %d must be contiguous with %d elements (got %d)"
                                     % (i, k, int(counts[i]), t.numel()))
                ptrs.append(t.data_ptr() if t.numel() else None)
        if device is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.device = torch.device(device)
        self.n_lists = len(lists)
        count = self.n_lists * n
        # Allocated from the pool of the stream that uploads the lists (and whose kernels read them),
        # with no fill: a fill on another stream could land after the upload, and the allocator
        # orders a later reuse of the block after that stream's work.
        up = stream if stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.stream(up):
            self.dev = torch.empty(max(count, 2), dtype=torch.int64, device=self.device)
        host = (ctypes.c_void_p * max(count, 1))(*ptrs)
        _check(lib.zero1_list_ptrs_upload(plan.handle, host, self.n_lists, 2 if dtype == torch.bfloat16 else 4,
                                          ctypes.c_void_p(self.dev.data_ptr()), self.dev.numel() * 8,
                                          _stream_ptr(up, self.device)), "zero1_list_ptrs_upload")
        self.tensors = lists if keep else None
        self.dtype = dtype
        self.counts = counts  # the plan's shard sizes: the calls check the lists against their plan

    @property
    def ptr(self):
        return ctypes.c_void_p(self.dev.data_ptr())


def _list_args(plan, table, stream, device):
    # The library cannot see inside device memory: a run table of another plan would
    # index past the pointer lists, so only the table this plan uploaded is accepted.
    if not isinstance(table, torch.Tensor) or plan.__dict__.get("_list_tables", {}).get(table.device) is not table:
        raise ValueError("table must be this plan's device run table (Plan.list_table)")
    if table.device != device:
        raise ValueError("table is on %s, the lists on %s" % (table.device, device))
    return ctypes.c_void_p(table.data_ptr()), _stream_ptr(stream, device)


def _lists(plan, pl, name, dtype, device, one_list=True):
    """Device pointer of checked PointerLists: built for this plan's shard sizes, of
    ``dtype``, on ``device``, holding one list (or 1..MAX_MICRO micro-batch lists)."""
    if not isinstance(pl, PointerLists):
        raise TypeError("%s must be PointerLists" % name)
    counts = plan.layout().counts
    if pl.counts is not counts and not np.array_equal(pl.counts, counts):
        raise ValueError("%s was built for a plan with other shard sizes" % name)
    if pl.dtype != dtype:
        raise TypeError("%s must hold %s shards (got %s)" % (name, dtype, pl.dtype))
    if pl.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, pl.device, device))
    if one_list and pl.n_lists != 1:
        raise ValueError("%s must be a single list (got %d)" % (name, pl.n_lists))
    return pl.ptr


def list_accumulate(plan, table, grads: PointerLists, micro: PointerLists, overwrite_first=True, stream=None):
    """zero1_list_accumulate: every fp32 gradient shard = [itself +] the sum of its bf16
    micro-batch shards (``micro`` holds one list per micro-batch)."""
    lib = load_library()
    dev = grads.device
    tp, sp = _list_args(plan, table, stream, dev)
    gp = _lists(plan, grads, "grads", torch.float32, dev)
    mp = _lists(plan, micro, "micro", torch.bfloat16, dev, one_list=False)
    _check(lib.zero1_list_accumulate(plan.handle, tp, gp, mp, micro.n_lists, 1 if overwrite_first else 0, sp),
           "zero1_list_accumulate")


def list_accumulate_norm(plan, table, grads: PointerLists, micro: PointerLists, workspace, norm_out,
                         overwrite_first=True, extra_sumsq=0.0, divisor=1.0, stream=None):
    """zero1_list_accumulate_norm: accumulate, divide by ``divisor`` and take the norm record."""
    lib = load_library()
    dev = grads.device
    tp, sp = _list_args(plan, table, stream, dev)
    gp = _lists(plan, grads, "grads", torch.float32, dev)
    mp = _lists(plan, micro, "micro", torch.bfloat16, dev, one_list=False)
    ws = _ptr(workspace, torch.uint8, None, "workspace", dev)
    no = _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_list_accumulate_norm(plan.handle, tp, gp, mp, micro.n_lists,
                                          1 if overwrite_first else 0, float(divisor), float(extra_sumsq), ws,
                                          workspace.numel(), no, sp), "zero1_list_accumulate_norm")


def list_grad_norm(plan, table, grads: PointerLists, workspace, norm_out, extra_sumsq=0.0, stream=None):
    """zero1_list_grad_norm: the norm record of the gradient shards."""
    lib = load_library()
    dev = grads.device
    tp, sp = _list_args(plan, table, stream, dev)
    gp = _lists(plan, grads, "grads", torch.float32, dev)
    ws = _ptr(workspace, torch.uint8, None, "workspace", dev)
    no = _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_list_grad_norm(plan.handle, tp, gp, float(extra_sumsq), ws, workspace.numel(), no, sp),
           "zero1_list_grad_norm")


def list_micro_norm(plan, table, micro: PointerLists, workspace, norm_out, extra_sumsq=0.0, divisor=1.0,
                    stream=None):
    """zero1_list_micro_norm: the norm record of one micro-batch's gradient over the tensor lists,
    without writing the gradient (what list_accumulate_norm(overwrite_first=True) would record)."""
    lib = load_library()
    dev = micro.device
    tp, sp = _list_args(plan, table, stream, dev)
    mp = _lists(plan, micro, "micro", torch.bfloat16, dev)
    ws = _ptr(workspace, torch.uint8, None, "workspace", dev)
    no = _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_list_micro_norm(plan.handle, tp, mp, float(divisor), float(extra_sumsq), ws, workspace.numel(),
                                     no, sp), "zero1_list_micro_norm")


def list_step_accumulate(plan, table, master: PointerLists, exp_avg: PointerLists, exp_avg_sq: PointerLists,
                         grads: PointerLists, micro: PointerLists, weight_bf16, hparams, step_t, norm_out=None,
                         divisor=1.0, stream=None):
    """zero1_list_step_accumulate: list_step for one micro-batch's gradient, written to the gradient
    lists in the same pass (the results of list_accumulate_norm + list_step)."""
    lib = load_library()
    dev = master.device
    tp, sp = _list_args(plan, table, stream, dev)
    ptrs = _step_lists(plan, master, exp_avg, exp_avg_sq, grads, weight_bf16, dev)
    mp = _lists(plan, micro, "micro", torch.bfloat16, dev)
    hp = hparams if isinstance(hparams, Hparams) else Hparams(**hparams)
    no = None if norm_out is None else _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_list_step_accumulate(plan.handle, tp, ptrs[0], ptrs[1], ptrs[2], ptrs[3], mp, float(divisor),
                                          ptrs[4], ctypes.byref(hp._c()), int(step_t), no, sp),
           "zero1_list_step_accumulate")


def _step_lists(plan, master, exp_avg, exp_avg_sq, grads, weight_bf16, dev):
    f32 = [_lists(plan, pl, name, torch.float32, dev) for pl, name in
           ((master, "master"), (exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq"), (grads, "grads"))]
    w = None if weight_bf16 is None else _lists(plan, weight_bf16, "weight_bf16", torch.bfloat16, dev)
    return f32 + [w]


def list_step(plan, table, master: PointerLists, exp_avg: PointerLists, exp_avg_sq: PointerLists,
              grads: PointerLists, weight_bf16, hparams, step_t, norm_out=None, stream=None):
    """zero1_list_step: clip + AdamW + bf16 copy over the tensor lists (weight_bf16 may be None)."""
    lib = load_library()
    dev = master.device
    tp, sp = _list_args(plan, table, stream, dev)
    ptrs = _step_lists(plan, master, exp_avg, exp_avg_sq, grads, weight_bf16, dev)
    hp = hparams if isinstance(hparams, Hparams) else Hparams(**hparams)
    no = None if norm_out is None else _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_list_step(plan.handle, tp, *ptrs, ctypes.byref(hp._c()), int(step_t), no, sp),
           "zero1_list_step")


def list_step_dev(plan, table, master: PointerLists, exp_avg: PointerLists, exp_avg_sq: PointerLists,
                  grads: PointerLists, weight_bf16, d_scalars, norm_out=None, stream=None):
    """zero1_list_step_dev: list_step with the step scalars in device memory (``d_scalars``, a
    CUDA uint8 tensor holding step_scalars() bytes), for CUDA-graph replay."""
    lib = load_library()
    dev = master.device
    tp, sp = _list_args(plan, table, stream, dev)
    ptrs = _step_lists(plan, master, exp_avg, exp_avg_sq, grads, weight_bf16, dev)
    sc = _ptr(d_scalars, torch.uint8, None, "d_scalars", dev)
    if d_scalars.numel() < STEP_SCALARS_BYTES:
        raise ValueError("d_scalars holds %d bytes, the step scalars need %d" % (d_scalars.numel(), STEP_SCALARS_BYTES))
    no = None if norm_out is None else _norm_ptr(norm_out, device=dev)
    _check(lib.zero1_list_step_dev(plan.handle, tp, *ptrs, sc, no, sp), "zero1_list_step_dev")
