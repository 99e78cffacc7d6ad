"""Benchmark of the ZeRO-1 local-shard optimizer step on one GB300 (or N, one rank per GPU).

One "step" is the whole hot path over one batch of synthetic gradients:
  K-1 x zero1_accumulate (bf16 micro-batch gradient -> fp32 grad), zero1_accumulate_norm
  (the last micro-batch and the gradient norm in one pass), zero1_step (clip + AdamW on
  fp32 master/m/v + bf16 weight copy).
Default workload: the Llama-3.1-8B-shaped parameter list sharded over dp=8, rank 0
(1,003,782,656 local parameters, K=1).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the scalar CPU oracle on this host's cores instead (the
reference arm); it is a deliberately slow program, reported for context.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "AdamW shard-step params/sec and HBM GB/s (fraction of GB300 peak), 1 GPU"
OUT = sys.stdout  # where the JSON line goes (main() keeps the real stdout for it alone)
STEP_BYTES_PER_ELEM = 30          # adamw_step: grad 4 R, master/m/v 12 R + 12 W, bf16 2 W
NOMINAL_HBM_GBS = 7900.0          # GB300 HBM3e, nominal


def accumulate_bytes_per_elem(k, k_way=False):
    if k_way:  # all K micro-batches in one pass: 2K R + 4 W
        return 2 * k + 4
    # first micro-batch overwrites (2 R + 4 W); each further one is 2 + 4 R + 4 W
    return 6 + 10 * (k - 1)


L2_BYTES = 129e6  # GB300 L2


def path_bytes_for(args, P, K, total=None, world=1):
    """Algorithmic bytes of one step over P local parameters (padding excluded).  A
    --data-parallel rank also moves, per micro-batch, its model-layout gradient through the
    pack (2 R + 2 W per model parameter) and the all-to-all (2 R + 2 W), and adds the world's
    chunks (2 B each per local parameter); after the step the all-gather (2 R per local, 2 W
    per model parameter) and the unpack (2 R + 2 W per model parameter)."""
    if getattr(args, "data_parallel", False):
        total = P if total is None else total
        acc = sum(2 * world + (4 if k == 0 else 8) for k in range(K)) * P
        return K * 8 * total + acc + STEP_BYTES_PER_ELEM * P + 2 * P + 6 * total
    if uses_micro_step(args, K):  # the norm from the micro-batch (2), the step that writes the gradient (32)
        return 34 * P
    return ((accumulate_bytes_per_elem(K, args.k_way) + STEP_BYTES_PER_ELEM) * P + (4 * P if args.unfused else 0) +
            (8 * P if args.exchange else 0))


def uses_micro_step(args, K):
    """One micro-batch in the plain arena step: its norm taken from the micro-batch, then the step
    that writes the gradient (zero1_micro_norm + zero1_step_accumulate), unless asked otherwise."""
    return (K == 1 and not (getattr(args, "accumulate_first", False) or args.k_way or args.unfused or args.exchange
                            or args.graph or getattr(args, "data_parallel", False)))


def flushes_l2(path_bytes):
    """A step whose bytes would mostly stay in L2 from one step to the next is timed with L2 flushed."""
    return path_bytes < 4 * L2_BYTES


def l2_note(path_bytes):
    if flushes_l2(path_bytes):
        return ("L2 flushed before every step (256 MB write outside the step's events): a step moves %.1f MB "
                "against the 129 MB L2; the timed steps carry no per-kernel events (a second pass times the "
                "parts)" % (path_bytes / 1e6))
    return "no flush: each step streams %.1f GB, far above the 129 MB L2" % (path_bytes / 1e9)


def data_parallel_workload(w, world):
    """--data-parallel: the workload's whole model over a ZeRO-1 job of `world` ranks."""
    w.dp_size, w.dp_rank = world, 0
    w.description = "%s-shaped list, whole model (%d params), ZeRO-1 data-parallel job of %d rank%s, K=%d" % (
        w.name, sum(w.params.numels), world, "s" if world > 1 else "", w.micro_batches)
    return w


def rank_dp_rank(w, world, rank):
    """The data-parallel shard rank `rank` of a `world`-GPU job steps (weak scaling: one shard per GPU)."""
    return (w.dp_rank + rank) % w.dp_size if world > 1 else w.dp_rank


def step_config(args, w, local, job, arena, dp_rank):
    """The `config` record of a bench line: the same keys and values for the GPU arm and the
    reference (oracle) arm of one workload and one set of options."""
    return {
        "workload": w.description,
        "local_params_per_gpu": int(local),
        "params_per_step_all_ranks": int(job),
        "arena_elems": int(arena),
        "micro_batches": w.micro_batches,
        "dp_size": w.dp_size,
        "dp_rank": int(dp_rank),
        "parallelism": ("zero1 data-parallel job, dp%d (one shard per GPU, real collectives)" % w.dp_size
                        if getattr(args, "data_parallel", False) else "zero1 dp%d shard per GPU" % w.dp_size),
        "seed": w.seed,
        "norm": ("separate pass" if args.unfused else
                 "taken from the one micro-batch; the step writes the gradient (zero1_micro_norm + "
                 "zero1_step_accumulate)" if uses_micro_step(args, w.micro_batches) else
                 "fused into the last micro-batch's accumulation"),
        "accumulate": ("all K micro-batches in one pass (K-way)" if args.k_way
                       else "one call per micro-batch, as they arrive"),
        "exchange": ("reduce-scatter (pack, all-to-all of bf16 chunks, owner's fp32 sum in (micro-batch, rank) "
                     "order, divide by the world size), sum-of-squares all-reduce, all-gather + unpack of the bf16 "
                     "weights" if getattr(args, "data_parallel", False) else
                     "pack the reduce-scatter input and unpack the bf16 weights, model layout <-> arena"
                     if args.exchange else "none (the local step only)"),
        "launch": ("one CUDA graph per step (StepGraph)" if args.graph else
                   "one library call per step (zero1_local_step)" if getattr(args, "one_call", False) else
                   "eager calls"),
        "layout": ("tensor lists: one allocation per tensor shard, a 16384-element run table"
                   if args.tensor_list else "arenas: one padded buffer per quantity"),
        "l2": l2_note(path_bytes_for(args, local, w.micro_batches, int(sum(w.params.numels)), w.dp_size)),
    }


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


TRAFFIC_SOURCES = {"adamw_step": ["adamw_step.cu", "elementwise.cuh", "l2_policy.cuh", "launch.cuh", "store8.cuh"],
                   "adamw_step_accumulate": ["adamw_step.cu", "elementwise.cuh", "l2_policy.cuh", "launch.cuh",
                                             "store8.cuh"],
                   "list_step": ["tensor_list.cu", "elementwise.cuh", "l2_policy.cuh", "launch.cuh"],
                   "list_step_accumulate": ["tensor_list.cu", "elementwise.cuh", "l2_policy.cuh", "launch.cuh"]}
# algorithmic bytes per parameter of each step kernel: the one-micro-batch form reads the 2-byte
# micro-batch instead of the 4-byte gradient and writes the gradient (4)
STEP_KERNEL_BYTES = {"adamw_step": STEP_BYTES_PER_ELEM, "list_step": STEP_BYTES_PER_ELEM, "adamw_step_accumulate": 32,
                     "list_step_accumulate": 32}
# the kernel each record's launches belong to, and how the roofline names it
STEP_KERNEL_NAMES = {"adamw_step": ("adamw_step_kernel", "adamw_step_kernel"),
                     "adamw_step_accumulate": ("adamw_step_kernel", "adamw_step_kernel (one-micro-batch form)"),
                     "list_step": ("list_step_kernel", "list_step_kernel"),
                     "list_step_accumulate": ("list_step_kernel", "list_step_kernel (one-micro-batch form)")}


def kernel_source_hash(kernel):
    """First 16 hex digits of the SHA-256 of the kernel's sources (the kernel file, the
    per-element arithmetic and the launch helper it includes)."""
    csrc = os.path.join(ROOT, "zero_sharded_mixed_local_gb300", "csrc")
    h = hashlib.sha256()
    for src in TRAFFIC_SOURCES[kernel]:
        with open(os.path.join(csrc, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record_path(kernel, workload=None):
    """profiles/traffic_<kernel>_<workload>.json; without `workload`, the one record of `kernel`
    (None if there is none)."""
    if workload is not None:
        return os.path.join(ROOT, "profiles", "traffic_%s_%s.json" % (kernel, workload))
    from zero_sharded_mixed_local_gb300.workloads import WORKLOADS  # kernel names share prefixes
    found = [p for p in (traffic_record_path(kernel, name) for name in WORKLOADS) if os.path.exists(p)]
    return found[0] if len(found) == 1 else None


def profile_traffic(kernel, params):
    """DRAM bytes per launch of `kernel` ("adamw_step" or "list_step") over `params` parameters:
    the machine-written record profiles/traffic_<kernel>.json holds the ncu DRAM read + write
    bytes of launches on a small workload, per parameter; scaled here to `params`.  None if the
    record is missing or was taken on other kernel sources."""
    path = traffic_record_path(kernel)
    if path is None:
        return None, None
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("kernel_source_sha256_16") != kernel_source_hash(kernel):
            return None, None
        return int(round(float(rec["traffic_bytes_per_param"]) * params)), (
            "%s: ncu DRAM read + write on %s (%d params per launch, %d launches), %.4f B/param, scaled to %d params"
            % (os.path.relpath(path, ROOT), rec["capture"]["workload"],
               rec["capture"]["params_per_launch"], rec["capture"]["launches"], rec["traffic_bytes_per_param"],
               params))
    except (OSError, KeyError, ValueError, TypeError):
        return None, None


def parse_ncu_csv(path, kernel):
    """Per-launch (dram read, dram write, duration ns) of the launches of `kernel` in an ncu
    `--csv --log-file` metrics list."""
    import csv
    rows = {}
    with open(path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        if kernel not in r["Kernel Name"]:
            continue
        d = rows.setdefault(r["ID"], {})
        unit, value = r["Metric Unit"], float(r["Metric Value"].replace(",", ""))
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9,
                 "ns": 1, "nsecond": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}[unit]
        d[r["Metric Name"]] = value * scale
    return [(d["dram__bytes_read.sum"], d["dram__bytes_write.sum"], d.get("gpu__time_duration.sum"))
            for _, d in sorted(rows.items(), key=lambda kv: int(kv[0]))]


def write_traffic_record(csv_path, kernel, workload, command, params, out=None):
    """Summarise an ncu capture of `kernel` on `workload` (`params` parameters per launch) into
    the machine-written record profile_traffic() reads."""
    launches = parse_ncu_csv(csv_path, STEP_KERNEL_NAMES[kernel][0])
    if not launches:
        raise SystemExit("no %s_kernel launches in %s" % (kernel, csv_path))
    rd = statistics.mean(x[0] for x in launches)
    wr = statistics.mean(x[1] for x in launches)
    durs = [x[2] for x in launches if x[2] is not None]
    rec = {
        "kernel": STEP_KERNEL_NAMES[kernel][1],
        "kernel_source_sha256_16": kernel_source_hash(kernel),
        "capture": {"workload": workload, "params_per_launch": int(params), "launches": len(launches),
                    "command": command, "csv": os.path.basename(csv_path)},
        "dram_read_bytes_per_launch": int(round(rd)),
        "dram_write_bytes_per_launch": int(round(wr)),
        "traffic_bytes_per_launch": int(round(rd + wr)),
        "traffic_bytes_per_param": (rd + wr) / params,
        "algorithmic_bytes_per_param": STEP_KERNEL_BYTES[kernel],
        "ncu_duration_us_per_launch": statistics.mean(durs) / 1e3 if durs else None,
        "note": "cold-cache, serialised ncu launches: use the bytes, not the duration",
    }
    out = out or traffic_record_path(kernel, workload)
    with open(out, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms around the timed region.
    Each sample carries nvidia-smi's own timestamp, so the median SM clock is taken over the
    samples that fall inside the region (all samples if none do); the throttle reasons are
    collected over every sample, a superset of the region's."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None
        self.region = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self, t_begin, t_end):
        """The timed region in host wall-clock seconds (time.time())."""
        self.region = (t_begin, t_end)

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        samples, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                samples.append((self._when(parts[0]), float(parts[2])))
                mx = float(parts[3])
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not samples:
            return None
        inside = [mhz for when, mhz in samples
                  if self.region is not None and when is not None and self.region[0] <= when <= self.region[1]]
        return {"sm_mhz": statistics.median(inside or [mhz for _, mhz in samples]), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(samples), "samples_in_timed_region": len(inside),
                "interval_ms": self.INTERVAL_MS}


def dist_setup(one_rank_group=False):
    """(world, rank, device index) from the launcher's environment, and a process group when there
    are several ranks (or, with `one_rank_group`, a one-rank NCCL group on this GPU).

    The collectives run on NCCL, one rank per GPU.  ZERO1_BENCH_BACKEND=gloo is a functional check
    of the multi-rank code on a box with fewer GPUs than ranks: the ranks share the visible GPUs
    round-robin and the collectives run on gloo (no rank's kernel waits for another's).  Its numbers
    are not a multi-GPU measurement, and the line says which backend ran."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    backend = os.environ.get("ZERO1_BENCH_BACKEND", "nccl")
    if backend not in ("nccl", "gloo"):
        raise SystemExit("ZERO1_BENCH_BACKEND must be nccl or gloo")
    device = local if backend == "nccl" else local % max(1, torch.cuda.device_count())
    if world > 1 or one_rank_group:
        import torch.distributed as dist
        torch.cuda.set_device(device)
        if world > 1 and backend == "gloo":
            dist.init_process_group("gloo")
        elif world > 1:
            dist.init_process_group("nccl", device_id=torch.device("cuda", device))
        else:
            import socket
            sock = socket.socket()
            sock.bind(("127.0.0.1", 0))
            port = sock.getsockname()[1]
            sock.close()
            dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0, world_size=1,
                                    device_id=torch.device("cuda", device))
    return world, rank, device


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _collective_device():
    import torch.distributed as dist
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def sum_over_ranks(x, world):
    """Whole-job total of a per-rank count (the ranks' shards differ by the remainder rule)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.int64, device=_collective_device())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


THROTTLE_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clock_rejection(clk):
    """Why a timed region's clock record rejects its number, or None: a hardware or thermal slowdown
    seen during it, or a median SM clock well below the maximum with no reason given (a clock lock left
    behind).  sw_power_cap is kept (normal for a 1.4 kW part under load) and shows in `reasons`."""
    if not clk:
        return None
    bad = [r for r in clk.get("reasons", []) if r in THROTTLE_REASONS]
    if bad:
        return "throttled: " + ", ".join(bad)
    mx, med = clk.get("sm_max_mhz"), clk.get("sm_mhz")
    if mx and med and med < 0.9 * mx and not clk.get("reasons"):
        return "SM clock %.0f of %.0f MHz with no throttle reason" % (med, mx)
    return None


def max_over_ranks(x, world):
    """The slowest rank's time: the whole job waits for it."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=_collective_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU (oracle)
def oracle_sample_step(master, m, v, micros, no_decay_split, hp, t, threads=1, grad=None, w=None):
    """One oracle step over host arrays (the sample), returning seconds.  `grad` and `w`
    (fp32 and bf16-bits scratch of the sample's length) may be passed in so that their
    first-touch page faults stay out of the timed region.

    With threads > 1 the oracle's own functions run on contiguous element ranges in
    parallel (ctypes releases the GIL): accumulate and the range's sum of squares, then,
    after the partial sums are added in range order, AdamW with the bf16 copy.  Every
    element gets the same operations as in the single pass; only the sum of squares is
    added in a different order (to ~1e-16 relative), so the results are bit-identical
    whenever the fp32 clip coefficient is."""
    import oracle
    n = master.size
    grad = np.zeros(n, np.float32) if grad is None else grad
    w = np.zeros(n, np.uint16) if w is None else w
    t0 = time.perf_counter()
    if threads <= 1:
        oracle.accumulate_all(grad, micros)
        s = oracle.sumsq(grad)
        ok, norm, coef = oracle.clip_coef(s, hp["clip_grad"])
        oracle.adamw(master, m, v, grad, [no_decay_split, n - no_decay_split], [0, 1], hp, t, coef, w=w)
        return time.perf_counter() - t0
    from concurrent.futures import ThreadPoolExecutor
    cuts = [min(n, (n * i // threads) // 8 * 8) for i in range(threads)] + [n]
    ranges = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]

    def grad_part(r):
        a, b = r
        oracle.accumulate_all(grad[a:b], [mb[a:b] for mb in micros])
        return oracle.sumsq(grad[a:b])

    with ThreadPoolExecutor(max_workers=len(ranges)) as ex:
        s = sum(ex.map(grad_part, ranges))  # map keeps range order
        ok, norm, coef = oracle.clip_coef(s, hp["clip_grad"])

        def step_part(r):
            a, b = r
            dec = max(0, min(b, no_decay_split) - a)
            oracle.adamw(master[a:b], m[a:b], v[a:b], grad[a:b], [dec, (b - a) - dec], [0, 1], hp, t, coef,
                         w=w[a:b])

        list(ex.map(step_part, ranges))
    return time.perf_counter() - t0


def host_threads():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def host_sample(w, n_sample, seed=0):
    """A bounded host sample of the workload: n_sample elements drawn like its decayed
    tensors (master N(0, 0.02), K bf16 gradients N(0, sigma^2), m = v = 0)."""
    g = torch.Generator().manual_seed(seed)
    master = (torch.randn(n_sample, generator=g) * 0.02).numpy()
    micros = [(torch.randn(n_sample, generator=g) * w.grad_sigma).to(torch.bfloat16).view(torch.int16)
              .numpy().view(np.uint16) for _ in range(w.micro_batches)]
    return master, np.zeros(n_sample, np.float32), np.zeros(n_sample, np.float32), micros


def timed_oracle_steps(w, n, threads, budget_s, max_steps=50):
    """params/s of repeated oracle steps on one n-element sample, after an untimed step
    that touches every buffer (page faults are not oracle work)."""
    master, m, v, mic = host_sample(w, n, seed=1)
    grad, wb = np.zeros(n, np.float32), np.zeros(n, np.uint16)
    oracle_sample_step(master, m, v, mic, n, w.hp, 1, threads, grad, wb)
    steps, total = 0, 0.0
    while steps < max_steps and (steps == 0 or total < budget_s):
        total += oracle_sample_step(master, m, v, mic, n, w.hp, 2 + steps, threads, grad, wb)
        steps += 1
    return steps * n / total, steps, total


def cpu_baseline(w, target_s=10.0, max_elems=1 << 27):
    """Time the oracle as it stands on a bounded sample for about target_s seconds: two thirds on
    every host core (contiguous ranges, the headline value), the rest on one core."""
    threads = host_threads()
    res = {}
    for nt in sorted({threads, 1}, reverse=True):
        budget = (target_s * 2 / 3 if nt > 1 else target_s / 3) if threads > 1 else target_s
        probe = 1 << 21
        per_elem = 1.0 / timed_oracle_steps(w, probe, nt, 0.0, max_steps=1)[0]
        n = int(min(max(probe, budget / 4 / per_elem), max_elems)) // 8 * 8   # at least ~4 steps
        res[nt] = (n,) + timed_oracle_steps(w, n, nt, budget, max_steps=1000)
    n, value, steps, total = res[threads]
    n1, value1, steps1, total1 = res[1]
    return {"value": value, "unit": "params/s", "cores": threads, "kind": "oracle",
            "sample": "%d elements drawn like the workload's decayed tensors; %d full steps (K=%d accumulate, norm, "
                      "AdamW + bf16 copy) of scalar C on %d threads over contiguous ranges, %.1f s "
                      "(%.0f core-seconds), after one untimed step" % (n, steps, w.micro_batches, threads, total,
                                                                       total * threads),
            "single_core": {"value": value1, "elements": n1, "steps": steps1, "seconds": total1}}


def oracle_shard_sizes(w, dp_rank):
    """(local elements, padded arena elements) of one dp rank's shard: the oracle's shard split,
    each shard padded to a multiple of 8 elements as the arenas are."""
    import oracle
    _, count, local = oracle.plan(w.params.numels, w.dp_size, dp_rank)
    return int(local), int(sum((int(c) + 7) // 8 * 8 for c in count))


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    threads = host_threads()
    per_elem = 1.0 / timed_oracle_steps(w, 1 << 20, threads, 0.0, max_steps=1)[0]
    value1 = timed_oracle_steps(w, 1 << 22, 1, 2.0, max_steps=4)[0]
    # each step a bounded sample, sized so the whole run stays within a few minutes
    budget_s = 120.0 / max(1, args.steps + args.warmup)
    n = max(1 << 20, min(int(budget_s / max(per_elem, 1e-12)), 1 << 27)) // 8 * 8
    m_, mm, vv, mic = host_sample(w, n, seed=1)
    grad, wb = np.zeros(n, np.float32), np.zeros(n, np.uint16)
    for t in range(1, args.warmup + 1):
        oracle_sample_step(m_, mm, vv, mic, n, w.hp, t, threads, grad, wb)
    times = [oracle_sample_step(m_, mm, vv, mic, n, w.hp, args.warmup + t, threads, grad, wb)
             for t in range(1, args.steps + 1)]
    sec = sum(times) / len(times)
    value = n / sec
    # the same workload record as the GPU arm: rank 0's shard, and every rank's shard in the job total
    dp0 = rank_dp_rank(w, world, 0)
    local, arena = oracle_shard_sizes(w, dp0)
    job = sum(oracle_shard_sizes(w, rank_dp_rank(w, world, r))[0] for r in range(world))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "strong" if args.data_parallel else "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": step_config(args, w, local, job, arena, dp0),
        "oracle_sample": {"sample_elements": n,
                          "launch": "scalar C oracle on %d host threads over contiguous element ranges" % threads,
                          "note": "each step runs the whole path (K-micro-batch accumulate, norm, AdamW + bf16 "
                                  "copy) over this many elements drawn like the workload's decayed tensors; "
                                  "params/s = elements / step time"},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": threads, "kind": "oracle",
                         "sample": "%d elements drawn like the workload's decayed tensors, per step" % n,
                         "single_core": {"value": value1, "elements": 1 << 22}},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), file=OUT, flush=True)


# ------------------------------------------------------------------ GPU
def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-torch-baseline", action="store_true",
                    help="skip the stock-PyTorch version of the step on the same GPU")
    ap.add_argument("--checkpoint-io", action="store_true",
                    help="also time an optimizer-shard checkpoint of the state (save_async, save, load) on "
                         "the host's disk, outside the timed step")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0)
    ap.add_argument("--unfused", action="store_true",
                    help="take the norm in its own pass (zero1_grad_norm) instead of fusing it into the last "
                         "micro-batch's accumulation")
    ap.add_argument("--graph", action="store_true",
                    help="replay the step as a CUDA graph (StepGraph) instead of eager calls; one GPU only")
    ap.add_argument("--tensor-list", action="store_true",
                    help="run the tensor-list calls (one allocation per tensor shard, a run table walked by "
                         "the kernels) instead of the arena calls")
    ap.add_argument("--k-way", action="store_true",
                    help="accumulate all K micro-batch gradients (already resident) in one fused pass with the "
                         "norm, instead of one call per micro-batch as they arrive")
    ap.add_argument("--accumulate-first", action="store_true",
                    help="with one micro-batch, still accumulate it (with the norm) before the step instead of "
                         "taking the norm from the micro-batch and letting the step write the gradient")
    ap.add_argument("--one-call", action="store_true",
                    help="the whole local step as one library call (zero1_local_step: all K micro-batches, already "
                         "resident, accumulated with the norm in one pass, then the step); implies --k-way")
    ap.add_argument("--exchange", action="store_true",
                    help="add the copies around the local step: pack the last micro-batch's reduce-scatter input "
                         "from a model-layout bf16 gradient (zero1_shard_gather) and unpack the bf16 weights into "
                         "the model layout (zero1_shard_scatter)")
    ap.add_argument("--data-parallel", action="store_true",
                    help="the workload's whole model stepped by a ZeRO-1 job of this run's ranks (dp size = the "
                         "number of GPUs, rank r owns shard r): per micro-batch the pack, the all-to-all and the "
                         "owner's fp32 accumulation, the sum-of-squares all-reduce, the local step, the all-gather "
                         "and unpack of the bf16 weights (DataParallelStep, NCCL; one GPU runs a one-rank group)")
    ap.add_argument("--micro-batches", type=int, default=None,
                    help="override the workload's K (used to profile the one-micro-batch path on a small shard)")
    ap.add_argument("--seed", type=int, default=None,
                    help="seed of the synthetic inputs (default: the workload's own, 0); rank r adds r")
    ap.add_argument("--write-traffic-record", metavar="NCU_CSV", default=None,
                    help="no GPU work: summarise an ncu --csv metrics list (dram__bytes_read.sum, "
                         "dram__bytes_write.sum, gpu__time_duration.sum) of the step kernel on --workload into "
                         "profiles/traffic_<kernel>.json, the record roofline.traffic is scaled from")
    ap.add_argument("--traffic-command", default="",
                    help="with --write-traffic-record: the ncu command that made the CSV, stored in the record")
    args = ap.parse_args()
    if args.tensor_list and args.unfused:
        raise SystemExit("--tensor-list runs the fused calls")
    if args.one_call:
        if args.unfused or args.graph or args.tensor_list or args.exchange or args.data_parallel:
            raise SystemExit("--one-call runs the arena step as one eager call")
        args.k_way = True
    if args.k_way and (args.unfused or args.graph):
        raise SystemExit("--k-way runs the fused eager calls")
    if args.exchange and (args.tensor_list or args.graph):
        raise SystemExit("--exchange runs the arena calls eagerly")
    if args.data_parallel and (args.tensor_list or args.graph or args.exchange or args.k_way or args.unfused):
        raise SystemExit("--data-parallel runs the arena calls eagerly, one call per micro-batch")
    if args.tensor_list or args.exchange or args.data_parallel:
        args.no_e2e = True  # the end-to-end leg stages arenas for the plain step
    if args.data_parallel:
        args.no_torch_baseline = True
    return args


EVENTS = ("x0", "a0", "n0", "s0", "s1", "x1")  # exchange in, accumulate, last pass, step, exchange out


class StepBench:
    """One rank's bench state: the plan, the buffers of the chosen layout and the step.

    With N ranks each rank steps a different data-parallel shard of the same model
    (weak scaling); the one exchange on the path is the all-reduce of the sum of
    squares."""

    def __init__(self, args, w, z, world, rank, local):
        from zero_sharded_mixed_local_gb300.workloads import InputGenerator, Layout
        self.args, self.w, self.z, self.world = args, w, z, world
        self.dev = dev = torch.device("cuda", local)
        self.dp_rank = rank_dp_rank(w, world, rank)
        t0 = time.perf_counter()
        self.plan = plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, self.dp_rank)
        self.plan_ms = (time.perf_counter() - t0) * 1e3  # a1, on the host, once per job
        L = plan.layout()
        gen = InputGenerator(w, Layout(L.counts, L.offsets, L.no_decay, L.arena_numel), dev, seed=w.seed + rank)
        self.P, self.K = plan.local_numel, w.micro_batches
        self.master = gen.master()
        self.m, self.v, self.grad = gen.zeros(), gen.zeros(), gen.zeros()
        self.wbf = gen.zeros(torch.bfloat16)
        self.micros = gen.micro_grads()
        self.ws, self.nout = plan.new_workspace(dev), z.new_norm_out(dev)
        self.hp = z.Hparams(**w.hp)
        self.group = None
        if world > 1:
            import torch.distributed as dist
            self.group = dist.group.WORLD
        self.stream = torch.cuda.current_stream(dev)
        self.t = 0
        self.lists = self.lopt = None
        if args.tensor_list:
            self._to_tensor_lists()
        self.full_g = self.full_w = None
        if args.exchange:
            # the model-layout gradient holds this rank's shard values where the plan puts them
            self.full_g = torch.zeros(plan.total_numel, dtype=torch.bfloat16, device=dev)
            self.full_w = torch.zeros(plan.total_numel, dtype=torch.bfloat16, device=dev)
            z.shard_scatter(plan, self.micros[self.K - 1], self.full_g)
        self.graph = None
        if args.graph:
            self._capture_graph()
        torch.cuda.synchronize()

    def _to_tensor_lists(self):
        """One allocation per tensor shard, as a framework holds per-parameter state, filled from
        the generated arenas (which are then freed) and reached through pointer lists."""
        z, plan, dev = self.z, self.plan, self.dev

        def split(buf):
            return [t.clone() for t in plan.shard_views(buf)]

        w = self.w
        lopt = z.ShardListAdamW(w.params.numels, w.params.no_decay, w.dp_size, self.dp_rank, hparams=self.hp,
                                device=dev, master=split(self.master), exp_avg=split(self.m),
                                exp_avg_sq=split(self.v), grad=split(self.grad), weight_bf16=split(self.wbf))
        L = lopt.pointer_lists
        plan = self.plan = lopt.plan  # the list calls take the plan whose run table they use
        micro_shards = [split(mb) for mb in self.micros]
        self.lists = {"master": L["master"], "m": L["exp_avg"], "v": L["exp_avg_sq"], "grad": L["grad"],
                      "w": L["weight_bf16"],
                      "micro": [z.PointerLists(plan, ms, torch.bfloat16, dev) for ms in micro_shards],
                      "micro_all": z.PointerLists(plan, micro_shards, torch.bfloat16, dev)}  # K lists back to back
        self.master = self.m = self.v = self.grad = self.wbf = self.micros = None
        torch.cuda.empty_cache()
        self.table, self.lws = lopt.table, lopt.workspace
        lopt.norm_out = self.nout
        self.lopt = lopt

    def _capture_graph(self):
        if self.world > 1:
            raise SystemExit("--graph runs one rank (the captured step holds no all-reduce)")
        if self.lopt is not None:
            self.graph = self.z.StepGraph(self.lopt, self.lists["micro"])
        else:
            from types import SimpleNamespace
            state = SimpleNamespace(plan=self.plan, grad=self.grad, workspace=self.ws, norm_out=self.nout,
                                    master=self.master, exp_avg=self.m, exp_avg_sq=self.v, weight_bf16=self.wbf,
                                    hp=self.hp, t=0, device=self.dev)
            self.graph = self.z.StepGraph(state, self.micros)

    @property
    def step_kernel(self):
        return (("list_step" if self.lists is not None else "adamw_step") +
                ("_accumulate" if uses_micro_step(self.args, self.K) else ""))

    def step(self, rec=None):
        """One pass of the hot path; `rec` (a dict of CUDA events, EVENTS) brackets its parts."""
        mark = (lambda k: rec[k].record(self.stream)) if rec is not None else (lambda k: None)
        if self.graph is not None:  # one graph launch: no events inside it
            mark("a0")
            self.graph.replay()
            mark("s1")
        elif self.lists is not None:
            self._list_step(mark)
        else:
            self._arena_step(mark)

    def _list_step(self, mark):
        z, a, K, L, s = self.z, self.args, self.K, self.lists, self.stream
        self.t += 1
        mark("a0")
        if uses_micro_step(a, K):  # one micro-batch: its norm, then the step that writes the gradients
            mark("n0")
            z.list_micro_norm(self.plan, self.table, L["micro"][0], self.lws, self.nout, stream=s)
            if self.group is not None:
                z.allreduce_sumsq_(self.nout, self.group)
            mark("s0")
            z.list_step_accumulate(self.plan, self.table, L["master"], L["m"], L["v"], L["grad"], L["micro"][0], L["w"],
                                   self.hp, self.t, self.nout, stream=s)
            mark("s1")
            return
        for k in range(0 if a.k_way else K - 1):
            z.list_accumulate(self.plan, self.table, L["grad"], L["micro"][k], overwrite_first=(k == 0), stream=s)
        mark("n0")
        if a.k_way:
            z.list_accumulate_norm(self.plan, self.table, L["grad"], L["micro_all"], self.lws, self.nout,
                                   overwrite_first=True, stream=s)
        else:
            z.list_accumulate_norm(self.plan, self.table, L["grad"], L["micro"][K - 1], self.lws, self.nout,
                                   overwrite_first=(K == 1), stream=s)
        if self.group is not None:
            z.allreduce_sumsq_(self.nout, self.group)
        mark("s0")
        z.list_step(self.plan, self.table, L["master"], L["m"], L["v"], L["grad"], L["w"], self.hp, self.t,
                    self.nout, stream=s)
        mark("s1")

    def _arena_step(self, mark):
        z, a, K, s, plan = self.z, self.args, self.K, self.stream, self.plan
        self.t += 1
        mark("x0")
        if self.full_g is not None:  # pack: this rank's chunk of the reduce-scatter input
            z.shard_gather(plan, self.full_g, self.micros[K - 1], stream=s)
        mark("a0")
        for k in range(0 if a.k_way else K - 1):
            z.accumulate(plan, self.grad, self.micros[k], overwrite_first=(k == 0), stream=s)
        mark("n0")
        if uses_micro_step(a, K):  # one micro-batch: its norm, then the step that writes the gradient
            z.micro_norm(plan, self.micros[0], self.ws, self.nout, stream=s)
            if self.group is not None:
                z.allreduce_sumsq_(self.nout, self.group)
            mark("s0")
            z.step_accumulate(plan, self.master, self.m, self.v, self.grad, self.micros[0], self.wbf, self.hp, self.t,
                              self.nout, stream=s)
            mark("s1")
            mark("x1")
            return
        if a.one_call:  # accumulate + norm and the step in one crossing of the C ABI
            z.local_step(plan, self.grad, self.micros, self.ws, self.nout, self.master, self.m, self.v, self.wbf,
                         self.hp, self.t, stream=s)
            mark("s0")
            mark("s1")
            mark("x1")
            return
        if a.k_way:
            z.accumulate_norm(plan, self.grad, self.micros, self.ws, self.nout, overwrite_first=True, stream=s)
        elif a.unfused:
            z.accumulate(plan, self.grad, self.micros[K - 1], overwrite_first=(K == 1), stream=s)
            z.grad_norm(plan, self.grad, self.ws, self.nout, 0.0, stream=s)
        else:  # the last micro-batch's accumulation also takes the gradient norm
            z.accumulate_norm(plan, self.grad, self.micros[K - 1], self.ws, self.nout, overwrite_first=(K == 1),
                              stream=s)
        if self.group is not None:
            z.allreduce_sumsq_(self.nout, self.group)
        mark("s0")
        z.step(plan, self.master, self.m, self.v, self.grad, self.wbf, self.hp, self.t, self.nout, stream=s)
        mark("s1")
        if self.full_w is not None:  # unpack: the bf16 weights into the model layout
            z.shard_scatter(plan, self.wbf, self.full_w, stream=s)
        mark("x1")

    def launches_per_step(self):
        a = self.args
        return (3 if a.k_way else self.K + 2) + (1 if a.unfused else 0) + (2 if self.full_g is not None else 0)

    def path_bytes(self):
        """Algorithmic bytes of one step (padding excluded)."""
        return path_bytes_for(self.args, self.P, self.K)


class DataParallelBench:
    """--data-parallel: the workload's whole model stepped by a ZeRO-1 job of the run's ranks,
    rank r owning shard r of dp = ranks.  One step is this rank's part of the job
    (DataParallelStep): per micro-batch the pack of its model-layout bf16 gradient, the
    all-to-all and the owner's ordered fp32 accumulation (the last one divided by the world
    size, with the norm), the sum-of-squares all-reduce, the local step, and the all-gather and
    unpack of the bf16 weights.  Rank r's gradients are its own draw (seed + r)."""

    def __init__(self, args, w, z, world, rank, local):
        import torch.distributed as dist
        from zero_sharded_mixed_local_gb300.exchange import DataParallelStep
        from zero_sharded_mixed_local_gb300.workloads import InputGenerator, Layout
        self.args, self.w, self.z, self.world = args, w, z, world
        self.dev = dev = torch.device("cuda", local)
        self.dp_rank = rank
        t0 = time.perf_counter()
        self.opt = opt = z.LocalShardAdamW(w.params.numels, w.params.no_decay, world, rank,
                                           hparams=z.Hparams(**w.hp), device=dev)
        self.plan = plan = opt.plan
        self.plan_ms = (time.perf_counter() - t0) * 1e3
        L = plan.layout()
        opt.master.copy_(InputGenerator(w, Layout(L.counts, L.offsets, L.no_decay, L.arena_numel), dev,
                                        seed=w.seed).master())
        opt.weight_bf16.copy_(opt.master.to(torch.bfloat16))
        model = Layout.packed(w.params.numels, w.params.no_decay)
        self.micros = InputGenerator(w, model, dev, seed=w.seed + rank).micro_grads()
        self.dps = DataParallelStep(opt, group=dist.group.WORLD)
        self.weights = torch.zeros(plan.total_numel, dtype=torch.bfloat16, device=dev)
        self.P, self.K, self.total = plan.local_numel, w.micro_batches, plan.total_numel
        self.stream = torch.cuda.current_stream(dev)
        self.nout = opt.norm_out
        self.graph = self.lists = self.master = self.full_g = self.lopt = None
        self.t = 0
        torch.cuda.synchronize()

    step_kernel = "adamw_step"

    def step(self, rec=None):
        mark = (lambda k: rec[k].record(self.stream)) if rec is not None else (lambda k: None)
        mark("x0")
        for k, g in enumerate(self.micros):
            self.dps.reduce_scatter(g, last=(k == self.K - 1))
        mark("n0")
        self.dps.allreduce_sumsq()
        mark("s0")
        self.opt.step()
        mark("s1")
        self.dps.all_gather(self.weights)
        mark("x1")
        self.t = self.opt.t

    def path_bytes(self):
        return path_bytes_for(self.args, self.P, self.K, self.total, self.world)

    def report(self, recs):
        mean = lambda a, c: statistics.mean(r[a].elapsed_time(r[c]) for r in recs)  # noqa: E731
        parts = {"reduce_scatter": ("x0", "n0"), "allreduce_sumsq": ("n0", "s0"), "adamw_step": ("s0", "s1"),
                 "all_gather": ("s1", "x1")}
        kernels = {}
        for name, (a, c) in parts.items():
            times = [r[a].elapsed_time(r[c]) for r in recs]
            kernels[name] = {"ms": mean(a, c), "ms_median": statistics.median(times), "ms_min": min(times),
                             "ms_max": max(times)}
        kernels["adamw_step"]["gbs"] = STEP_BYTES_PER_ELEM * self.P / (kernels["adamw_step"]["ms"] * 1e-3) / 1e9
        kernels["reduce_scatter"]["note"] = ("per micro-batch: %d pack launches, the all-to-all, %d accumulate "
                                             "call(s)" % (self.world, -(-self.world // self.z.MAX_MICRO)))
        peak, peak_kind = measured_peaks()
        achieved = kernels["adamw_step"]["gbs"]
        traffic, traffic_src = profile_traffic("adamw_step", self.P)
        roofline = {"bound": "hbm", "kernel": "adamw_step_kernel", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                    "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_kind,
                    "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "bytes_per_param": STEP_BYTES_PER_ELEM,
                    "params_per_launch": self.P}
        return kernels, roofline

    def launches_per_step(self):
        per_micro = self.world + -(-self.world // self.z.MAX_MICRO)
        return self.K * per_micro + 1 + 1 + self.world  # + final reduction, step, unpacks


def time_steps(b, args, world, local):
    """W untimed steps, then K timed ones between barriers and synchronises, with the clocks
    sampled meanwhile; returns (per-step event records, max-over-ranks ms per step, clock
    summary, L2 note).  A step whose bytes would mostly stay in L2 from one step to the next
    gets L2 flushed before it (a 256 MB write, outside the step's own events), and its time is
    the mean of the per-step event pairs; larger steps are timed as one region."""
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    flush = None
    if flushes_l2(b.path_bytes()):
        flush = torch.empty(64 << 20, dtype=torch.float32, device=b.dev)  # 256 MB, twice the L2
    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        b.step()
    torch.cuda.synchronize()
    barrier(world)
    visible = [d for d in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if d.strip()]
    clocks = ClockSampler(visible[local].strip() if local < len(visible) else local)  # index or UUID
    clocks.start()
    recs = [{k: ev() for k in EVENTS + ("t0", "t1")} for _ in range(args.steps)]
    start, end = ev(), ev()
    torch.cuda.synchronize()
    barrier(world)
    launches0 = b.z.launch_count()
    t_begin = time.time()
    start.record(b.stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        recs[i]["t0"].record(b.stream)
        # A small step is bound by the host's launches: events recorded inside it would add their
        # own host time, so its timed steps carry only t0 / t1 and the per-kernel events come
        # from a second pass below.
        b.step(None if flush is not None else recs[i])
        recs[i]["t1"].record(b.stream)
    end.record(b.stream)
    b.launches_counted = b.z.launch_count() - launches0  # graph replays launch nothing from the host
    torch.cuda.synchronize()
    clocks.mark(t_begin, time.time())
    barrier(world)
    clk = clocks.stop()
    if flush is not None:
        ms = statistics.mean(r["t0"].elapsed_time(r["t1"]) for r in recs)
        for i in range(args.steps):  # the breakdown pass: the same steps with every part's events
            flush.zero_()
            b.step(recs[i])
        torch.cuda.synchronize()
    else:
        ms = start.elapsed_time(end) / args.steps
    return recs, max_over_ranks(ms, world), clk, l2_note(b.path_bytes())


def kernel_report(b, recs, args):
    """Per-kernel times (CUDA events around each part of the step) and their GB/s."""
    if b.graph is not None:  # one graph launch per step: no per-kernel events inside it
        return None, None
    P, K = b.P, b.K
    mean = lambda a, c: statistics.mean(r[a].elapsed_time(r[c]) for r in recs)  # noqa: E731
    if args.one_call:  # one call per step: its kernels are not separated by events
        times = [r["n0"].elapsed_time(r["s0"]) for r in recs]
        per_param = accumulate_bytes_per_elem(K, True) + STEP_BYTES_PER_ELEM
        ms = statistics.mean(times)
        achieved = per_param * P / (ms * 1e-3) / 1e9
        kernels = {"local_step": {"ms": ms, "gbs": achieved, "launches_per_step": 3, "bytes_per_param": per_param,
                                  "ms_median": statistics.median(times), "ms_min": min(times), "ms_max": max(times)}}
        peak, peak_kind = measured_peaks()
        roofline = {"bound": "hbm", "kernel": "zero1_local_step (accumulate_norm_kway_kernel, sumsq_final_kernel, "
                                              "adamw_step_kernel)", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": None, "traffic_source": None,
                    "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_kind,
                    "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "bytes_per_param": per_param,
                    "params_per_launch": P}
        return kernels, roofline
    acc_ms, accnorm_ms, step_ms = mean("a0", "n0"), mean("n0", "s0"), mean("s0", "s1")
    norm_bytes = 4 * P if args.unfused else 0
    last_bytes = accumulate_bytes_per_elem(K, True) * P if args.k_way else (6 if K == 1 else 10) * P + norm_bytes
    step_bytes = STEP_KERNEL_BYTES[b.step_kernel]
    if uses_micro_step(args, K):  # the norm pass reads the micro-batch only
        last_bytes = 2 * P
    kernels = {
        "accumulate": {"ms": acc_ms, "gbs": (accumulate_bytes_per_elem(K) * P - last_bytes) / (acc_ms * 1e-3) / 1e9
                       if K > 1 and not args.k_way else None, "launches_per_step": 0 if args.k_way else K - 1},
        ("accumulate+grad_norm" if args.unfused else "micro_norm" if uses_micro_step(args, K) else
         "accumulate_norm"): {
            "ms": accnorm_ms, "gbs": last_bytes / (accnorm_ms * 1e-3) / 1e9,
            "launches_per_step": 3 if args.unfused else 2},
        b.step_kernel: {"ms": step_ms, "gbs": step_bytes * P / (step_ms * 1e-3) / 1e9,
                        "launches_per_step": 1},
    }
    if kernels["accumulate"]["launches_per_step"] == 0:  # K = 1 or K-way: its events bracket nothing
        del kernels["accumulate"]
    if b.full_g is not None:  # the layout copies move 2 + 2 bytes per local element each
        for name, (x, y) in (("shard_gather", ("x0", "a0")), ("shard_scatter", ("s1", "x1"))):
            ms = mean(x, y)
            kernels[name] = {"ms": ms, "gbs": 4 * P / (ms * 1e-3) / 1e9, "launches_per_step": 1}
    pairs = {"accumulate": ("a0", "n0"), "accumulate_norm": ("n0", "s0"), "accumulate+grad_norm": ("n0", "s0"),
             "micro_norm": ("n0", "s0"), b.step_kernel: ("s0", "s1"), "shard_gather": ("x0", "a0"),
             "shard_scatter": ("s1", "x1")}
    for name, k in kernels.items():  # "ms" is the mean over the timed steps; the spread beside it
        times = [r[pairs[name][0]].elapsed_time(r[pairs[name][1]]) for r in recs]
        k["ms_median"], k["ms_min"], k["ms_max"] = statistics.median(times), min(times), max(times)
    peak, peak_kind = measured_peaks()
    achieved = kernels[b.step_kernel]["gbs"]
    traffic, traffic_src = profile_traffic(b.step_kernel, P)
    roofline = {"bound": "hbm", "kernel": STEP_KERNEL_NAMES[b.step_kernel][1],
                "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                "traffic_source": traffic_src,
                "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_kind,
                "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "bytes_per_param": step_bytes, "params_per_launch": P}
    return kernels, roofline


def run_e2e(b, args, world, P_job):
    """The same step end to end through the public API: host gradients in, norm record out.

    ``HostFedSteps`` (the package's host-fed loop, which the GPU tests check against the
    synchronous calls and the oracle) copies every step's micro-batch gradients from
    pinned host memory to the device on a side stream, into two staging sets, so step
    t+1's transfer (link-bound, on DMA engines) overlaps step t's kernels (HBM-bound, on
    the SMs); every step's 24-byte norm record is copied back and read on the host, one
    step behind, as a training loop logs it."""
    z, stream = b.z, b.stream
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    host_micros = [mb.cpu().pin_memory() for mb in b.micros]
    loop = z.HostFedSteps(b.plan, b.master, b.m, b.v, b.wbf, b.hp, b.K, t=b.t, k_way=args.k_way, group=b.group,
                          stream=stream, stage0=b.micros, grad0=b.grad, workspace0=b.ws, norm_out0=b.nout)
    seen = loop.run(host_micros, 2)
    torch.cuda.synchronize()
    h2d_bytes = loop.h2d_bytes_per_step
    # the host link's own speed on this machine, for reading the e2e number: one plain copy
    c0, c1 = ev(), ev()
    c0.record(stream)
    for k in range(b.K):
        loop.stage[0][k].copy_(host_micros[k], non_blocking=True)
    c1.record(stream)
    torch.cuda.synchronize()
    h2d_gbs = h2d_bytes / (c0.elapsed_time(c1) * 1e-3) / 1e9
    barrier(world)
    e0, e1 = ev(), ev()
    e0.record(stream)
    seen += loop.run(host_micros, args.steps, first_event=e0, time_copies=True)
    e1.record(stream)
    torch.cuda.synchronize()
    b.t = loop.t
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    copy_ms = statistics.mean(x.elapsed_time(y) for x, y in loop.copy_times)
    assert all(r["status"] == 0 for r in seen)
    return {"value": P_job / (e2e_ms * 1e-3), "unit": "params/s", "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": loop.d2h_bytes_per_step,
            "h2d_copy_gbs_before": h2d_gbs, "h2d_copy_ms_in_loop": copy_ms,
            "h2d_copy_gbs_in_loop": h2d_bytes / (copy_ms * 1e-3) / 1e9,
            "how": "HostFedSteps: pinned host gradients copied by the DMA engines on a side stream into two "
                   "staging sets, overlapping the previous step's kernels; norm record read back every step"}


def torch_baseline(b, args):
    """The same step in stock PyTorch, on the same GPU and the same arenas, the way the pages'
    nanotron configuration runs it (accumulate_grad_in_fp32, clip_grad 1.0, torch_adam_is_fused):
    the bf16 micro-batch gradients copied / added into the fp32 gradient, clip_grad_norm_
    (foreach), torch.optim.AdamW(fused=True) with a decay and a no-decay group, then the bf16 copy
    of the master.  A GPU comparison for the fused kernels; run last, since it changes the state.
    Its own arithmetic differs in order (lerp, addcdiv) and it writes the clipped gradient back."""
    if b.master is None or b.world > 1:
        return None
    P, K, hp = b.P, b.K, b.hp
    master, grad, wbf, micros = b.master, b.grad, b.wbf, b.micros
    groups = []
    for g, wd in ((0, hp.weight_decay), (1, 0.0)):
        lo, hi = b.plan.group_range(g)
        if hi > lo:
            pv = master[lo:hi]
            pv.grad = grad[lo:hi]
            groups.append({"params": [pv], "weight_decay": wd})
    params = [g["params"][0] for g in groups]
    opt = torch.optim.AdamW(groups, lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps, fused=True)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    parts = ("accumulate", "clip_grad_norm_", "adamw_fused", "bf16_copy")

    def step(rec=None):
        def mark(j):
            if rec is not None:
                rec[j].record()
        mark(0)
        grad.copy_(micros[0])
        for k in range(1, K):
            grad.add_(micros[k])
        mark(1)
        torch.nn.utils.clip_grad_norm_(params, hp.clip_grad, foreach=True)
        mark(2)
        opt.step()
        mark(3)
        wbf.copy_(master)
        mark(4)

    flush = torch.empty(64 << 20, dtype=torch.float32, device=b.dev) if flushes_l2(b.path_bytes()) else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    recs = []
    for _ in range(args.steps):
        if flush is not None:
            flush.zero_()
        recs.append([ev() for _ in range(5)])
        step(recs[-1])
    torch.cuda.synchronize()
    ms = statistics.mean(r[0].elapsed_time(r[4]) for r in recs)
    op_bytes = (accumulate_bytes_per_elem(K), 4 + 8, 28, 6)  # clip: norm read, then the scale R+W
    ops = {}
    for j, (name, nb) in enumerate(zip(parts, op_bytes)):
        t = statistics.mean(r[j].elapsed_time(r[j + 1]) for r in recs)
        ops[name] = {"ms": t, "bytes_per_param": nb, "gbs": nb * P / (t * 1e-3) / 1e9}
    per_param = accumulate_bytes_per_elem(K) + 4 + 8 + 28 + 6  # norm read, clip scale R+W, AdamW, bf16 copy
    del opt
    return {"value": P / (ms * 1e-3), "unit": "params/s", "ms_per_step": ms, "bytes_per_param": per_param,
            "hbm_gbs": per_param * P / (ms * 1e-3) / 1e9, "ops": ops,
            "timing": "CUDA events around each op of every step, mean over the timed steps%s" % (
                " (L2 flushed before each step)" if flush is not None else ""),
            "how": "stock PyTorch %s on the same arenas: copy_/add_ of the K bf16 micro-batches into the fp32 "
                   "gradient, clip_grad_norm_(foreach=True), torch.optim.AdamW(fused=True) with decay and no-decay "
                   "groups, bf16 copy_ of the master" % torch.__version__}


def checkpoint_io(b):
    """This rank's optimizer-shard checkpoint (master, m, v) on the host disk, after the timed
    steps: how long save_async holds the caller (the device-to-host snapshot) with new and with
    reused page-locked staging, the whole save (fsync'd files), and a load into scrambled state
    that must restore it bit for bit."""
    import shutil
    import tempfile
    z = b.z
    states = ((b.lopt.master, b.lopt.exp_avg, b.lopt.exp_avg_sq) if b.lopt is not None
              else (b.master, b.m, b.v))
    if any(x is None for x in states):
        return None  # an arena graph run keeps its state in the graph's own object
    flat = lambda x: list(x) if isinstance(x, (list, tuple)) else [x]  # noqa: E731
    before = [t.clone() for x in states for t in flat(x)]
    nbytes = 12 * b.P
    d = tempfile.mkdtemp(prefix="zero1-ckpt-")
    out = {"bytes": nbytes, "where": "the host's local disk, fsync'd; %s" % (
        "per-tensor shard lists" if b.lopt is not None else "arenas")}
    try:
        for label in ("new_staging", "reused_staging"):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fut = z.checkpoint.save_async(d, b.plan, *states, step_t=max(b.t, 1))
            t1 = time.perf_counter()
            fut.result()
            t2 = time.perf_counter()
            out["snapshot_ms_" + label] = (t1 - t0) * 1e3
            out["save_s_" + label] = t2 - t0
        out["snapshot_gbs"] = nbytes / (out["snapshot_ms_reused_staging"] * 1e-3) / 1e9
        z.checkpoint.release_staging()
        t0 = time.perf_counter()
        z.checkpoint.prepare_staging(b.plan)  # what a loop pays once, at start-up, to avoid the first cost
        out["prepare_staging_s"] = time.perf_counter() - t0
        out["save_gbs"] = nbytes / out["save_s_reused_staging"] / 1e9
        for x in states:
            for t in flat(x):
                t.fill_(-1.0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        z.checkpoint.load(d, b.plan, *states)
        torch.cuda.synchronize()
        out["load_s"] = time.perf_counter() - t0
        out["load_gbs"] = nbytes / out["load_s"] / 1e9
        after = [t for x in states for t in flat(x)]
        out["restored_bit_exact"] = all(torch.equal(u.view(torch.int32), v.view(torch.int32))
                                        for u, v in zip(before, after))
    finally:
        shutil.rmtree(d, ignore_errors=True)
        z.checkpoint.release_staging()
    if not out["restored_bit_exact"]:
        raise SystemExit("checkpoint load did not restore the state")
    return out


def claim_stdout():
    """The JSON line is the only thing this program writes to stdout: a duplicate of the real
    stdout is kept for it, and file descriptor 1 is pointed at stderr, so a library banner
    (NCCL prints its version from C) cannot add a line."""
    sys.stdout.flush()
    out = os.fdopen(os.dup(1), "w")
    os.dup2(2, 1)
    return out


def main():
    global OUT
    OUT = claim_stdout()
    args = parse_args()
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    w = get_workload(args.workload)
    if args.micro_batches is not None:
        w.micro_batches = args.micro_batches
        w.description += " (K overridden to %d)" % args.micro_batches
    if args.seed is not None:
        w.seed = args.seed

    if args.write_traffic_record:
        import zero_sharded_mixed_local_gb300 as z
        local = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank).local_numel  # host-only call
        kernel = (("list_step" if args.tensor_list else "adamw_step") +
                  ("_accumulate" if uses_micro_step(args, w.micro_batches) else ""))
        rec = write_traffic_record(args.write_traffic_record, kernel, args.workload, args.traffic_command, local)
        print(json.dumps(rec), file=OUT, flush=True)
        return

    if args.data_parallel:
        data_parallel_workload(w, int(os.environ.get("WORLD_SIZE", "1")))

    if args.impl == "reference":
        run_reference(args, w, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return

    import zero_sharded_mixed_local_gb300 as z

    world, rank, local = dist_setup(one_rank_group=args.data_parallel)
    torch.cuda.set_device(torch.device("cuda", local))
    z.load_library()
    if args.data_parallel:
        b = DataParallelBench(args, w, z, world, rank, local)
    else:
        b = StepBench(args, w, z, world, rank, local)

    recs, ms_step, clk, _ = time_steps(b, args, world, local)
    remeasured = None
    why = clock_rejection(clk)
    if max_over_ranks(1.0 if why else 0.0, world) > 0:  # any rank's clocks reject: every rank measures again
        remeasured = {"first_ms_per_step": ms_step, "first_clocks": clk, "reason": why or "another rank's clocks"}
        recs, ms_step, clk, _ = time_steps(b, args, world, local)
    P_job = sum_over_ranks(b.P, world)  # parameters all ranks step per step
    kernels, roofline = b.report(recs) if args.data_parallel else kernel_report(b, recs, args)
    z.read_norm(b.nout, b.stream)
    path_bytes = b.path_bytes()

    e2e = run_e2e(b, args, world, P_job) if not args.no_e2e and b.graph is None else None

    ckpt = checkpoint_io(b) if args.checkpoint_io and world == 1 else None
    tb = None if args.no_torch_baseline else torch_baseline(b, args)  # last: it changes the state

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_baseline_seconds)
        cpu.pop("seconds", None)
        cpu.pop("elements", None)

    if rank == 0:
        out = {
            "metric": METRIC,
            "value": P_job / (ms_step * 1e-3),
            "unit": "params/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "strong" if args.data_parallel else "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": step_config(args, w, b.P, P_job, b.plan.arena_numel, b.dp_rank),
            "hbm_gbs_step": path_bytes / (ms_step * 1e-3) / 1e9,
            "kernels": kernels,
            "roofline": roofline,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk,
            "clocks_rejection": clock_rejection(clk),  # None: the clocks admit this number
            # counted by the library in eager runs; a graph replays the launches of its one capture
            "gpu_launches": b.launches_counted if b.graph is None else args.steps * b.launches_per_step(),
        }
        if remeasured is not None:
            out["remeasured"] = remeasured
        if world > 1 or args.data_parallel:
            import torch.distributed as dist
            out["collectives"] = dist.get_backend()
        out["plan"] = {"build_ms": b.plan_ms, "tensors": len(w.params.numels),
                       "list_table_bytes": int(b.z.load_library().zero1_list_table_bytes(b.plan.handle)),
                       "layout_table_bytes": int(b.z.load_library().zero1_layout_table_bytes(b.plan.handle))}
        if ckpt is not None:
            out["checkpoint"] = ckpt
        if tb is not None:
            tb["ours_over_torch"] = out["value"] / tb["value"]
            out["torch_baseline"] = tb
        print(json.dumps(out), file=OUT, flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
