"""Host-side pieces of bench.py (no GPU): the CPU baseline legs run the oracle on
contiguous element ranges in parallel and must give the single pass's results bit
for bit, and the reference arm prints the contract's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from zero_sharded_mixed_local_gb300.workloads import get_workload  # noqa: E402


def _sample(w, n, seed):
    master, m, v, micros = bench.host_sample(w, n, seed=seed)
    return master.copy(), m.copy(), v.copy(), micros


def test_threaded_oracle_step_equals_the_single_pass():
    w = get_workload("smollm1p7b")  # K = 8
    n = 100_003 // 8 * 8 + 5   # ragged: not a multiple of the thread count or of 8
    hp = dict(w.hp, clip_grad=1e-3)  # clipping active
    a = _sample(w, n, 3)
    b = _sample(w, n, 3)
    split = n - 1234            # the last 1234 elements excluded from decay
    for t in (1, 2):
        bench.oracle_sample_step(a[0], a[1], a[2], a[3], split, hp, t, threads=1)
        bench.oracle_sample_step(b[0], b[1], b[2], b[3], split, hp, t, threads=7)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "toy",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    d = json.loads(out.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    # the config record is the GPU arm's own, built from the library's plan of the same shard
    import zero_sharded_mixed_local_gb300 as z
    w = get_workload("toy")
    plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, w.dp_rank)
    assert d["config"] == bench.step_config(_default_args(), w, plan.local_numel, plan.local_numel,
                                            plan.arena_numel, w.dp_rank)
    assert d["oracle_sample"]["sample_elements"] > 0 and "sample_elements" not in d["config"]


def _default_args():
    import argparse
    return argparse.Namespace(k_way=False, unfused=False, exchange=False, graph=False, tensor_list=False)


def test_reference_shard_sizes_are_the_plans_for_every_workload_and_rank():
    """The reference arm derives the shard sizes of its config from the oracle's split; they
    equal the library plan's local and padded arena sizes, for every workload and for the
    dp ranks a multi-GPU job steps."""
    import zero_sharded_mixed_local_gb300 as z
    from zero_sharded_mixed_local_gb300.workloads import WORKLOADS
    for name in WORKLOADS:
        w = get_workload(name)
        for world in (1, 2, 8):
            for r in range(min(world, 3)):
                dp = bench.rank_dp_rank(w, world, r)
                plan = z.Plan(w.params.numels, w.params.no_decay, w.dp_size, dp)
                assert bench.oracle_shard_sizes(w, dp) == (plan.local_numel, plan.arena_numel), (name, world, r)


def _rank_worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b.barrier(world)
        total = b.sum_over_ranks(1_000_000_007 + rank, world)   # shard sizes differ by rank
        slowest = b.max_over_ranks(5.0 + rank * 0.25, world)     # per-rank step times
        q.put((rank, total, slowest))
    finally:
        dist.destroy_process_group()
        q.close()
        q.join_thread()


def test_bench_rank_helpers_with_gloo():
    """The whole-job bookkeeping of a multi-rank bench run, as two gloo processes: the job's
    parameter count is the sum of every rank's shard, the step time the slowest rank's."""
    import socket
    import torch.multiprocessing as mp
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2_000_000_015, 5.25), (1, 2_000_000_015, 5.25)]


def test_clock_samples_inside_the_timed_region():
    """The median SM clock comes from the nvidia-smi samples stamped inside the timed region;
    throttle reasons are gathered from every sample (a superset of the region's)."""
    c = bench.ClockSampler(0)
    c.lines = [
        "2026/12/02 10:18:33.100, 0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:18:33.150, 0, 1980, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:18:33.200, 0, 1990, 2070, 1310.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:18:34.150, 0, 1500, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "not a sample line",
    ]
    c.mark(c._when("2026/12/02 10:18:33.120"), c._when("2026/12/02 10:18:33.500"))

    class _Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            pass

    c.proc = _Done()
    got = c.stop()
    assert got["samples"] == 4 and got["samples_in_timed_region"] == 2
    assert got["sm_mhz"] == 1985.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]


def test_traffic_record_from_an_ncu_metrics_list(tmp_path):
    """bench.py --write-traffic-record turns ncu's CSV metrics list into the record the bench
    scales roofline.traffic from: per-launch DRAM read + write of the step kernel only (other
    kernels and units ignored), per parameter, with the kernel sources' hash."""
    head = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
            '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n')

    def row(i, name, metric, unit, value):
        return ('"%d","1","python3","h","%s","1","7","(256, 1, 1)","(9, 1, 1)","0","10.3",'
                '"Command line profiler metrics","%s","%s","%s"\n' % (i, name, metric, unit, value))

    step = "void zero1::<unnamed>::adamw_step_kernel<true, false>(zero1::StepParams, long)"
    lines = ["==PROF== Connected to process 1\n", head]
    for i, (rd, wr) in enumerate(((1600.0, 1400.0), (1602.0, 1398.0))):
        lines += [row(2 * i, "void at::fill_kernel(int)", "dram__bytes_read.sum", "byte", "99"),
                  row(2 * i + 1, step, "dram__bytes_read.sum", "Kbyte", "%.3f" % (rd / 1e3)),
                  row(2 * i + 1, step, "dram__bytes_write.sum", "byte", "%d" % wr),
                  row(2 * i + 1, step, "gpu__time_duration.sum", "us", "4.5")]
    csv_path = tmp_path / "traffic.csv"
    csv_path.write_text("".join(lines))
    out = tmp_path / "rec.json"
    rec = bench.write_traffic_record(str(csv_path), "adamw_step", "tiny", "ncu ...", 100, out=str(out))
    assert rec["capture"]["launches"] == 2
    assert rec["dram_read_bytes_per_launch"] == 1601 and rec["dram_write_bytes_per_launch"] == 1399
    assert rec["traffic_bytes_per_param"] == 30.0 and rec["ncu_duration_us_per_launch"] == 4.5
    assert rec["kernel_source_sha256_16"] == bench.kernel_source_hash("adamw_step")
    assert json.loads(out.read_text()) == rec


def test_committed_traffic_records_match_the_kernel_sources():
    """The records bench.py reads were taken on the kernels as they are (else it reports null)."""
    for kernel in ("adamw_step", "adamw_step_accumulate", "list_step", "list_step_accumulate"):
        path = bench.traffic_record_path(kernel)
        assert path is not None and os.path.basename(path).startswith("traffic_%s_" % kernel), kernel
        rec = json.load(open(path))
        assert rec["kernel_source_sha256_16"] == bench.kernel_source_hash(kernel), kernel
        got, src = bench.profile_traffic(kernel, 1_003_782_656)
        assert got == int(round(rec["traffic_bytes_per_param"] * 1_003_782_656)) and src


def test_clock_rejection_rule():
    """A hardware or thermal slowdown, or an SM clock well below its maximum with no reason, rejects the
    timed region's number; sw_power_cap alone does not."""
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.clock_rejection(ok) is None and bench.clock_rejection(None) is None
    assert bench.clock_rejection(dict(ok, reasons=["sw_power_cap"], sm_mhz=1800.0)) is None
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert r in bench.clock_rejection(dict(ok, reasons=[r, "sw_power_cap"]))
    assert "no throttle reason" in bench.clock_rejection(dict(ok, sm_mhz=1200.0))
    assert bench.clock_rejection(dict(ok, sm_mhz=1900.0)) is None  # within 10% of the maximum
