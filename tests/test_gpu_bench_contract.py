"""bench.py's JSON line on a GPU: one small run, checked against the keys and units the
measurement contract asks for (the driver runs the full-size default itself)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, lines
    return json.loads(lines[0])


@pytest.mark.parametrize("extra", [[], ["--tensor-list"]])
def test_bench_line_has_the_contract_keys(extra):
    d = _run("--workload", "toy", "--steps", "3", "--warmup", "3", "--cpu-baseline-seconds", "1", *extra)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "clocks", "gpu_launches", "e2e"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["unit"] == "params/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert "workload" in d["config"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    assert d["gpu_launches"] == 3 * (2 + 2)  # K=2: one accumulate, the fused pass (2 kernels), the step
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert "clocks_rejection" in d  # None when the clocks admit the number, else why they do not
    if not extra:
        e = d["e2e"]
        assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 24
        tb = d["torch_baseline"]  # the stock PyTorch step on the same GPU
        assert tb["value"] > 0 and tb["bytes_per_param"] == 6 + 10 + 4 + 8 + 28 + 6  # K = 2
    for k in d["kernels"].values():
        assert k["ms_min"] <= k["ms_median"] <= k["ms_max"]
    assert d["plan"]["tensors"] == 20 and d["plan"]["build_ms"] >= 0 and d["plan"]["list_table_bytes"] > 0
    assert d["clocks"]["interval_ms"] == 50 and d["clocks"]["samples"] >= d["clocks"]["samples_in_timed_region"]


@pytest.mark.parametrize("extra", [[], ["--tensor-list"]])
def test_bench_checkpoint_io_restores_the_state(extra):
    d = _run("--workload", "toy", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-e2e",
             "--checkpoint-io", *extra)
    c = d["checkpoint"]
    assert c["restored_bit_exact"] is True and c["bytes"] == 12 * d["config"]["local_params_per_gpu"]
    assert c["save_gbs"] > 0 and c["load_gbs"] > 0 and c["snapshot_gbs"] > 0


def test_bench_data_parallel_line():
    """--data-parallel on one GPU: the whole toy model through DataParallelStep in a one-rank NCCL
    group (pack, all-to-all, ordered accumulation, all-reduce, step, all-gather, unpack)."""
    d = _run("--workload", "toy", "--data-parallel", "--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    assert d["scaling"] == "strong" and d["value"] > 0
    c = d["config"]
    assert c["dp_size"] == 1 and c["local_params_per_gpu"] == c["params_per_step_all_ranks"] == 3147008
    assert set(d["kernels"]) == {"reduce_scatter", "allreduce_sumsq", "adamw_step", "all_gather"}
    # per step, K = 2: a pack and an accumulate for the first micro-batch, a pack and the fused pass
    # (2 kernels) for the last, the step, the unpack
    assert d["gpu_launches"] == 3 * 7
    assert d["roofline"]["kernel"] == "adamw_step_kernel" and d["roofline"]["params_per_launch"] == 3147008


@pytest.mark.parametrize("extra", [[], ["--tensor-list"]])
def test_bench_one_micro_batch_line(extra):
    """K = 1, the bench's default path: the micro-batch norm (2 kernels) and the step that writes the
    gradient (1 kernel) per step, with the roofline on the step's one-micro-batch form at 32 B/param and
    its traffic from the committed record."""
    d = _run("--workload", "toy", "--micro-batches", "1", "--steps", "3", "--warmup", "3", "--no-cpu-baseline",
             "--no-e2e", "--no-torch-baseline", *extra)
    step = "list_step_accumulate" if extra else "adamw_step_accumulate"
    assert d["gpu_launches"] == 3 * 3
    assert set(d["kernels"]) >= {"micro_norm", step}
    r = d["roofline"]
    assert r["kernel"].endswith("(one-micro-batch form)") and r["bytes_per_param"] == 32
    assert r["traffic"] is not None and r["traffic_source"].startswith("profiles/traffic_" + step + "_")
    assert d["config"]["micro_batches"] == 1
    assert d["clocks_rejection"] is None or "remeasured" in d


def test_bench_one_call_line():
    """--one-call: the whole toy step as one zero1_local_step call (K-way pass, final reduction,
    step: three launches per step)."""
    d = _run("--workload", "toy", "--one-call", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-e2e",
             "--no-torch-baseline")
    assert d["gpu_launches"] == 3 * 3 and set(d["kernels"]) == {"local_step"}
    assert d["config"]["launch"] == "one library call per step (zero1_local_step)"
    assert d["roofline"]["bytes_per_param"] == 2 * 2 + 4 + 30


def _torchrun(nproc, *args):
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    env = dict(os.environ, ZERO1_BENCH_BACKEND="gloo")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=%d" % nproc,
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", str(nproc), *args]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_multi_rank_path_two_ranks_on_gloo():
    """The bench's multi-rank code (per-rank dp shards, the summed job size, the slowest rank's
    time, the sum-of-squares all-reduce on a CUDA record, in the timed steps and inside the
    host-fed e2e loop) with two ranks sharing this GPU over gloo: one line from rank 0, weak
    scaling over dp ranks 0 and 1 of the toy dp4 split."""
    import zero_sharded_mixed_local_gb300 as z
    from zero_sharded_mixed_local_gb300.workloads import get_workload
    d = _torchrun(2, "--workload", "toy", "--steps", "3", "--warmup", "3", "--no-torch-baseline")
    w = get_workload("toy")
    sizes = [z.Plan(w.params.numels, w.params.no_decay, w.dp_size, r).local_numel for r in (0, 1)]
    assert d["n_gpus"] == 2 and d["collectives"] == "gloo" and d["scaling"] == "weak"
    assert d["config"]["params_per_step_all_ranks"] == sum(sizes)
    assert d["config"]["local_params_per_gpu"] == sizes[0] and d["config"]["dp_rank"] == 0
    assert d["value"] > 0 and d["cpu_baseline"] is None
    assert d["gpu_launches"] == 3 * (2 + 2)  # rank 0's own launches
    # the e2e leg: HostFedSteps with the all-reduce inside its loop, every step's record read back
    assert d["e2e"]["value"] > 0 and d["e2e"]["d2h_bytes_per_step"] == 24


def test_bench_data_parallel_two_ranks_on_gloo():
    """--data-parallel with two ranks: DataParallelStep's host-staged collectives between two
    processes sharing this GPU (the toy model split dp2)."""
    d = _torchrun(2, "--workload", "toy", "--data-parallel", "--steps", "3", "--warmup", "3")
    assert d["n_gpus"] == 2 and d["collectives"] == "gloo" and d["scaling"] == "strong"
    c = d["config"]
    assert c["dp_size"] == 2 and c["params_per_step_all_ranks"] == 3147008
    assert set(d["kernels"]) == {"reduce_scatter", "allreduce_sumsq", "adamw_step", "all_gather"}
    # rank 0 per step: 2 packs + 1 accumulate call per micro-batch (+1 for the fused pass), the step, 2 unpacks
    assert d["gpu_launches"] == 3 * (2 * (2 + 1) + 1 + 1 + 2)
