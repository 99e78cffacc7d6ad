"""The C ABI used from a plain C program (tests/c_abi_step.c): no Python, no torch
on the call path.  The host-only plan queries run on CPU; the full local step
runs on a GPU and is checked against the oracle."""
import os
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NUMELS = [1000, 7, 4096, 33, 16385]
NO_DECAY = [0, 1, 0, 1, 0]
DP, RANK = 3, 1


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    from zero_sharded_mixed_local_gb300 import build
    lib = build.build_library()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path_factory.mktemp("cabi") / "c_abi_step")
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "c_abi_step.c"), "-o", exe, "-L", libdir, "-lzero1",
           "-Wl,-rpath," + libdir, "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_plan_from_c_matches_the_oracle(program):
    out = subprocess.run([program, "plan"], check=True, capture_output=True, text=True).stdout.splitlines()
    start, count, local = oracle.plan(NUMELS, DP, RANK)
    head = out[0].split()
    assert int(head[1]) == sum(NUMELS) and int(head[3]) == local
    for i, line in enumerate(out[1:]):
        f = line.split()
        assert int(f[3]) == start[i] and int(f[5]) == count[i] and int(f[7]) % 8 == 0


def _inputs(n, offsets, counts):
    """The C program's deterministic inputs (grad_bits, master_val) at the shard positions."""
    g = np.zeros(n, np.uint16)
    p = np.zeros(n, np.float32)
    for o, c in zip(offsets, counts):
        j = np.arange(o, o + c, dtype=np.int64)
        g[o:o + c] = (0x3a00 + (j * 37) % 512 - 256 + np.where(j & 1, 0x8000, 0)).astype(np.uint16)
        p[o:o + c] = ((j * 13) % 200 - 100).astype(np.float32) * np.float32(1e-4)
    return g, p


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["step", "list", "onecall"])
def test_step_from_c_matches_the_oracle(program, tmp_path, mode):
    """The arena calls, the tensor-list calls on one cudaMalloc per tensor shard, and the whole
    step as one zero1_local_step call."""
    outp = str(tmp_path / "out.bin")
    r = subprocess.run([program, mode, outp], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lines = subprocess.run([program, "plan"], check=True, capture_output=True, text=True).stdout.splitlines()
    n = int(lines[0].split()[5])
    offs = [int(l.split()[7]) for l in lines[1:]]
    cnts = [int(l.split()[5]) for l in lines[1:]]
    raw = open(outp, "rb").read()
    grad, master, m, v = [np.frombuffer(raw, np.float32, n, 4 * n * k) for k in range(4)]
    w = np.frombuffer(raw, np.uint16, n, 16 * n)
    sumsq = np.frombuffer(raw, np.float64, 1, 18 * n)[0]

    g_bits, p0 = _inputs(n, offs, cnts)
    G = np.zeros(n, np.float32)
    oracle.accumulate(G, g_bits, overwrite=True)
    assert np.array_equal(grad.view(np.uint32), G.view(np.uint32))
    ref = oracle.sumsq(G)
    assert abs(sumsq - ref) <= 1e-12 * ref
    ok, norm, coef = oracle.clip_coef(ref, 1.0)
    # arena order: decayed tensors (0, 2, 4) then the excluded ones (1, 3), padding included
    group1 = min(o for o, nd in zip(offs, NO_DECAY) if nd)
    P, M, V = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    hp = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    oracle.adamw(P, M, V, G, [group1, n - group1], [0, 1], hp, 1, coef)
    for a, b in ((master, P), (m, M), (v, V)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.array_equal(w, oracle.bf16_rne(P))
