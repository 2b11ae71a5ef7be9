"""The benchmark's multi-rank logic on CPU: world size 2 over gloo.

Tokens are independent, so every rank runs its own copy of the layer on its
own tokens (weak scaling) and the ranks exchange nothing in the data path; the
only communication is a barrier around the timed region and a MAX reduction of
the elapsed times.  These tests run that host logic with two processes.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier(world)
        # each rank's own elapsed ms and e2e seconds; every rank must see the maxima
        mine = [10.0 + 5.0 * rank, 3.0 - rank]
        got = bench.reduce_max(world, mine, torch.device("cpu"))
        value = bench.job_throughput(T=64, steps=100, world=world, elapsed_ms=got[0])
        q.put((rank, got, value))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, got, value in res:
        assert got == [15.0, 3.0], (rank, got)
        # 2 ranks x 100 steps x 64 tokens in the slowest rank's 15 ms
        assert value == pytest.approx(2 * 100 * 64 / 15e-3)


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1, [1.0, 2.0], torch.device("cpu")) == [1.0, 2.0]
    bench.barrier(1)
    assert bench.job_throughput(1, 1000, 1, 100.0) == pytest.approx(1e4)


def test_reference_arm_under_torchrun():
    """Two ranks of the reference arm: rank 0 alone prints one JSON line; rank 1 exits 0 without work."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny", "--gpus", "2",
           "--steps", "3", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["steps"] == 3
    assert j["value"] > 0 and j["e2e"]["h2d_bytes_per_step"] == 0
    assert j["cpu_baseline"]["kind"] == "oracle"


def test_bench_arguments_and_bytes():
    """Argument forms the benchmark accepts, and the algorithmic bytes of a layer step against the
    per-expert figure (3 d f int4 weights + 3 d f / 32 fp32 scales) and the router's weights."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    a = bench.parse_args([])
    assert (a.workload, a.mode, a.gpus, a.impl) == ("decode", "workload", 1, "ours")
    for wl in ("decode", "batched_decode", "prefill", "stack", "tiny"):
        assert bench.parse_args(["--workload", wl]).workload == wl
    assert bench.parse_args(["--mode", "prefill"]).mode == "prefill"
    with pytest.raises(SystemExit):
        bench.parse_args(["--workload", "nope"])
    # the FFN path of a single-layer workload: its own unless forced
    for wl, own in (("decode", "decode"), ("batched_decode", "decode"), ("prefill", "prefill")):
        assert bench.path_for(bench.parse_args([]), wl) == own
        for forced in ("decode", "prefill", "hybrid"):
            assert bench.path_for(bench.parse_args(["--mode", forced]), wl) == forced
    sh = workloads.WORKLOADS["decode"]
    b = bench.layer_bytes(sh, n_uniq=8)
    assert b["expert_block"] == 23_592_960
    assert b["ffn"] == 9 * 23_592_960 and b["nibbles"] == 9 * 18_874_368
    assert b["layer"] == b["ffn"] + 256 * 6144 * 4 + 256 * 4 + 2 * 1 * 6144 * 4


def test_kernel_source_hash_and_traffic_record():
    """The traffic record is used only while its hash matches the kernel sources."""
    sys.path.insert(0, ROOT)
    import bench
    h = bench.kernel_source_hash(ROOT)
    assert len(h) == 16 and h == bench.kernel_source_hash(ROOT)
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    assert "ffn" in rec
    for key in rec:
        got = bench.ncu_traffic(ROOT, key)
        assert got == (rec[key]["dram_bytes_per_launch"] if rec[key]["source_hash"] == h else None)
    assert bench.ncu_traffic(ROOT, "no_such_workload") is None
    # keyed to the FFN kernels' own sources: every listed file exists, and a change to one of them
    # (simulated on a copy of the tree) changes the hash
    import shutil
    import tempfile
    with tempfile.TemporaryDirectory() as tmp:
        csrc = os.path.join(tmp, "int4_routed_expert_sigmoid_gb300", "csrc")
        shutil.copytree(os.path.join(ROOT, "int4_routed_expert_sigmoid_gb300", "csrc"), csrc)
        assert bench.kernel_source_hash(tmp) == h
        with open(os.path.join(csrc, bench.FFN_SOURCES[0]), "a") as fh:
            fh.write("\n")
        assert bench.kernel_source_hash(tmp) != h
