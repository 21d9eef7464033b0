"""Host-side logic of bench.py: argument defaults, weak-scaling throughput, and the max-over-ranks
timing reduction run as two gloo ranks on the CPU (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as tmp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    assert (r, w) == (rank, world)
    t = bench.dist_max(world, 10.0 + rank, "cpu")        # rank 1 is the slow one
    bench.dist_barrier(world)
    out[rank] = (t, bench.job_throughput(world, 1024, 10, t))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_with_two_gloo_ranks():
    port = _free_port()
    mgr = tmp.Manager()
    out = mgr.dict()
    tmp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0][0] == out[1][0] == 11.0
    # 2 ranks x 1024 queries x 10 steps in 11 ms
    assert out[0][1] == pytest.approx(2 * 1024 * 10 / 0.011)


def test_defaults_are_the_96k_workload():
    import bench
    a = bench.parse_args([])
    assert a.workload == "llama8b_n96k_32layers" and a.gpus == 1 and a.warmup >= 3
    assert bench.job_throughput(1, 1024, 5, 1000.0) == pytest.approx(5120.0)


def test_reference_arm_prints_the_contract_line():
    # the oracle arm on the smallest workload: one JSON line with the keys the driver reads
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_f32_n4096", "--steps", "1", "--warmup", "1",
                          "--cpu-seconds", "1"], capture_output=True, text=True, timeout=300,
                         cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "queries/s"
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config"):
        assert key in line, key
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"]
