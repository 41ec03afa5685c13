"""Host logic of bench.py on CPU: the max-over-ranks timing reduction with two
gloo ranks, the environment parsing, and the JSON fields of the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    bench.barrier()
    got = bench.reduce_max(10.0 + 5.0 * rank)
    dist.destroy_process_group()
    q.put((rank, ws, r, local, got))


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 0, 0, 15.0), (1, 2, 1, 1, 15.0)]


def test_reduce_max_without_process_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5) == 3.5


@pytest.mark.slow
def test_reference_arm_prints_contract_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--steps", "3",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_gpus_flag_launches_its_ranks():
    """A plain `bench.py --gpus 2` (no WORLD_SIZE) starts two ranks itself;
    they meet over gloo, rank 0 alone prints the line and reports both."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_PORT")}
    env["OMP_NUM_THREADS"] = "1"
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def test_gpus_flag_must_match_the_launched_world():
    env = dict(os.environ, RANK="0", WORLD_SIZE="2")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--gpus", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode != 0 and "WORLD_SIZE=2" in res.stderr


def test_both_arms_describe_the_workload_with_the_same_config():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    for name in workloads.CONFIGS:
        w = workloads.get(name)
        c = bench.config_of(w)
        assert c["workload"].startswith(name + ": N=%d E=%d K=%d R=%d H=%d" % (w.N, w.E, w.K, w.R, w.H))
        assert ("flushed" in c["l2"]) == (name == "tiny")


def test_default_workload_is_the_large_one():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.build_parser().parse_args([])
    assert args.config == "large" and args.gpus == 1 and args.impl == "ours"
