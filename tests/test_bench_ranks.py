"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks agree on the
max-over-ranks time and pass the barrier; the reference arm prints one line on
rank 0 and does no work on the other ranks."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    cpu = torch.device("cpu")
    bench.barrier(dist, cpu)
    t = bench.max_over_ranks(1.5 * (r + 1), dist, cpu)   # rank r "took" 1.5 (r + 1) ms
    bench.barrier(dist, cpu)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "max": t}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [g["rank"] for g in got] == [0, 1]
    assert all(g["world"] == 2 and g["max"] == 3.0 for g in got)


def _bench(rank, world, extra=()):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny", "--steps", "3", "--warmup", "3", *extra]
    return subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_quietly():
    p = _bench(rank=1, world=2, extra=("--gpus", "2"))
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    p = _bench(rank=0, world=1)
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
