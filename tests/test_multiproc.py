"""Multi-process host logic, world size 2 over gloo on 127.0.0.1 (no GPU).

The hot path shards as independent replicas: every rank owns its sequences, kv heads and
edges, and no collective touches the data. What spans ranks is the timing protocol of
`bench.py` (a barrier on both sides of the timed region and the maximum of the per-rank
step times, so the job is as slow as its slowest replica) and the reference arm, which
rank 0 alone runs and prints while the other ranks leave without work.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def rank_env(rank, world, port):
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
               WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    return env


def run_ranks(script, world, timeout=180):
    port = free_port()
    procs = [subprocess.Popen([sys.executable, "-c", script], env=rank_env(r, world, port),
                              cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True) for r in range(world)]
    out = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        out.append((p.returncode, o, e))
    return out


TIMING = r"""
import json
import bench
world, rank, _ = bench.dist_setup(2)
bench.barrier(world)
# per-rank step times: rank 0 takes 1.5 ms, rank 1 takes 2.5 ms
slowest = bench.max_over_ranks(1.5 + rank, world)
bench.barrier(world)
print(json.dumps({"rank": rank, "world": world, "slowest": slowest}))
import torch.distributed as dist
dist.destroy_process_group()
"""


def test_barrier_and_max_over_ranks_over_gloo():
    res = run_ranks(TIMING, 2)
    for rc, _, err in res:
        assert rc == 0, err[-2000:]
    lines = [json.loads(o.strip().splitlines()[-1]) for _, o, _ in res]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    assert all(d["world"] == 2 for d in lines)
    # every rank reports the slowest replica's time
    assert all(d["slowest"] == 2.5 for d in lines)


SINGLE = r"""
import json
import bench
world, rank, _ = bench.dist_setup(1)
print(json.dumps({"world": world, "rank": rank, "max": bench.max_over_ranks(3.25, world)}))
"""


def test_single_rank_needs_no_process_group():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    p = subprocess.run([sys.executable, "-c", SINGLE], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr[-2000:]
    assert json.loads(p.stdout.strip().splitlines()[-1]) == {"world": 1, "rank": 0, "max": 3.25}


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--cpu-seconds", "0.3", "--workload", "append_prompt"]
    p = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"]["workload"] == "append_prompt"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
