"""The N > 1 path on the CPU: two ranks over gloo on 127.0.0.1.

Under torchrun every rank runs its own replica of the layer ("replicas only":
the layer is not sharded across GPUs, so the data path has no collective).
The one collective is the benchmark's timing reduction: every rank takes the
slowest rank's time, and the job's throughput is all ranks' tokens over that
time.  The reference arm runs on rank 0 alone; the other ranks exit 0 without
work."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys, datetime
import torch
import torch.distributed as dist
sys.path.insert(0, os.environ["BENCH_ROOT"])
import bench
rank, world, local = bench.dist_env()
dist.init_process_group("gloo", timeout=datetime.timedelta(seconds=60))
ms = [1.25, 3.5][rank]                       # rank 1 is the slow replica
slowest = bench.max_over_ranks(ms, world, "cpu")
value = bench.replica_throughput(world, 32, slowest)
dist.barrier()
print(json.dumps({"rank": rank, "world": world, "slowest": slowest, "value": value}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(**kw):
    env = dict(os.environ)
    env.update({k: str(v) for k, v in kw.items()})
    env["CUDA_VISIBLE_DEVICES"] = ""
    env.setdefault("OMP_NUM_THREADS", "2")
    return env


def test_two_gloo_ranks_take_the_slowest_replica():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], cwd=ROOT, stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True,
                              env=_env(RANK=r, LOCAL_RANK=r, WORLD_SIZE=2, MASTER_ADDR="127.0.0.1",
                                       MASTER_PORT=port, BENCH_ROOT=ROOT))
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for r, o in enumerate(outs):
        assert o["rank"] == r and o["world"] == 2
        assert o["slowest"] == 3.5                        # both ranks see the slowest rank's time
        assert o["value"] == 2 * 32 / 3.5e-3              # both replicas' tokens over that time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.0, 1, "cpu") == 2.0
    assert bench.replica_throughput(1, 32, 0.5) == 64000.0


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=_env())
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
