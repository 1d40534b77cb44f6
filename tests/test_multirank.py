"""The bench's N > 1 host path on CPU: two gloo ranks, no GPU.

Every (batch, head) is independent, so ranks run replicas and exchange nothing
on the data path; what they share is a host barrier and the max over ranks of
the timed region.  These tests run that logic as two real processes.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
world, rank, local, pg = bench.dist_setup()
bench.barrier(pg)
t = bench.max_over_ranks(pg, 0.25 * (rank + 1))
bench.barrier(pg)
print(json.dumps({"rank": rank, "world": world, "local": local, "max": t}))
pg.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    return env


def test_two_gloo_ranks_agree_on_the_max_time():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", WORKER, ROOT], env=_env(r, 2, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    got = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda x: x["rank"])
    assert [g["rank"] for g in got] == [0, 1]
    assert all(g["world"] == 2 and g["max"] == 0.5 for g in got)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "3", "--warmup", "3", "--reference-budget", "2",
           "--workload", "tiny_causal_b1h4t256d64"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
