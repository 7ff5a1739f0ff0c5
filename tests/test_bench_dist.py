"""bench.py's multi-rank plumbing on the CPU: two gloo ranks launched the way
torchrun launches the benchmark (RANK / WORLD_SIZE / MASTER_* from the
environment, rendezvous on 127.0.0.1). Each rank of the GPU arm replays the
whole step (replicas, no exchange), so the only collectives are the barrier
and the max over ranks of the step time; the reference arm runs on rank 0
alone and the other ranks exit without output."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_BODY = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
dist, rank, world = bench._dist()
assert world == 2 and rank == int(os.environ["RANK"])
bench._barrier(dist)
m = bench._max_over_ranks(dist, 1.5 + 2.0 * rank)
print(json.dumps({{"rank": rank, "max": m}}), flush=True)
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_max():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_BODY.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
    got = sorted(json.loads(o.strip().splitlines()[-1])["rank"] for o, _ in outs)
    assert got == [0, 1]
    for o, _ in outs:
        assert json.loads(o.strip().splitlines()[-1])["max"] == 3.5


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["steps"] == 2
    assert res["value"] > 0 and res["e2e"]["value"] == res["value"]
    assert res["cpu_baseline"]["kind"] == "oracle"


def test_gpus_flag_starts_the_ranks_itself():
    """--gpus 2 without a torchrun environment: the script starts two local
    ranks (rendezvous on 127.0.0.1) and prints one line with n_gpus 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["OMP_NUM_THREADS"] = "2"
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--gpus", "2",
           "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2
    assert res["config"]["parallelism"] == "replicas x2 (no exchange)"


def test_reference_arm_prints_the_workload_config_of_the_gpu_arm():
    """Both arms describe the workload with the same config dict."""
    sys.path.insert(0, ROOT)
    import bench
    from paged_gqa_decode_02_gb300 import workloads as W
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    cfg, _ = bench.workload_config(W.CONFIGS["tiny"](), "tiny", 1, 1)
    assert res["config"] == cfg
