"""The bench's multi-rank host logic on CPU: two ranks over gloo.

Under torchrun every GPU runs its own batch (replicas, no data exchange); the
ranks meet only to take the slowest rank's time, and the whole-job rate counts
every rank's steps over that time. The reference arm runs on rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = """
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", rank=rank, world_size=world)
w = bench.rank_workload("batched", rank, world)
seeds = [None] * world
dist.all_gather_object(seeds, w.seed)
t = bench.max_over_ranks(1.0 + 0.5 * rank, world)       # a rank-dependent elapsed time
print(json.dumps(dict(rank=rank, seeds=seeds, t=t, rate=bench.whole_job_rate(world, 10, t))))
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time_and_run_distinct_batches():
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["t"] == 1.5                          # the slower rank's time, on both ranks
        assert o["rate"] == pytest.approx(2 * 10 / 1.5)
        assert len(set(o["seeds"])) == 2              # each rank its own batch


def test_one_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_rate(1, 7, 0.5) == 14.0
    assert bench.rank_workload("batched", 0, 1).seed == bench.rank_workload("batched", 5, 1).seed


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--config", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_line_carries_the_contract_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--config", "tiny"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    sys.path.insert(0, ROOT)
    import bench
    import ddtree_synth as S
    w = S.config("tiny")
    assert line["config"]["workload"] == "tiny" and line["config"]["global_batch"] == w.B
    assert line["config"]["seq_len"] == bench.mean_context(w) == 256   # the tiny workload's fixed context
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == (os.cpu_count() or 1) and cb["nproc"] == os.cpu_count()
    assert cb["cpu_model"]
    assert line["e2e"]["value"] == line["value"]
    # every reported step is a full oracle step that ran inside the command
    assert line["ms_per_step"] * (line["steps"] + line["warmup"]) / 1e3 <= line["wall_s"]
