"""The benchmark's N > 1 host logic on CPU: two ranks over gloo.

`bench.py --gpus N` runs N independent replicas of the path (no data-path collective); the
only cross-rank steps are the barrier around the timed region and the whole-job aggregation
(max elapsed over ranks, units summed).  The reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys
import textwrap

from conftest import ROOT

WORKER = textwrap.dedent("""
    import json, os, sys
    sys.path.insert(0, os.environ["REPO"])
    import torch.distributed as dist
    import bench
    rank = int(os.environ["RANK"])
    dist.init_process_group("gloo")
    world, r, _ = bench.dist_env()
    assert (world, r) == (2, rank)
    bench.barrier(world)
    # rank 0 took 1.5 s for 10 units, rank 1 took 2.0 s for 30 units
    t, u = bench.aggregate(1.5 + 0.5 * rank, 10.0 + 20.0 * rank, world)
    bench.barrier(world)
    dist.destroy_process_group()
    print(json.dumps({"rank": rank, "t": t, "u": u}))
""")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code_or_args, world=2, timeout=240):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), REPO=str(ROOT),
                   CUDA_VISIBLE_DEVICES="")
        cmd = [sys.executable, "-c", code_or_args] if isinstance(code_or_args, str) \
            else [sys.executable] + code_or_args
        procs.append(subprocess.Popen(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_aggregate_and_barrier_two_ranks():
    outs = _launch(WORKER)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in res:
        assert r["t"] == 2.0          # the slowest rank's time
        assert r["u"] == 40.0         # every rank's units


def test_reference_arm_runs_on_rank0_only():
    args = ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
            "--config", "c1_whole_p2"]
    outs = _launch(args)
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    line = json.loads(lines0[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
