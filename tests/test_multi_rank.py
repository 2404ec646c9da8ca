"""The multi-process (N > 1) host path of bench.py, on CPU with the gloo backend.

Decode has no exchange step between GPUs: with N ranks each rank runs a full replica of the
workload, and the only collective is the one that takes the slowest rank's times.  These tests
run that reduction in two real gloo processes rendezvousing on 127.0.0.1, check the whole-job
aggregation, and check that the reference arm runs on rank 0 alone under torchrun.
"""
import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# One rank: joins a gloo group from the torchrun-style environment, reduces its own pair of
# times with bench.max_over_ranks and prints the result as JSON.
_RANK_SCRIPT = textwrap.dedent("""
    import json, os, sys
    sys.path.insert(0, {root!r})
    import torch.distributed as dist
    import bench
    rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = {values!r}[rank]
    got = bench.max_over_ranks(mine, world)
    dist.destroy_process_group()
    print(json.dumps({{"rank": rank, "got": got}}))
""")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    env = dict(os.environ)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    env.pop("CUDA_VISIBLE_DEVICES", None)
    return env


def _run_ranks(values, timeout=120):
    world = len(values)
    port = _free_port()
    script = _RANK_SCRIPT.format(root=ROOT, values=values)
    procs = [subprocess.Popen([sys.executable, "-c", script], env=_env(r, world, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(world)]
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=timeout)
            assert p.returncode == 0, err[-2000:]
            outs.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
                p.wait()
    return sorted(outs, key=lambda d: d["rank"])


def test_max_over_ranks_two_gloo_ranks_agree_on_the_slowest_times():
    # rank 0 is slower on the kernel clock, rank 1 on the end-to-end clock: both ranks must
    # report the element-wise maximum, not their own or the other rank's pair.
    outs = _run_ranks([[2.0, 1.5], [1.25, 5.0]])
    assert [o["rank"] for o in outs] == [0, 1]
    for o in outs:
        assert o["got"] == [2.0, 5.0]


def test_max_over_ranks_four_gloo_ranks():
    vals = [[1.0, 9.0, 3.0], [4.0, 2.0, 3.5], [0.5, 0.25, 8.0], [3.0, 1.0, 1.0]]
    outs = _run_ranks(vals)
    for o in outs:
        assert o["got"] == [4.0, 9.0, 8.0]


def test_max_over_ranks_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks([3, 1.5], 1) == [3.0, 1.5]


def test_replica_value_is_whole_job_throughput():
    import bench
    # one replica moving 1 GB in 1 ms is 1000 GB/s; N replicas in the same (slowest) time
    # move N times the bytes
    assert bench.replica_value(1e9, 1, 1.0) == pytest.approx(1000.0)
    assert bench.replica_value(1e9, 2, 1.0) == pytest.approx(2000.0)
    assert bench.replica_value(1e9, 8, 2.0) == pytest.approx(4000.0)


@pytest.mark.parametrize("workload", ["worked", "mla"])
def test_reference_arm_on_a_nonzero_rank_exits_quietly(workload):
    env = _env(1, 2, _free_port())
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", workload, "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    env = dict(os.environ)
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
           "--workload", "worked", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
