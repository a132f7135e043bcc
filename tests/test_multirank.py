"""The bench's N > 1 path on the CPU: world-size-2 gloo ranks on 127.0.0.1.

Every rank runs the whole workload on its own GPU (independent sequences: no collective on
the data path), so the only multi-process logic is the control plane: rank identities from
the environment, the host barrier, the max of the timings over ranks and the whole-job rate
(all ranks' units over the slowest rank's time).  The reference arm under torchrun runs on
rank 0 alone and prints one line.  Nothing here touches a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    cp = bench.ControlPlane()
    try:
        cp.barrier()
        m = cp.max_over_ranks(times[rank])
        rate = bench.whole_job_rate(cp.world, 131072, m)
        q.put((rank, cp.rank, cp.world, m, rate))
    finally:
        cp.close()


@pytest.mark.parametrize("times", [(12.5, 40.0), (33.0, 7.25)])
def test_two_gloo_ranks_take_the_slowest(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slow = max(times)
    for rank, crank, cworld, m, rate in got:
        assert (crank, cworld) == (rank, 2)
        assert m == slow
        assert rate == pytest.approx(2 * 131072 / (slow / 1e3))


def test_single_process_has_no_collective():
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    code = ("import sys; sys.path.insert(0, %r); import bench; cp = bench.ControlPlane(); "
            "assert cp.world == 1 and cp.dist is None; assert cp.max_over_ranks(3.5) == 3.5; "
            "cp.barrier(); cp.close(); print('ok')" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("ok")


def test_reference_arm_under_torchrun():
    """`bench.py --impl reference` launched under torchrun with two ranks, as an N > 1 run
    is launched: rank 0 alone runs the oracle and prints one JSON line; the other rank exits
    0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-tokens", "16"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
