"""The multi-rank (N > 1) host path of bench.py on CPU: two gloo ranks.

Sequences are independent units, so N ranks run N replicas with no
collective on the data path; what the ranks share is the barrier around the
timed region and the maximum of the per-rank times.  These tests run that
logic as world_size-2 process groups on the host (gloo, 127.0.0.1)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, ws, local = bench._dist()
    assert (r, ws, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench._barrier(ws)
    # each rank's own time; every rank must see the slowest one
    got = bench._max_over_ranks(1.5 + rank, ws)
    out.put((rank, got))
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    assert res == [(0, 2.5), (1, 2.5)]


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched as the driver launches N = 2:
    rank 0 alone runs the oracle and prints one JSON line; rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1", "--config", "llada_single"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
