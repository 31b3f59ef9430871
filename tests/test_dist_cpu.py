"""The multi-process path of bench.py on CPU: two `gloo` ranks (world_size 2) exercise the
barrier and the max-over-ranks timing reduction, and the reference arm under torchrun,
where rank 0 alone runs and prints one JSON line and the other rank exits 0."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init(use_cuda=False)
    d.barrier()
    v = d.max(1.5 * (rank + 1))            # each rank's own "time"; all must see the largest
    d.barrier()
    q.put((rank, v))
    d.pg.destroy_process_group()


def test_dist_barrier_and_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 3.0, 1: 3.0}


def test_single_process_dist_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    if d.world != 1:
        pytest.skip("running under a launcher")
    d.init(use_cuda=False)
    d.barrier()
    assert d.max(2.5) == 2.5


@pytest.mark.timeout(600)
def test_reference_arm_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
