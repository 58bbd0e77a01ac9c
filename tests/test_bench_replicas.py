"""The N > 1 host path of bench.py on CPU: world size 2 over gloo.  Each rank
is an independent replica; the job's throughput is the units of all ranks
over the slowest rank's time, with barriers on both sides."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.dist_init(w, "gloo")
    bench.barrier()
    elapsed = 1.0 + rank          # rank 1 is the slow one
    units = 10.0 * (rank + 1)     # 10 + 20 units in total
    value, t = bench.aggregate(elapsed, units)
    out[rank] = (value, t, bench.reduce_max(float(rank)), bench.reduce_sum(1.0))
    bench.barrier()
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replicas_aggregate_over_gloo():
    world = 2
    port = _free_port()
    # spawn, not fork: the test process may already run threads (the oracle's OpenMP pool)
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        value, t, mx, n = res[rank]
        assert t == pytest.approx(2.0)
        assert value == pytest.approx(30.0 / 2.0)
        assert mx == 1.0 and n == 2.0


def test_single_process_aggregate_is_local():
    import bench
    value, t = bench.aggregate(2.0, 8.0)
    assert (value, t) == (4.0, 2.0)


def test_bench_arguments_default_to_one_gpu():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.warmup >= 3 and a.steps >= 1


def test_reference_arm_under_torchrun_prints_once():
    """The reference arm launched like the scaling runs (torchrun, two ranks
    on this host): rank 0 alone times the oracle and prints one line; the
    other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    from pathlib import Path
    root = Path(__file__).resolve().parent.parent
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           str(root / "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
