"""The replica aggregation of bench.py under torch.distributed (gloo, world_size 2, CPU): every rank
streams the same bytes; the whole-job value is the total over ranks divided by the slowest rank's
time, which every rank learns through the all-gather."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = 1.0 + rank  # rank 1 is the slower replica
        times = bench.max_over_ranks(t, world)
        value, tmax = bench.aggregate(1e9, times)
        q.put((rank, times, value, tmax))
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, value, tmax in res:
        assert times == [1.0, 2.0]
        assert tmax == 2.0
        assert value == pytest.approx(2 * 1e9 / 2.0 / 1e9)  # 2 ranks x 1 GB over the slowest 2 s


def test_aggregate_single_rank():
    import bench
    v, t = bench.aggregate(17555292160, [0.0075])
    assert t == 0.0075 and v == pytest.approx(17555292160 / 0.0075 / 1e9)


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, env_extra=None):
    import subprocess
    import sys
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_the_contract_line():
    """The oracle arm (bench.py --impl reference) prints one JSON line with the GPU arm's metric and
    unit, the cpu_baseline it measured and an e2e object, on the host cores alone."""
    import json
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["impl"] == "reference"
    assert d["value"] > 0 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 runs the oracle arm; the others exit 0 without output."""
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "0"], {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_does_not_load_the_product_library():
    """The oracle arm times the fp64 oracle alone: its process maps oracle/liboracle.so and never
    libverify.so (the shapes come from the library-free geometry module)."""
    import subprocess
    import sys
    code = ("import sys, runpy; sys.argv = ['bench.py', '--impl', 'reference', '--steps', '1', '--warmup', '0', "
            "'--layers', '1']; runpy.run_path('bench.py', run_name='__main__'); "
            "maps = open('/proc/self/maps').read(); "
            "print('LIBVERIFY' if 'libverify' in maps else 'CLEAN', 'ORACLE' if 'liboracle' in maps else 'NO-ORACLE')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().splitlines()[-1] == "CLEAN ORACLE"
