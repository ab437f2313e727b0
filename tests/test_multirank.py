"""The multi-rank side of bench.py on the CPU: two gloo ranks (the layer has
no exchange step, so N GPUs run N independent replicas and only the timing
is reduced across ranks) and the reference arm under two ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + 0.5 * rank, dist, "cpu")  # the ranks' step times differ
        q.put((rank, ms, bench.job_tokens_per_s(world, 64, ms)))
    finally:
        dist.destroy_process_group()


def test_timing_is_the_slowest_ranks_and_value_counts_every_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 1.5  # max over ranks, on every rank
        assert value == pytest.approx(2 * 64 / 1.5e-3)


def test_single_rank_has_no_reduction():
    import bench
    assert bench.max_over_ranks(2.0, None, "cpu") == 2.0
    assert bench.job_tokens_per_s(1, 64, 2.0) == pytest.approx(32000.0)


def test_reference_arm_prints_on_rank_zero_only():
    outs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(_free_port()))
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                            "--gpus", "2", "--steps", "3", "--warmup", "3"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip())
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
