"""The N > 1 path on the CPU: two ranks over gloo (127.0.0.1).

The work shards by request (each rank decodes its own batch; no collective in
the data path), so what runs across ranks is the timing: a barrier and the
maximum of the ranks' times, which bench.py reports. Tested here: that
maximum, the per-rank workloads (same shapes, different seeds), and the
benchmark's reference arm launched with torch.distributed.run on two ranks
(rank 0 alone runs the CPU oracle and prints one JSON line; rank 1 exits 0).
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
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 1.5 + 2.0 * rank
        got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        wl = bench.make_workload("cfg2", 4, rank)
        out.put((rank, got, wl.seed, wl.seq_lens.tolist(), wl.q_heads, wl.kv_heads))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_per_rank_workloads():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, s0, l0, hq0, hk0), (r1, m1, s1, l1, hq1, hk1) = res
    assert m0 == m1 == 3.5                 # both ranks see the slowest rank's time
    assert s0 != s1 and l0 != l1           # each rank serves its own requests
    assert (hq0, hk0) == (hq1, hk1) and len(l0) == len(l1) == 4


def test_max_over_ranks_without_a_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25, None, "cpu") == 2.25


@pytest.mark.timeout(600)
def test_reference_arm_on_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "cfg1", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1                 # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
