"""The N > 1 host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The hot path shards into independent replicas (channels never interact), so
the only multi-rank logic is the timing reduction: the job's step time is the
slowest rank's, and the whole-job value counts every rank's state updates.
The reference arm runs on rank 0 only.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")      # rank 1 is slower
        value = bench.job_value(1000, world, slowest)
        # the reference arm prints on rank 0 only
        out = io.StringIO()
        with redirect_stdout(out):
            bench.run_reference(_args(), rank, world)
        q.put((rank, slowest, value, out.getvalue()))
    finally:
        dist.destroy_process_group()


def _args():
    class A:
        pass
    a = A()
    a.workload, a.small, a.steps, a.warmup = "tiny_fp32_b1_d16_l256_n16", False, 1, 0
    return a


@pytest.mark.timeout(300)
def test_two_ranks_max_time_and_reference_on_rank0():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, slowest, value, out = q.get(timeout=240)
        res[rank] = (slowest, value, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        slowest, value, _ = res[rank]
        assert slowest == 15.0                            # every rank sees the slowest rank's time
        assert value == pytest.approx(1000 * world / 15e-3)
    line = json.loads(res[0][2].strip())
    assert line["impl"] == "reference" and line["n_gpus"] == world
    assert line["config"]["parallelism"] == "replicas x2"
    assert res[1][2] == ""                                # rank 1 prints nothing
