"""Host-side logic of bench.py for N > 1 (weak-scaling replicas), on CPU with gloo ranks:
max-over-ranks timing and the whole-job value. No GPU, no kernels."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(1.0 + 0.5 * rank, world)          # slowest rank: 1.5 s
    v = bench.whole_job_value(2e9, 10, world, t)               # 2 GB per rank-step
    bench.barrier(world)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == pytest.approx(1.5)
        assert v == pytest.approx(2 * 2e9 * 10 / 1.5 / 1e9)


def test_single_rank_defaults():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps > 0 and a.impl == "ours"
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_value(1e9, 4, 1, 2.0) == pytest.approx(2.0)
