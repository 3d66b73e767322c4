"""The N>1 benchmark path on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own replica of the workload (tokens are independent, so
the layer needs no collective on the data path); the job's value is the
tokens of all ranks over the slowest rank's timed seconds.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, seconds, units, out_q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    value, max_s, total = bench.aggregate(seconds[rank], units[rank], world, dist, "cpu")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    ref_line = bench.run_reference(args, bench.synth.small_config("mr", 64, 64, 64, 4, 2, "f32")) \
        if rank != 0 else "skipped-on-rank0"
    out_q.put((rank, value, max_s, total, ref_line))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_aggregate_and_reference_rank_split():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    seconds, units = [1.5, 2.0], [8192.0, 8192.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, seconds, units, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, max_s, total, ref_line in res:
        assert max_s == 2.0 and total == 16384.0
        assert abs(value - 16384.0 / 2.0) < 1e-9
        if rank == 1:
            assert ref_line is None  # the reference arm runs on rank 0 only


def test_single_rank_aggregate():
    import bench

    v, s, u = bench.aggregate(0.5, 1000.0, 1)
    assert (v, s, u) == (2000.0, 0.5, 1000.0)
