"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each with its own
per-rank time and bytes; the whole-job throughput uses all ranks' bytes over
the slowest rank's time (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    ms_local = 2.0 + rank            # rank 1 is the slower one
    ms, gbs = bench.aggregate(ms_local, 1e9)
    bench.barrier()
    out[rank] = (ms, gbs, bench.max_over_ranks(float(rank)))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, gbs, mx = res[rank]
        assert ms == pytest.approx(3.0)                    # max over ranks
        assert gbs == pytest.approx(2 * 1e9 / 3e-3 / 1e9)  # both ranks' bytes / slowest time
        assert mx == 1.0


def test_single_process_aggregation_is_identity():
    import bench
    ms, gbs = bench.aggregate(4.0, 2e9)
    assert ms == 4.0 and gbs == pytest.approx(2e9 / 4e-3 / 1e9)


def test_reference_arm_other_ranks_exit(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    assert capsys.readouterr().out == ""
