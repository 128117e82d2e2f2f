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


def test_reference_arm_json_line(monkeypatch, capsys):
    """Rank 0 of the reference arm (the CPU oracle, a bounded sample per step)
    prints one JSON line with the keys the benchmark contract names."""
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
