"""The multi-GPU path of bench.py is N independent replicas (the int4g path
needs no exchange).  Its host logic -- the barrier-bracketed timed region and
the job-wide aggregation (max step time over ranks, bytes of all ranks) --
runs here as two gloo ranks on CPU."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    import torch
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    # a rank's own line, as run_gpu returns it: rank r is the slower the larger r
    line = {"metric": bench.METRIC, "value": 0.0, "unit": "GB/s", "n_gpus": 1, "ms_per_step": 0.1 * (rank + 1),
            "config": {"workload": bench.WORKLOAD, "weight_bytes_per_step": 2.0e8, "parallelism": "single"},
            "e2e": {"value": 100.0 - 10.0 * rank, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}

    def max_over_ranks(v):
        t = torch.tensor([float(v)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    agg = bench.aggregate_replicas(line, world, max_over_ranks)
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump(agg, f)
    dist.destroy_process_group()


def test_two_gloo_replicas_aggregate(tmp_path):
    out = tmp_path / "agg.json"
    mp.start_processes(_rank_main, args=(2, _free_port(), str(out)), nprocs=2, join=True, start_method="spawn")
    agg = json.loads(out.read_text())
    assert agg["n_gpus"] == 2
    assert agg["ms_per_step"] == pytest.approx(0.2)                       # the slower rank
    assert agg["value"] == pytest.approx(2 * 2.0e8 / 0.2e-3 / 1e9, rel=1e-6)   # both ranks' bytes
    assert agg["e2e"]["value"] == pytest.approx(2 * 90.0)                 # 2 x the slower rank
    assert agg["config"]["parallelism"] == "replicas2"
