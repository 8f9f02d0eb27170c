"""The multi-GPU bench path is replicas only: every rank runs the suite on
its own GPU and rank 0 reports the whole job.  The aggregation runs here on
two gloo ranks over the CPU with made-up per-rank results."""
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
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = {"ms_per_step": 5.0 + rank, "value": 0.0, "gpu_launches": 160,
           "config": {"schedule_bytes_per_step": 10_000_000_000},
           "e2e": {"ms_per_step": 80.0 + 3 * rank, "value": 0.0, "unit": "GB/s",
                   "h2d_bytes_per_step": 100, "d2h_bytes_per_step": 200}}
    out = bench.combine_replicas(res, world)
    bench.barrier()
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump(out, f)
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_bytes(tmp_path):
    out_path = str(tmp_path / "line.json")
    mp.start_processes(_rank_main, args=(2, _free_port(), out_path), nprocs=2, join=True, start_method="spawn")
    out = json.load(open(out_path))
    assert out["n_gpus"] == 2
    assert out["ms_per_step"] == 6.0                  # max over ranks
    assert out["value"] == round(2e10 / 6.0e6, 1)     # both replicas' bytes
    assert out["e2e"]["ms_per_step"] == 83.0
    assert out["e2e"]["value"] == round(2e10 / 83.0e6, 1)
    assert out["e2e"]["h2d_bytes_per_step"] == 200 and out["e2e"]["d2h_bytes_per_step"] == 400
    assert out["gpu_launches"] == 320
