"""The multi-rank path of bench.py on CPU: two gloo ranks each build their own
replica of the workload (own seed, own sequences), then agree on the slowest
rank's time and the job's total bytes -- the only exchange the benchmark
makes (decode itself has none)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from paged_kv_decode_26_gb300 import workloads as wl
        seed = bench.rank_seed(2, rank)
        case = wl.make_case(2, seed=seed, S=3, lens=("uniform", 20, 90), H=2, Hk=2, D=64)
        kv, _ = wl.kv_bytes(case)
        fake_ms = 1.0 + 0.5 * rank
        ms, = bench.reduce_over_ranks([fake_ms], "max", dist, world, "cpu")
        total, = bench.reduce_over_ranks([kv], "sum", dist, world, "cpu")
        torch.save({"seed": seed, "kv": kv, "ms": ms, "total": total,
                    "value": bench.job_gbs(total, ms), "lens": case.context_lens.tolist()},
                   os.path.join(out_dir, f"r{rank}.pt"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r0, r1 = (torch.load(tmp_path / f"r{i}.pt") for i in range(world))
    assert r0["seed"] != r1["seed"]
    assert r0["lens"] != r1["lens"]                       # independent sequences per rank
    assert r0["ms"] == r1["ms"] == 1.5                    # the slowest rank's time
    assert r0["total"] == r1["total"] == r0["kv"] + r1["kv"]
    assert r0["value"] == pytest.approx((r0["kv"] + r1["kv"]) / 1.5e-3 / 1e9)


def test_single_rank_helpers():
    import bench
    assert bench.reduce_over_ranks([3.0, 4.0], "max", None, 1, "cpu") == [3.0, 4.0]
    assert bench.job_gbs(2e9, 1000.0) == pytest.approx(2.0)
    assert bench.rank_seed(2, 0) == 1 and bench.rank_seed(2, 1) != bench.rank_seed(2, 0)
