"""The N > 1 path of bench.py on the CPU: two ranks over gloo (the GPU run uses NCCL the same
way). The path shards nothing (replicas: every rank quantizes its own tensor); the only
collective is the max of the timed region over ranks, and the reference arm runs on rank 0
alone. Both are checked here with world_size 2."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import argparse

    import torch.distributed as dist

    import bench
    args = argparse.Namespace(impl="ours", gpus=world, steps=1, warmup=3,
                              workload=bench.DEFAULT_WORKLOAD)
    w, r, _ = bench.dist_setup(args)
    bench.barrier(w)
    results[rank] = (w, r, bench.max_over_ranks(w, 1.5 + rank))
    # the reference arm: rank 0 alone does work; the others return at once
    if rank != 0:
        results[10 + rank] = bench.run_reference(argparse.Namespace(
            impl="reference", gpus=world, steps=1, warmup=3, workload=bench.DEFAULT_WORKLOAD), w, r)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_ranks_max_over_ranks_and_reference_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        assert results[0] == (2, 0, 2.5) and results[1] == (2, 1, 2.5)
        assert results[11] is None


def test_aggregate_value_counts_every_rank():
    import bench
    # two ranks of the same ideal bytes over the slowest rank's time
    assert bench.aggregate_gbs(1e9, 10, 2, 2.0) == pytest.approx(10.0)


def test_rotation_sets_cover_three_l2_capacities():
    import bench
    l2 = 126 << 20  # an L2 of 126 MiB
    for set_bytes in (1, 335_872, 104_857_600 + 2_097_152, 183_500_800, 419_430_400, 3 * l2):
        k = bench.rotation_sets(set_bytes, l2)
        assert k * set_bytes >= 3 * l2 and (k == 1 or (k - 1) * set_bytes < 3 * l2)
    assert bench.rotation_sets(419_430_400, l2) == 1      # inputs alone larger than L2
