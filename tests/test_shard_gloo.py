"""Multi-rank host logic on CPU with the gloo backend, world size 2 (and 3):
frame sharding covers every frame exactly once, per-rank blocks gather back
in order, and timings reduce to the maximum over ranks."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from residual_vector_quantisation_gb300.shard import frame_range, gather_rows, reduce_max


def test_frame_range_partitions_exactly():
    for n in (0, 1, 7, 250, 192000, 192001):
        for world in (1, 2, 3, 8):
            covered = []
            sizes = []
            for r in range(world):
                a, b = frame_range(n, r, world)
                covered.extend(range(a, b))
                sizes.append(b - a)
            assert covered == list(range(n))
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        frame_range(10, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n_total, result_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        a, b = frame_range(n_total, rank, world)
        # stand-in for this rank's encode output: row i carries its global frame index
        local = torch.arange(a, b, dtype=torch.int32)[:, None].repeat(1, 4) * 10 + torch.arange(4, dtype=torch.int32)
        full = gather_rows(local, n_total)
        t = reduce_max(0.5 + rank)
        dist.barrier()
        result_q.put((rank, full.shape[0], bool(torch.equal(full[:, 0], torch.arange(n_total, dtype=torch.int32) * 10)),
                      t))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n_total", [(2, 101), (3, 1000)])
def test_gloo_gather_and_reduce(world, n_total):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n_total, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rows, ordered, t in results:
        assert rows == n_total and ordered
        assert t == 0.5 + (world - 1)
