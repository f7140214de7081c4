"""Multi-GPU layout is replicas only: each rank runs its own batch with no
data-path collective; the benchmark only reduces its timings.  The host-side
glue (rank setup, max-over-ranks, whole-job aggregation) runs here as two
gloo ranks on the CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world), "KB_DIST_BACKEND": "gloo"})
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # rank r took (r + 1) * 10 ms for the same per-rank work of 1e12 FLOPs
    t_max = bench.reduce_max((rank + 1) * 0.010, w)
    value = bench.aggregate(1e12, w, t_max)
    out[rank] = (t_max, value)
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_aggregate():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        t_max, value = out[rank]
        assert t_max == pytest.approx(0.020)
        assert value == pytest.approx(2 * 1e12 / 0.020)     # whole-job units / slowest rank's time


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup(1) == (0, 1, 0)
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate(10.0, 1, 2.0) == 5.0


def test_multi_gpu_flag_requires_a_launcher(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    with pytest.raises(SystemExit):
        bench.dist_setup(2)


def test_roofline_units():
    assert bench.prefill_flops(1, 16384) == 4 * 32 * 128 * 16384 * 16385 // 2
    assert bench.decode_bytes(16, 8192) == 2 * 16 * 8 * 8192 * 128 * 2 + 2 * 16 * 32 * 128 * 2
