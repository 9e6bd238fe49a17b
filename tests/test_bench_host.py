"""Host-side logic of bench.py that needs no GPU.

The multi-GPU bench runs independent replicas (weak scaling, no collective on the data path);
rank 0 reports the whole job as the units summed over ranks divided by the slowest rank's
elapsed time.  That aggregation is checked here with two gloo ranks on the CPU, and the byte
accounting helpers against their definitions.
"""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [0.25, 0.40][rank]
        units = [1.0e9, 3.0e9][rank]
        bench.barrier(world)
        out[rank] = bench.aggregate(elapsed, units, world)
    finally:
        dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    import torch.multiprocessing as mp
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        res = dict(out)
    # every rank sees the same whole-job numbers: slowest rank's time, all ranks' units
    assert res[0] == pytest.approx((0.40, 4.0e9))
    assert res[1] == pytest.approx((0.40, 4.0e9))


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(0.5, 123.0, 1) == (0.5, 123.0)


def test_byte_accounting():
    c, n = 128, 262_144
    u, split = 84_899, 518
    # step: p, m, v read + written, last_step read + written (DormancyDecay), gradient values and indices
    assert bench.step_bytes(u, c, n, True) == u * c * 24 + u * 16 + n * c * 4 + n * 8
    assert bench.step_bytes(u, c, n, False) == u * c * 24 + u * 8 + n * c * 4 + n * 8
    # row kernel: the rows it updates (not those finished by the combine kernels) and every gradient value
    rows = u - split
    assert bench.fused_kernel_bytes(u, split, c, n, True) == rows * c * 24 + rows * 16 + n * c * 4


def test_recorded_traffic_tracks_the_kernel_sources(monkeypatch):
    t = bench.recorded_traffic()
    assert t is None or t > 0
    monkeypatch.setattr(bench, "row_kernel_digest", lambda: "0" * 16)
    assert bench.recorded_traffic() is None
