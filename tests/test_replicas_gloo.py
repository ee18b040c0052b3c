"""The multi-GPU path of the bench is N independent replicas with no
collective on the data path: the job's step time is the slowest replica's
(max over ranks) and the whole-job rate adds the replicas' rates. Checked
with two gloo ranks on the CPU."""
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


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        step_ms = [0.25, 0.31][rank]                        # the second replica is slower
        got = bench.max_over_ranks(step_ms, world, torch.device("cpu"))
        dist.barrier()
        q.put((rank, got, bench.replica_aggregate(got, world)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_step_and_the_summed_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, agg in out:
        assert got == pytest.approx(0.31)                    # max over ranks, on every rank
        assert agg["steps_per_s"] == pytest.approx(2 * 1e3 / 0.31, rel=1e-3)


def test_one_rank_reports_its_own_time():
    import bench
    assert bench.max_over_ranks(0.42, 1, torch.device("cpu")) == pytest.approx(0.42)
    assert bench.replica_aggregate(0.5, 1)["steps_per_s"] == pytest.approx(2000.0)


def test_decode_roofline_picks_the_binding_peak():
    """The decode line reports the roofline whose time is the larger: bytes over
    the HBM peak, or flops over the bf16 tensor peak."""
    import bench
    pk = {"hbm_gbs": 6480.8, "bf16_tflops": 1749.2}
    # Two queries over an fp8 cache: 584 GFLOP against 747 MB is tensor-bound.
    r = bench.decode_roofline(746_717_184, 584_079_900_672, 878.1, 686.88, pk, "measured", None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(686.88 / 1749.2, abs=1e-4)
    assert r["hbm_frac"] == pytest.approx(878.1 / 6480.8, abs=1e-4)
    # One query over a bf16 cache: 242 FLOP per byte is below the ridge.
    r = bench.decode_roofline(686_055_680, 686_055_680 * 242, 3400.0, 820.0, pk, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(3400.0 / 6480.8, abs=1e-4)
