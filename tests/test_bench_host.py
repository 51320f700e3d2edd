"""Host-side logic of bench.py that needs no GPU: the algorithmic byte model, the
clock-sample parser, and the N>1 aggregation (max time, summed work over ranks)
run as two gloo ranks on the CPU."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes_per_element():
    n = 16384 * 6144
    b = bench.algorithmic_bytes(n)
    assert b["amax"] / n == pytest.approx(4.25)        # read 4 B, write 2 x 4 B / 32
    assert b["cast"] / n == pytest.approx(6.0625)      # read 4 B + 2 scale B / 32, write 2 B
    assert b["amax"] == 427_819_008 and b["cast"] == 610_271_232
    assert b["reduce_scales"] == b["reduce"] + n // 16
    ro = bench.algorithmic_bytes(n, colwise=False)
    assert ro["cast"] / n == pytest.approx(4 + 1 / 32 + 1)


def test_clock_summary_parser():
    c = bench.ClockSampler(0)
    c.out = ("0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active\n"
             "0, 1980, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
             "garbage line\n")
    s = c.summary()
    assert s["sm_mhz"] == pytest.approx(1972.5) and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.aggregate_over_ranks(1.0 + rank, 10.0 * (rank + 1), world)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_single_rank_aggregation_is_identity():
    assert bench.aggregate_over_ranks(0.5, 7.0, 1) == (0.5, 7.0)


def test_sharded_step_bytes():
    from mxfp8_master_weight_gb300 import driver
    specs = [driver.WeightSpec(64, 64, True), driver.WeightSpec(32, 64, False)]
    b = bench.sharded_step_bytes(specs, num_slots=2, packed_entries=1000)
    n0, n1 = 64 * 64, 32 * 64
    amax = n0 * 4 + 2 * n0 // 32 * 4 + n1 * 4 + n1 // 32 * 4
    cast = n0 * 4 + 2 * n0 // 32 + 2 * n0 + n1 * 4 + n1 // 32 + n1
    assert b == amax + cast + 2 * 1000 * 4 + 1000 * 4 + 1000
    ph = bench.sharded_phase_bytes(specs, num_slots=2, packed_entries=1000)
    assert ph == {"amax": amax, "reduce_scales": 2 * 1000 * 4 + 1000 * 4 + 1000, "cast": cast}
    assert sum(ph.values()) == b


def test_stats_and_kernel_digest():
    s = bench.stats([3.0, 1.0, 2.0, 10.0])
    assert s["median"] == 2.5 and s["mean"] == 4.0 and s["n"] == 4
    from mxfp8_master_weight_gb300 import build
    d = build.kernel_digest()
    assert len(d) == 64 and d != build.source_digest()


def test_cpu_all_cores_run_matches_single_core_bytes():
    """The all-cores oracle baseline splits whole 32-row bands over worker processes and
    accounts for exactly the bytes of the single-threaded run of the same rows."""
    rng = np.random.default_rng(0)
    rows = 96
    data = (rng.standard_normal(rows * bench.COLS) * 0.02).astype(np.float32)
    wall, b, used = bench.cpu_all_cores_run(data, rows, 2)
    _, b1 = bench.cpu_sample_run(data, 0, rows)
    assert used == 2 and b == b1 and wall > 0
    assert isinstance(bench.cpu_model(), str)


def test_nvfp4_algorithmic_bytes_per_element():
    n = 16384 * 6144
    b = bench.nvfp4_algorithmic_bytes(n)
    assert b["amax"] / n == pytest.approx(4.5)        # read 4 B, write 2 x 4 B / 16
    assert b["scales"] / n == pytest.approx(0.625)    # read 2 x 4 B / 16, write 2 B / 16
    assert b["cast"] / n == pytest.approx(5.125)      # read 4 B + 2 B / 16, write 2 x 0.5 B


def test_copy_bound_closed_forms():
    link = {"h2d_gbs": 200.0, "d2h_gbs": 100.0, "concurrent_h2d_gbs": 150.0, "concurrent_d2h_gbs": 50.0}
    # one direction only: that direction alone at its own rate
    assert bench.copy_bound_s(400e9, 0, link) == pytest.approx(2.0)
    assert bench.copy_bound_s(0, 300e9, link) == pytest.approx(3.0)
    # copy-out ends first: 50 GB at 50 GB/s (1 s, while 150 GB go in), then 250 GB alone at 200
    assert bench.copy_bound_s(400e9, 50e9, link) == pytest.approx(1.0 + 250 / 200)
    # copy-in ends first: 150 GB in 1 s (50 GB out meanwhile), then 50 GB out alone at 100
    assert bench.copy_bound_s(150e9, 100e9, link) == pytest.approx(1.0 + 0.5)
    # never below either direction alone, never above the two run one after the other
    for a, b in ((400e9, 200e9), (10e9, 300e9), (1e9, 1e9)):
        t = bench.copy_bound_s(a, b, link)
        assert max(a / 200e9, b / 100e9) - 1e-12 <= t <= a / 150e9 + b / 50e9 + 1e-12


def test_spread_percentiles():
    assert bench.spread([]) == {}
    s = bench.spread([float(v) for v in range(1, 21)])
    assert s == {"median": 10.5, "p10": 3.0, "p90": 19.0, "max": 20.0}
