"""Host logic of bench.py, on the CPU: the whole-job value, the max over
ranks with two gloo ranks (the N > 1 path), the clock-record parser, the
oracle sample and the profile-summary lookup."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench


def test_job_value_sums_ranks_over_slowest():
    assert bench.job_value(1e12, 10, 1, 10.0) == pytest.approx(1.0)
    assert bench.job_value(1e12, 10, 4, 10.0) == pytest.approx(4.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    bench.barrier(world)
    m = bench.reduce_max(1.5 + rank, world)
    q.put((rank, m))
    bench.barrier(world)
    dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_reduce_max_single_rank_is_identity():
    assert bench.reduce_max(3.25, 1) == 3.25


def test_clock_parser():
    text = ("1965, 2070, 1100.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "1980, 2070, 1200.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "garbage line\n"
            "2010, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    r = bench.ClockSampler.parse(text)
    assert r["sm_mhz"] == 1980 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"] and r["samples"] == 3
    assert bench.ClockSampler.parse("") is None


def test_sample_rows_and_flops():
    rows = bench.sample_rows(8192, 100, 3)
    assert rows.size == 100 and rows.min() >= 0 and rows.max() < 8192
    assert not np.array_equal(rows, bench.sample_rows(8192, 100, 4))
    assert bench.oracle_rows_flops([0, 9], 16, 64, True) == (1 + 10) * 12 * 64
    assert bench.oracle_rows_flops([0, 9], 16, 64, False) == 2 * 16 * 12 * 64


def test_profiled_traffic_requires_matching_kernel(tmp_path, monkeypatch):
    f = tmp_path / "p.md"
    f.write_text(f"workload: b2h16t8192\nkernel_source_sha256: {bench.kernel_source_hash()}\n"
                 "traffic_bytes_per_launch: 1.5e9\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(f))
    assert bench.profiled_traffic("b2h16t8192") == 1.5e9
    assert bench.profiled_traffic("b4h16t2048") is None
    f.write_text("workload: b2h16t8192\nkernel_source_sha256: 0000\ntraffic_bytes_per_launch: 1.5e9\n")
    assert bench.profiled_traffic("b2h16t8192") is None


def test_headline_flops_count():
    w = bench.W.WORKLOADS["b2h16t8192"]
    assert w.flops == 2 * 16 * (8192 * 8193 // 2) * 12 * 64
    assert abs(w.flops / 1e9 - 824.734) < 1e-3


def test_l2_flush_is_named_in_config():
    w = bench.W.WORKLOADS["b2h16t8192"]
    assert "then a 256 MiB read" in bench.config_of(w, 0.5)["l2"]
    assert "then a 256 MiB read" in bench.config_of(w, 0.5, "write-read")["l2"]
    only_write = bench.config_of(w, 0.5, "write")["l2"]
    assert "256 MiB write" in only_write and "read" not in only_write


def test_gpus_flag_must_match_the_ranks(monkeypatch):
    # one process cannot stand in for N GPUs: without a launcher --gpus 2
    # fails loudly instead of running one replica
    for var in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert e.value.code != 0
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "0"])
    # a launcher that started a different number of ranks than --gpus says
    monkeypatch.setenv("WORLD_SIZE", "4")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "2", "--impl", "reference"])
    bench.check_world(1, 1)
    bench.check_world(2, 2)


def test_clock_scaled_peak():
    r = bench.clock_peak(1500.0, {"sm_mhz": 2000.0}, 152)
    assert r["peak"] == pytest.approx(152 * 2000e6 * 8192 / 1e12)
    assert r["frac"] == pytest.approx(1500.0 / r["peak"])
    assert bench.clock_peak(1500.0, None, 152) is None


def test_wait_profile_summary_shares():
    # [role][total, q, k, v, item_start, tensor, epilogue, peer]
    z5 = [0] * 10
    raw = ([1000, 0, 0, 0, 100, 500, 0, 100, 0, 0, 0, 0, 0] + z5 +            # producer
           [2000, 100, 200, 200, 0, 0, 0, 700, 900, 3, 400, 2, 150] + z5 +    # MMA issuers
           [8000, 0, 0, 0, 400, 1200, 400, 400, 0, 0, 0, 0, 0,                # softmax warps
            300, 900, 200, 10, 2, 60, 40, 30, 20, 10])
    spans = [1000, 5000, 1200, 9000, 0, 0]
    s = bench.wait_profile_summary(raw, spans)
    assert s["tma_stall_share"] == pytest.approx(0.25)
    assert s["roles"]["producer"]["tensor"] == pytest.approx(0.5)
    assert s["roles"]["softmax_warps"]["peer"] == pytest.approx(0.05)
    assert s["tensor_wait_share_softmax"] == pytest.approx(0.25)
    kt = s["roles"]["mma_issuers"]["key_tiles"]
    assert kt["mean_lead_cycles"] == pytest.approx(300) and kt["late_waits"] == 2
    # key waits: 200 cycles over 3 waits with a floor of 50 each -> 50 cycles beyond it
    assert s["k_wait_share_beyond_floor"] == pytest.approx(50 / 2000)
    assert s["cta_span_last_launch"]["ctas"] == 2
    assert s["cta_span_last_launch"]["last_end_us"] == pytest.approx(8.0)
    pw = s["roles"]["softmax_warps"]["per_warp_cycles"]
    assert pw["first_tile"] == pytest.approx(150) and pw["other_tile"] == pytest.approx(112.5)
    assert pw["epilogue"] == pytest.approx(100) and pw["epilogue_o_load"] == pytest.approx(30)


def test_bwd_wait_profile_summary():
    n = len(bench.BWD_WAIT_KINDS)
    raw = [0] * (3 * n)
    raw[0:3] = [1000, 200, 300]                      # producer: total, K/V slot, query stage
    raw[n + 0], raw[n + 4], raw[n + 6] = 2000, 500, 1000   # MMA: total, scores read out, operands
    ew = 2 * n
    raw[ew + 0] = 8000
    raw[ew + 8:ew + 14] = [800, 0, 400, 4000, 1200, 800]   # scores, stats, read, math, prev, stores
    raw[ew + 15], raw[ew + 16], raw[ew + 17] = 400, 4, 2
    s = bench.bwd_wait_profile_summary(raw)
    r = s["roles"]
    assert r["producer"]["kv_slot_free"] == pytest.approx(0.2)
    assert r["mma_issuer"]["operands_ready"] == pytest.approx(0.5)
    assert "row_statistics" not in r["elementwise_warps"]
    pt = r["elementwise_warps"]["per_tile_cycles"]
    assert pt["math"] == pytest.approx(1000) and pt["all"] == pytest.approx(2000)
    assert r["elementwise_warps"]["per_item_epilogue_cycles"] == pytest.approx(200)


def test_dq_wait_profile_summary():
    n = len(bench.DQ_WAIT_KINDS)
    raw = [0] * (3 * n)
    raw[n + 0], raw[n + 7] = 1000, 250                 # MMA: waiting for dS a quarter of its time
    ew = 2 * n
    raw[ew + 0] = 6400
    raw[ew + 9:ew + 13] = [400, 800, 2400, 800]        # scores, TMEM read, math, dS store
    raw[ew + 14], raw[ew + 15], raw[ew + 16] = 300, 4, 1
    s = bench.dq_wait_profile_summary(raw)
    assert s["roles"]["mma_issuer"]["ds_ready"] == pytest.approx(0.25)
    pt = s["roles"]["elementwise_warps"]["per_tile_cycles"]
    assert pt["math"] == pytest.approx(600) and pt["all"] == pytest.approx(1600)
    assert s["roles"]["elementwise_warps"]["per_item_epilogue_cycles"] == pytest.approx(300)
