"""bench.py host logic on the CPU: rank aggregation over gloo (world size 2)
and the reference arm's JSON line."""
import json
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    d = bench.init_dist(world, "gloo")
    cpu = torch.device("cpu")
    bench.barrier(d, cpu)
    slowest = bench.max_over_ranks(10.0 + rank, d, cpu)      # rank 1 is slower
    value = bench.whole_job_tflops(2 * 10 ** 12, 4, world, slowest * 4 / 1e3)
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"slowest_ms": slowest, "value": value}, f)
    dist.destroy_process_group()


def test_rank_aggregation_gloo_world2(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    outs = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    for o in outs:
        assert o["slowest_ms"] == 11.0                        # max over ranks
        # both ranks did 4 products of 2e12 FLOP in 44 ms: 2*4*2e12 / 0.044 s
        assert abs(o["value"] - 2 * 4 * 2e12 / 0.044 / 1e12) < 1e-6


def test_whole_job_tflops_single_rank():
    assert bench.whole_job_tflops(10 ** 12, 10, 1, 1.0) == 10.0


def test_reference_arm_line(capsys):
    bench.main(["--impl", "reference", "--config", "100x37x70", "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in line
    assert line["unit"] == "TFLOPS" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_source_hash_is_stable_and_per_kernel():
    for kernel in bench.KERNEL_SOURCES:
        assert bench.source_hash(kernel) == bench.source_hash(kernel)
        assert len(bench.source_hash(kernel)) == 16
    assert bench.source_hash("tc_pair_kernel") != bench.source_hash("tc_gemm_kernel")


def test_recorded_traffic_matches_the_current_sources():
    # profiles/traffic.json is keyed by the kernel's own sources: a figure
    # recorded for other sources reads as null
    import json
    import os
    path = os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")
    with open(path) as f:
        table = json.load(f)
    import workloads
    for key, rec in table.items():
        kernel, config, mode = key.split("/")
        assert config in workloads.PROBLEMS and kernel in bench.KERNEL_SOURCES, key
        want = rec["dram_bytes_per_launch"] if rec["source_sha"] == bench.source_hash(kernel) else None
        assert bench.recorded_traffic(kernel, config, mode) == want
    assert bench.recorded_traffic("tc_pair_kernel", "no-such-config", "tc3x") is None
    # the default bench line's problem is among the recorded ones
    assert any(k.split("/")[1] == bench.parse_args([]).config for k in table)


def test_oracle_table_rows(capsys, monkeypatch):
    """--oracle-table: one JSON line per problem and thread count, with the
    host's cores and CPU model (here restricted to the two tiny problems)."""
    import workloads
    small = {k: v for k, v in workloads.PROBLEMS.items() if k in ("100x37x70", "100x37x70-int")}
    monkeypatch.setattr(workloads, "PROBLEMS", small)
    assert bench.main(["--oracle-table"]) == 0
    rows = [json.loads(l) for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    import oracle
    everyone = oracle.max_threads()
    assert [(r["oracle_table"], r["threads"]) for r in rows] == \
        [("100x37x70", everyone), ("100x37x70", 1), ("100x37x70-int", everyone), ("100x37x70-int", 1)]
    cores, model = bench.host_cpu()
    for r in rows:
        assert r["seconds"] > 0 and r["tflops"] > 0 and r["timing"] == "measured"
        assert (r["M"], r["K"], r["N"]) == (100, 37, 70)
        assert r["host_cores"] == cores >= 1 and r["cpu_model"] == model


RATES = {"tf32_flop_per_clk_sm": 4000.0, "tf32_pair_flop_per_clk_sm": 4096.0,
         "ffma_flop_per_clk_sm": 250.0, "sm_mhz": 1500.0, "num_sms": 100}
PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}


def test_roofline_takes_the_probed_rate_times_the_sampled_clock():
    clocks = {"sm_mhz": 2000.0, "window": "timed steps"}
    flop, nbytes = 2 * 8192 ** 3, 4 * 3 * 8192 ** 2
    pair = bench.roofline("tc_pair_kernel", "tc3x", flop, nbytes, 1e-3, RATES, clocks, PEAKS, "measured")
    assert pair["bound"] == "tensor"
    assert abs(pair["peak"] - 4096.0 * 100 * 2000e6 / 1e12) < 1e-9          # pair rate x SMs x clock
    assert abs(pair["achieved"] - 3 * flop / 1e-3 / 1e12) < 1e-6            # three products per FLOP
    assert abs(pair["frac"] - pair["achieved"] / pair["peak"]) < 1e-12
    assert abs(pair["secondary"]["peak"] - 2000.0 * 1.1 / 2.25) < 1e-9
    single = bench.roofline("tc_gemm_kernel", "tc1x", flop, nbytes, 1e-3, RATES, clocks, PEAKS, "measured")
    assert abs(single["peak"] - 4000.0 * 100 * 2000e6 / 1e12) < 1e-9       # single-SM rate
    assert abs(single["achieved"] - flop / 1e-3 / 1e12) < 1e-6               # one product
    ffma = bench.roofline("ffma_gemm_kernel", "ffma", flop, nbytes, 1e-3, RATES, clocks, PEAKS, "measured")
    assert ffma["bound"] == "alu" and abs(ffma["peak"] - 250.0 * 100 * 2000e6 / 1e12) < 1e-9
    # no clock samples: the clock the probe saw
    noclk = bench.roofline("ffma_gemm_kernel", "ffma", flop, nbytes, 1e-3, RATES, None, PEAKS, "measured")
    assert abs(noclk["peak"] - 250.0 * 100 * 1500e6 / 1e12) < 1e-9


def test_roofline_prefers_the_kernels_own_clock():
    flop, nbytes = 2 * 8192 ** 3, 4 * 3 * 8192 ** 2
    clocks = bench.with_kernel_clock({"sm_mhz": 2070.0, "window": "timed steps"},
                                     (1000, 2000), (1000 + 1_750_000, 2000 + 1_000_000))
    assert abs(clocks["kernel_sm_mhz"] - 1750.0) < 1e-9     # 1.75 M clocks in 1 ms
    pair = bench.roofline("tc_pair_kernel", "tc3x", flop, nbytes, 1e-3, RATES, clocks, PEAKS, "measured")
    assert abs(pair["peak"] - 4096.0 * 100 * 1750e6 / 1e12) < 1e-9
    at = pair["at_reported_clock"]
    assert at["sm_mhz"] == 2070.0 and abs(at["peak"] - 4096.0 * 100 * 2070e6 / 1e12) < 1e-9
    assert abs(at["frac"] - pair["achieved"] / at["peak"]) < 1e-12 and at["frac"] < pair["frac"]
    # a record that did not move (no persistent launch timed) leaves the summary as it was
    same = {"sm_mhz": 2070.0, "window": "timed steps"}
    assert bench.with_kernel_clock(same, (5, 5), (5, 5)) == same
    assert bench.with_kernel_clock(None, (0, 0), (100, 50))["kernel_sm_mhz"] == 2000.0
    # the memory roof does not depend on the clock
    M, K, N = 65536, 1024, 64
    r = bench.roofline("tc_gemm_kernel", "tc3x", 2 * M * N * K, 4 * (M * K + K * N + M * N), 60e-6,
                       RATES, clocks, PEAKS, "measured")
    assert r["bound"] == "hbm" and "at_reported_clock" not in r


def test_roofline_of_a_skinny_shape_is_memory_bound():
    M, K, N = 65536, 1024, 64
    flop, nbytes = 2 * M * N * K, 4 * (M * K + K * N + M * N)
    r = bench.roofline("tc_gemm_kernel", "tc3x", flop, nbytes, 60e-6, RATES,
                       {"sm_mhz": 2000.0, "window": "timed steps"}, PEAKS, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6000.0
    assert abs(r["achieved"] - nbytes / 60e-6 / 1e9) < 1e-6


def _smi_line(t, mhz, cap="Not Active"):
    import datetime
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return "%s, 0, %d, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, %s" % (stamp, mhz, cap)


def test_clock_summary_takes_the_timed_window():
    s = bench.ClockSampler(0, enabled=False)
    t0 = 1_800_000_000.0
    s.lines = [_smi_line(t0 + 0.02 * i, 2070 if i < 10 else 1700, "Active" if i >= 12 else "Not Active")
               for i in range(20)]
    inside = s.summary(t0 + 0.2, t0 + 0.4)             # samples 10 .. 20
    assert inside["window"] == "timed steps" and inside["sm_mhz"] == 1700
    assert inside["reasons"] == ["sw_power_cap"] and inside["samples"] >= 3
    short = s.summary(t0 + 0.05, t0 + 0.07)             # fewer than 3 samples inside
    assert short["window"].startswith("warm-up and timed steps")
    assert short["sm_mhz"] == 2070 and short["samples"] == 4
    # the wider record covers every sample up to the end of the timed steps
    assert inside["with_warmup"]["samples"] == 20 and inside["with_warmup"]["min_sm_mhz"] == 1700
    assert bench.ClockSampler(0, enabled=False).summary() is None
