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
