"""Host logic of bench.py, no GPU: rank aggregation (gloo, world size 2), the
hash-gated ncu traffic record, and the reference (CPU oracle) arm."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank reports its own times; the slowest rank sets every entry
        vals = bench.aggregate_max([float(rank), 10.0 - rank, 3.0], "cpu", world)
        out[rank] = vals
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_aggregate_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert out[0] == out[1] == [1.0, 10.0, 3.0]


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate_max([1.5, 2.5], "cpu", 1) == [1.5, 2.5]


def test_traffic_reported_only_for_profiled_source(tmp_path, monkeypatch):
    import hashlib

    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    rec = {"decode": {"source": "k.cu", "sha256": hashlib.sha256(b"kernel v1").hexdigest(),
                      "bytes_per_launch": 123}}
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic() == {"decode": 123}
    src.write_text("kernel v2")  # the kernel changed since the capture
    assert bench.load_traffic() == {}


def test_committed_traffic_record_is_well_formed():
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")))
    for key in ("decode", "prefill"):
        assert rec[key]["bytes_per_launch"] > 0 and len(rec[key]["sha256"]) == 64
        assert os.path.exists(os.path.join(ROOT, rec[key]["source"]))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-seconds", "0.2"],
                       capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == bench.host_cores()  # one process per host core
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    # the same workload description as the GPU arm prints
    assert d["config"] == bench.bench_config(1)


def test_cpu_sample_sums_rows_over_processes():
    one = bench.cpu_oracle_sample(0.4, steps=1, procs=1)[0]
    two = bench.cpu_oracle_sample(0.4, steps=1, procs=2)[0]
    assert one["threads"] == 1 and two["threads"] == 2
    assert two["decode_rows"] >= 2 and two["prefill_rows"] >= 2
    assert one["decode_gbs"] > 0 and two["decode_gbs"] > 0


def test_reference_arm_other_ranks_print_nothing():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=120, env=dict(os.environ, RANK="1", WORLD_SIZE="2"))
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_decode_bytes_and_prefill_flops_match_closed_forms():
    kv, alg = bench.decode_bytes(1, 64, 8, 128, [8192])
    assert kv == 2 * 8 * 8192 * 128 * 2 == 33_554_432
    assert alg == kv + 64 * 128 * 2 * 2 + 64 * 4
    # causal 8K: sum_{i<8192} (i + 1) visible pairs per head
    assert bench.prefill_flops(1, 64, 128, 8192, 8192, 0, True) == 4 * 128 * 64 * 8192 * 8193 // 2
    # chunked: sum_{i<2048} (30721 + i) = 65,012,736 pairs per head and batch row
    assert bench.prefill_flops(2, 64, 128, 2048, 32768, 30720, True) == 4 * 128 * 64 * 2 * 65_012_736


def test_clock_samples_are_kept_inside_the_timed_region():
    rows = ["2026/12/02 10:00:00.000, 0, 1400, 2070, 300.0, 0x0, Not Active, Not Active, "
            "Not Active, Not Active",
            "2026/12/02 10:00:01.000, 0, 2070, 2070, 1200.0, 0x4, Not Active, Not Active, "
            "Not Active, Active",
            "2026/12/02 10:00:01.010, 0, 2055, 2070, 1250.0, 0x0, Not Active, Not Active, "
            "Not Active, Not Active",
            "2026/12/02 10:00:03.000, 0, 900, 2070, 200.0, 0x0, Active, Not Active, "
            "Not Active, Not Active"]
    import datetime

    t = lambda s_: datetime.datetime.strptime(s_, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    c = bench.ClockSampler.summarise(rows, (t("2026/12/02 10:00:00.990"),
                                            t("2026/12/02 10:00:01.020")))
    assert c["samples"] == 2 and c["samples_total"] == 4
    assert c["sm_mhz"] == (2070 + 2055) / 2 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]          # not the idle samples' hw_slowdown
    c = bench.ClockSampler.summarise(rows, (0.0, 1.0))  # nothing inside: all samples
    assert c["samples"] == 0 and c["samples_total"] == 4 and "hw_slowdown" in c["reasons"]
