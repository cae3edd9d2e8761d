"""Host-side logic of bench.py, on the CPU: clock parsing, the whole-job
metric, max-over-ranks aggregation across two gloo ranks, the ncu traffic
lookup, and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_summarize_clocks_reports_median_and_reasons():
    lines = [
        "0, 2070, 2070, 700.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    c = bench.summarize_clocks(lines)
    assert c["sm_mhz"] == 2040.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert bench.summarize_clocks([])["sm_mhz"] is None


def test_whole_job_metric_and_percentiles():
    # 2 ranks x 10 steps x 1e9 bytes in 4 s (max over ranks) = 5 GB/s
    assert bench.whole_job_gbs(10**9, 10, 2, 4.0) == pytest.approx(5.0)
    assert bench.percentile([1, 2, 3, 4, 5], 0.5) == 3
    assert bench.percentile([1, 2], 0.5) == pytest.approx(1.5)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_time = [3.0, 5.0][rank]
    mx = bench.aggregate_max(local_time, world)
    q.put((rank, mx, bench.whole_job_gbs(100, 4, world, mx)))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slower rank's time; value counts both ranks' units
    assert [r[1] for r in res] == [5.0, 5.0]
    assert res[0][2] == pytest.approx(100 * 4 * 2 / 5.0 / 1e9)


def test_traffic_lookup_is_tied_to_sources(tmp_path, monkeypatch):
    d = bench.kernel_source_digest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "x.md").write_text(
        f"traffic_bytes_per_launch: 123 workload=w cluster_size=8 source_digest={d}\n"
        "traffic_bytes_per_launch: 456 workload=w cluster_size=4 source_digest=deadbeef\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the csrc digest still comes from the repository
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: d)
    assert bench.recorded_traffic("w", 8) == 123
    assert bench.recorded_traffic("w", 4) is None  # stale digest
    assert bench.recorded_traffic("other", 8) is None


def test_reference_arm_prints_contract_line():
    wl = "tiny"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", wl, "--steps", "3", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s"
    assert line["metric"] == bench.METRIC and line["steps"] == 3
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"]["workload"] == wl and line["value"] > 0
