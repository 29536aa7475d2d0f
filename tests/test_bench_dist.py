"""bench.py's multi-rank host logic on CPU (gloo, world_size 2): barrier and
max-over-ranks timing, whole-job throughput = units of all ranks / max time,
and the reference arm running on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.barrier()
    value, ms = bench.aggregate(10.0 * (rank + 1), 1e12, d)   # rank 1 is the slow one: 20 ms
    q.put((rank, value, ms, d.max(rank)))
    d.close()


def test_aggregate_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, ms, mx in out:
        assert ms == 20.0                      # max over ranks
        assert abs(value - 100.0) < 1e-9       # 2 ranks x 1e12 flop / 20 ms = 100 TFLOP/s
        assert mx == 1


def _run_bench(rank):
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                           "tiny", "--steps", "2", "--warmup", "1"], env=env, capture_output=True, text=True,
                          timeout=300)


def test_reference_arm_prints_on_rank0_only():
    r1 = _run_bench(1)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_bench(0)
    assert r0.returncode == 0
    lines = [l for l in r0.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_percentiles_nearest_rank():
    import bench
    assert bench.percentiles(list(range(1, 11))) == {"p10": 1, "p50": 5, "p90": 9}
    assert bench.percentiles([3.0]) == {"p10": 3.0, "p50": 3.0, "p90": 3.0}
    assert bench.percentiles([]) == {}
    # order of the input does not matter
    assert bench.percentiles([9, 1, 5, 3, 7]) == bench.percentiles([1, 3, 5, 7, 9]) == {"p10": 1, "p50": 5, "p90": 9}


def test_clock_summary_window_and_reasons():
    import datetime

    import bench
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def line(dt_ms, mhz, watts, cap="Not Active", thermal="Not Active"):
        ts = (t0 + datetime.timedelta(milliseconds=dt_ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {mhz}, 2070, {watts}, 0x0, Not Active, Not Active, {thermal}, {cap}\n"

    lines = [line(0, 2070, 100), line(100, 1500, 1300, cap="Active"), line(200, 1400, 1350, cap="Active"),
             line(300, 1800, 900), line(400, 2070, 120), "garbage\n"]
    base = t0.timestamp()
    s = bench.clock_summary(lines, window=(base + 0.05, base + 0.25))
    assert s["samples"] == 5 and s["samples_in_value_region"] == 2
    assert s["sm_mhz"] == 1450.0                     # median of the two samples inside the window
    assert s["samples_under_load"] == 3              # power >= half of the 1350 W maximum
    assert s["sm_mhz_under_load_all_regions"] == 1500.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1350.0 and s["sm_max_mhz"] == 2070.0
    # no sample in the window: fall back to the samples under load
    s2 = bench.clock_summary(lines, window=(base + 10, base + 11))
    assert s2["samples_in_value_region"] == 0 and s2["sm_mhz"] == 1500.0
    s3 = bench.clock_summary([line(0, 1000, 500, thermal="Active")])
    assert s3["reasons"] == ["sw_thermal_slowdown"]
    assert bench.clock_summary(["garbage\n"]) is None


def test_strip_comments_keeps_code_and_literals():
    import bench
    src = ('int a = 1; // trailing\n/* block\n   comment */ const char *s = "x//y/*z*/";\n'
           "char q = '\"'; char e = '\\\\';\n\n   int b;   // c\n")
    out = bench.strip_comments(src)
    assert out.splitlines() == ['int a = 1;', 'const char *s = "x//y/*z*/";', "char q = '\"'; char e = '\\\\';",
                                'int b;']
    # comment and whitespace edits keep the hash; a code edit changes it
    assert bench.strip_comments(src.replace("trailing", "other words")) == out
    assert bench.strip_comments(src.replace("int b;", "int b2;")) != out


def test_profiled_traffic_follows_the_kernel_source_hash(tmp_path, monkeypatch):
    """roofline.traffic comes from profiles/traffic.json only while the entry's hash matches the
    kernel sources as compiled; every committed entry names its summary, which exists."""
    sys.path.insert(0, ROOT)
    import bench
    current = bench.sources_sha(bench.TGATHER_SOURCES)
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"k/ok": {"source_sha256_16": current, "dram_bytes_per_launch": 123.0},
                                "k/stale": {"source_sha256_16": "0" * 16, "dram_bytes_per_launch": 456.0}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.profiled_traffic("k/ok", bench.TGATHER_SOURCES) == 123.0
    assert bench.profiled_traffic("k/stale", bench.TGATHER_SOURCES) is None
    assert bench.profiled_traffic("k/missing", bench.TGATHER_SOURCES) is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.json"))
    assert bench.profiled_traffic("k/ok", bench.TGATHER_SOURCES) is None
    committed = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key, entry in committed.items():
        assert entry["dram_bytes_per_launch"] > 0, key
        assert os.path.exists(os.path.join(ROOT, "profiles", entry["summary"])), key
        assert entry["command"].startswith("ncu ") and "--clock-control none" in entry["command"], key


def test_bench_refuses_timings_of_calls_that_stopped_early():
    """A bounded device wait that expired leaves its status in the workspace, and the calls after it
    return at once: the bench must stop rather than report their times as throughput."""
    import pytest
    import torch
    import bench
    ws = torch.zeros(256, dtype=torch.uint8)
    bench.check_device_status(ws, "a clean region")
    ws[:4].view(torch.int32)[0] = -6
    with pytest.raises(RuntimeError, match="bounded device wait"):
        bench.check_device_status(ws, "a region with a timeout")
