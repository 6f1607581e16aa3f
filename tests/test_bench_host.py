"""bench.py's host-side logic without a GPU: the replica aggregation across
ranks (world_size 2 over gloo on 127.0.0.1), the algorithmic byte counts
and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times = [1.0, 2.0, 3.0] if rank == 0 else [2.0, 4.0, 6.0]  # rank 1 is the slow one
    tot, mean = bench.aggregate_times(times, world, torch.device("cpu"))
    out.put((rank, tot, mean))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_takes_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, tot, mean in got:
        assert tot == 12.0 and mean == 4.0
    sys.path.insert(0, ROOT)
    import bench
    # two replicas that each moved 1 GB per step, 3 steps, slowest rank 12 ms
    assert bench.replica_gbs(1e9, 3, 2, 12.0) == pytest.approx(500.0)


def test_workload_bytes():
    sys.path.insert(0, ROOT)
    import bench
    b = bench.workload_bytes(R=65536, H=2048, w_bytes=2048 * 4, P=456)
    assert b["rows_only"] == 6 * 65536 * 2048 + 4 * 65536 + 2048 * 4 + 4 * 2048
    assert b["pair"] == b["rows_only"] + 2 * 8 * 456 * 2048
    assert b["main"] == b["pair"] - 8 * 456 * 2048 - 4 * 2048
    r = bench.workload_bytes(R=10, H=8, w_bytes=16, P=1, dh=True, res=True)
    assert r["rows_only"] == 8 * 10 * 8 + 40 + 16 + 32
    assert r["fwd"] == 8 * 10 * 8 + 40 + 16


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "3", "--workload", "h1536_t256"], capture_output=True, text=True, env=env,
                         timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0



def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    import bench
    h = bench.kernel_source_hash()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "s.md").write_text("summary")
    rec = {"bwd_rows_kernel:w": {"source_hash": h, "dram_bytes_per_launch": 123, "summary": "profiles/s.md"},
           "bwd_rows_kernel:stale": {"source_hash": "0" * 16, "dram_bytes_per_launch": 456, "summary": "profiles/s.md"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: h)
    assert bench.recorded_traffic("bwd_rows_kernel", "w") == 123
    assert bench.traffic_record("bwd_rows_kernel", "w")["summary"] == "profiles/s.md"
    assert bench.recorded_traffic("bwd_rows_kernel", "stale") is None  # counters from other sources
    assert bench.traffic_record("bwd_rows_kernel", "missing") is None


def test_source_hash_ignores_comments_only():
    # the kernel-source hash that keys the traffic records is taken over the
    # sources without comments: a comment edit keeps the records, any edit
    # to code (a literal included) makes them stale
    import bench
    base = 'x = 1; // why\n/* how\n   more */ y = "s//t"; char c = \'/\';\n'
    same = 'x = 1;    // another reason\n\n/* two\n   lines */ y = "s//t"; char c = \'/\';  \n'
    assert bench.canonical_source(base) == bench.canonical_source(same)
    for changed in ('x = 2; // why\n/* how\n   more */ y = "s//t"; char c = \'/\';\n',
                    'x = 1; // why\n/* how\n   more */ y = "s/t"; char c = \'/\';\n',
                    'x = 1; // why\n/* how\n   more */ y = "s//t"; char c = \'*\';\n',
                    '// x = 1;\n/* how\n   more */ y = "s//t"; char c = \'/\';\n'):
        assert bench.canonical_source(changed) != bench.canonical_source(base), changed
    assert '"s//t"' in bench.canonical_source(base)


def test_traffic_record_follows_the_launch_plan(tmp_path, monkeypatch):
    # a record also holds the plan its counters were taken with: a table
    # change that gives the workload another launch makes it stale
    import bench
    h = bench.kernel_source_hash()
    (tmp_path / "profiles").mkdir()
    rec = {"bwd_rows_kernel:w": {"source_hash": h, "dram_bytes_per_launch": 5, "plan": {"ctas": 152}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: h)
    monkeypatch.setattr(bench, "workload_plan", lambda w: {"ctas": 152})
    assert bench.recorded_traffic("bwd_rows_kernel", "w") == 5
    monkeypatch.setattr(bench, "workload_plan", lambda w: {"ctas": 304})
    assert bench.recorded_traffic("bwd_rows_kernel", "w") is None


def test_kernel_hash_leaves_out_the_host_only_source():
    import bench
    csrc = os.path.join(ROOT, "bwd_dw_column_gb300", "csrc")
    files = sorted(os.listdir(csrc))
    assert "cake_api.cu" in files and bench.HOST_ONLY_SOURCES == ("cake_api.cu",)
    assert any(f.startswith("cake_bwd") for f in files)


NCU_CSV = """==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python","h","void cake::fwd_rows_kernel<3>(cake::FwdParams)","1","7","(416, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","9.99"
"1","1","python","h","void cake::bwd_rows_kernel<4, 1, 0, 0>(cake::BwdParams)","1","7","(416, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","800.5"
"1","1","python","h","void cake::bwd_rows_kernel<4, 1, 0, 0>(cake::BwdParams)","1","7","(416, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","400.25"
"1","1","python","h","void cake::bwd_rows_kernel<4, 1, 0, 0>(cake::BwdParams)","1","7","(416, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","usecond","200"
"2","1","python","h","void cake::bwd_rows_kernel<4, 1, 0, 0>(cake::BwdParams)","1","7","(416, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","801.5"
"2","1","python","h","void cake::bwd_rows_kernel<4, 1, 0, 0>(cake::BwdParams)","1","7","(416, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","400.75"
"2","1","python","h","void cake::bwd_rows_kernel<4, 1, 0, 0>(cake::BwdParams)","1","7","(416, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","ns","202000"
"""


def test_record_traffic_takes_counters_only_for_the_sources_they_came_from(tmp_path, monkeypatch):
    import bench
    h = bench.kernel_source_hash()
    (tmp_path / "profiles").mkdir()
    csv = tmp_path / "launches.csv"
    csv.write_text(NCU_CSV)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: h)
    ls = bench.parse_ncu_csv(str(csv), "bwd_rows_kernel")
    assert len(ls) == 2 and ls[0]["dram__bytes_read.sum"] == pytest.approx(800.5e6)
    args = bench.parse_args(["--record-traffic", str(csv), "--workload", "w", "--hash", "0" * 16])
    with pytest.raises(SystemExit):  # counters of other sources are refused
        bench.record_traffic(args)
    assert not (tmp_path / "profiles" / "traffic.json").exists()
    args = bench.parse_args(["--record-traffic", str(csv), "--workload", "w", "--hash", h, "--summary", "s.md",
                             "--scale", "2"])
    bench.record_traffic(args)
    ent = bench.traffic_record("bwd_rows_kernel", "w")
    assert ent["source_hash"] == h and ent["launches"] == 2
    assert ent["dram_bytes_per_launch"] == round(2 * (800.5e6 + 400.25e6 + 801.5e6 + 400.75e6) / 2)
    assert ent["ncu_us_per_launch"] == pytest.approx(402.0)
