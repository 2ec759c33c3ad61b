"""bench.py's host logic without a GPU: the metric formulas against the page's
printed table, the reference arm end to end, and the multi-rank aggregation
over a world-size-2 gloo process group."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _golden():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "busbw_pr154580.txt")):
        if line.strip() and not line.startswith("#"):
            table, mib, us, gbps = line.split()
            rows.append((table, float(mib), float(us), float(gbps)))
    return rows


def test_busbw_reproduces_the_pages_table():
    rows = _golden()
    assert len(rows) == 28
    for table, mib, us, gbps in rows:
        got = bench.busbw_gbps(mib * 2**20, us * 1e-6)
        # the page rounds time to 0.01 us and BusBw to 0.01 GB/s
        assert abs(got - gbps) <= 0.01 + gbps * 0.01 / us + 1e-9, (table, mib, got, gbps)


def test_moved_and_algorithmic_bytes():
    S = np.array([[1, 2], [3, 4]])
    assert bench.moved_bytes(S, 8) == 80
    assert bench.algorithmic_bytes(S, 8) == 160 + 24 * 4
    assert bench.whole_job_value(10.0, 4, 2.0) == 20.0


def test_traffic_counters_follow_their_kernels_sources(tmp_path, monkeypatch):
    """A counter is reported only while its kernel family's sources hash to
    the value recorded with it: the dispatch kernels and the exchange engines
    are built from different files."""
    ex, dp = bench.kernel_source_sha("a2av_bulk_kernel"), bench.kernel_source_sha("dispatch_x")
    assert ex != dp and ex == bench.kernel_source_sha("a2av_staged_multi_kernel")
    assert "dispatch.cu" in bench.kernel_sources("dispatch_place_copy_kernel")[0]
    assert "dispatch.cu" in bench.kernel_sources("combine_tiny_kernel")[0]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({
        "a2av_bulk_kernel:w": {"source_sha": ex, "dram_bytes": 50, "algorithmic_bytes": 100},
        "dispatch_copy_kernel:w": {"source_sha": ex, "dram_bytes": 50, "algorithmic_bytes": 100}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for rel in bench.kernel_sources("dispatch_x") + bench.kernel_sources("a2av_x"):
        (tmp_path / rel).parent.mkdir(parents=True, exist_ok=True)
        (tmp_path / rel).write_bytes(open(os.path.join(ROOT, rel), "rb").read())
    assert bench.measured_traffic("a2av_bulk_kernel:w", 1000) == 500
    assert bench.measured_traffic("dispatch_copy_kernel:w", 1000) is None  # recorded for other sources
    assert bench.measured_traffic("a2av_bulk_kernel:other", 1000) is None


def test_comments_do_not_change_a_kernels_hash():
    a = "int f(int x) { // doubled\n  return 2 * x; /* the\n value */ }\n"
    b = "int f(int x) {\n  return 2 * x;   }  // reworded comment\n"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(a.replace("2 * x", "3 * x"))


def test_workload_descriptions():
    assert "distinct (token, destination rank)" in bench.describe("cfg3", 0, 0, dedup=True)
    assert "distinct" not in bench.describe("cfg3", 0, 0)
    assert "4096 MiB/rank" in bench.describe("cfg2", 1 << 32, 0)


def test_reference_arm_runs_on_cpu():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--per-rank-bytes", str(1 << 22), "--steps", "3", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["steps"] == 3 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def _gloo_worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    b.dist_init("gloo")
    b.barrier()
    m = b.reduce_max(1.0 + rank)
    v = b.whole_job_value(5.0, world, m)
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_replicas_aggregate_over_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 1000
    procs = [ctx.Process(target=_gloo_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [m for _, m, _ in res] == [2.0, 2.0]  # max over ranks
    assert [v for _, _, v in res] == [5.0, 5.0]  # 2 ranks x 5 units / 2 s


def test_reference_config_equals_the_gpu_lines():
    """Both arms describe the workload with the same config dict."""
    import argparse
    import workloads as wl
    P = 1 << 22
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--per-rank-bytes", str(P), "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    got = json.loads(out.stdout.strip().splitlines()[-1])["config"]
    w = wl.cfg2(P)
    args = argparse.Namespace(workload="cfg2", op="dispatch", per_rank_bytes=P, seed=0,
                              tokens=8192, batch=8192, dedup=False, hidden=7168)
    want = bench.exchange_config(args, w.W, w.row_bytes, int(np.mean([b.size for b in w.inputs])),
                                 bench.moved_bytes(w.splits, w.row_bytes),
                                 sum(b.size for b in w.inputs) < 2 * bench.L2_BYTES, 1)
    assert got == want


def test_gpus_flag_must_match_the_launcher(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "1")
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2"])
    assert "WORLD_SIZE=1" in str(e.value)


def test_host_memory_shortfall_is_refused_not_shrunk(monkeypatch):
    import argparse
    import torch
    monkeypatch.setattr(bench, "host_memory_available", lambda: 8 << 30)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    args = argparse.Namespace(workload="cfg2", per_rank_bytes=1 << 32, seed=0)
    with pytest.raises(SystemExit) as e:
        bench.load_workload(args, torch)
    assert "Refusing" in str(e.value)
    assert args.per_rank_bytes == 1 << 32  # the request is untouched


def test_spawned_replicas_aggregate_over_gloo(tmp_path, capfd):
    """bench.py --gpus N without a launcher starts N local processes with the
    rank variables torchrun sets; here each runs a stand-in step over a gloo
    group and rank 0 prints the aggregated line."""
    script = tmp_path / "replica.py"
    script.write_text(
        "import json, os, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "rank, local, world = bench.dist_env()\n"
        "bench.dist_init('gloo')\n"
        "bench.barrier()\n"
        "t = bench.reduce_max(1.0 + rank)\n"
        "if rank == 0:\n"
        "    print(json.dumps({'world': world, 'local': local, 'max_s': t,\n"
        "                      'value': bench.whole_job_value(6.0, world, t),\n"
        "                      'argv': sys.argv[1:]}))\n")
    rc = bench.spawn_replicas(2, ["--gpus", "2", "--steps", "3"], script=str(script))
    assert rc == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["world"] == 2 and line["max_s"] == 2.0 and line["value"] == 6.0
    assert line["argv"] == ["--gpus", "2", "--steps", "3"]


def test_traffic_keys_name_the_workload_variant():
    import argparse
    a = argparse.Namespace(workload="cfg3", hidden=512, tokens=8192, dedup=False, batch=8192)
    assert bench.workload_key(a) == "cfg3_h512"
    a.hidden, a.tokens = 7168, 128
    assert bench.workload_key(a) == "cfg3_t128"
    a.workload = "cfg2"
    assert bench.workload_key(a) == "cfg2"
