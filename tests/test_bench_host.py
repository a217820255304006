"""Host-side logic of bench.py without a GPU: the multi-rank aggregation (two gloo ranks on the CPU,
as torchrun would start them), the reference arm's JSON line, and the traffic record lookup."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist = bench.dist_init(world)
    # rank r moved (r + 1) GB in (r + 1) * 0.5 s
    total, slowest = bench.aggregate(dist, (rank + 1) * 1e9, (rank + 1) * 0.5)
    q.put((rank, total, slowest))
    dist.destroy_process_group()


def test_two_rank_aggregation_is_sum_over_max():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, total, slowest in res:
        assert total == 3e9 and slowest == 1.0     # whole-job bytes over the slowest rank


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "c1", "--steps", "5", "--warmup", "3",
                          "--reference-seconds", "2"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_shape_flag_times_any_workload():
    """--shape MxKxL replaces the named config: the reference arm's line names it, and a K that is
    not a multiple of 16 is rejected before anything runs."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--shape", "96x17408x2", "--steps", "3", "--warmup", "3",
                          "--reference-seconds", "2"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    d = json.loads([ln for ln in out.stdout.splitlines() if ln.strip()][-1])
    cfg = d["config"]
    assert (cfg["M"], cfg["K"], cfg["L"]) == (96, 17408, 2) and "96x17408x2" in cfg["workload"]
    assert cfg["bytes_per_call"] == 96 * 17408 * 2 * 9 // 16 + 17408 * 2 * 9 // 16 + 2 * 96 * 2
    bad = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--shape", "96x100x1"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert bad.returncode != 0 and "multiple of 16" in bad.stderr


def test_warmup_below_three_is_rejected():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0


def test_traffic_record_requires_matching_sources(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    assert len(bench.kernel_source_digest()) == 16
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (prof / "traffic_c9.txt").write_text(
        "kernel_sources_sha256_16 = 0000000000000000\n"
        "dram_bytes_read_per_launch = 100\ndram_bytes_write_per_launch = 20\n")
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0000000000000000")
    assert bench.recorded_traffic("c9") == 120.0
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "ffffffffffffffff")
    assert bench.recorded_traffic("c9") is None


def test_code_only_digest_ignores_comments_not_code():
    import bench

    a = 'int x = 1; // note\n/* block\n comment */ const char* s = "a // b";\n'
    b = 'int x = 1;\n\n   const char* s = "a // b"; // other note'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(a.replace("x = 1", "x = 2"))
    assert '"a // b"' in bench._code_only(a)


def test_cpu_baseline_times_the_c_oracle_on_every_thread():
    import bench
    import workloads
    from oracle import cref

    r = bench.cpu_baseline(workloads.make("c1"), 1.0)
    assert r["kind"] == "oracle" and r["value"] > 0 and r["cores"] == cref.max_threads()
    assert r["single_thread"]["cores"] == 1 and r["single_thread"]["value"] > 0
    assert "plain C" in r["sample"] and r["host_cpus"] == (os.cpu_count() or 1)


def test_gpus_flag_starts_the_ranks_itself():
    """--gpus 2 without torchrun: bench.py starts two ranks (gloo on the CPU for the host-side
    exchange); under several ranks the reference arm runs on rank 0 alone, which prints the one
    line with n_gpus 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--config", "c1", "--steps", "3", "--warmup", "3",
                          "--reference-seconds", "2"], capture_output=True, text=True,
                         timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_gpus_flag_must_match_world_size():
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "3", "--config", "c1", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert out.returncode != 0 and "WORLD_SIZE" in out.stderr


def test_spawned_ranks_aggregate_over_gloo(tmp_path):
    """The ranks bench.py starts for --gpus N join one gloo group: a two-rank job through
    spawn_ranks whose ranks report sum-over-max exactly as the GPU arm does."""
    sys.path.insert(0, ROOT)
    import bench

    script = tmp_path / "rank.py"
    script.write_text(
        "import os, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "world, rank, _ = bench.dist_env()\n"
        "dist = bench.dist_init(world)\n"
        "total, slowest = bench.aggregate(dist, (rank + 1) * 1e9, (rank + 1) * 0.5)\n"
        "assert world == 2 and total == 3e9 and slowest == 1.0, (world, total, slowest)\n"
        "dist.destroy_process_group()\n")
    old = bench.__file__
    try:
        bench.__file__ = str(script)
        assert bench.spawn_ranks(2, []) == 0
    finally:
        bench.__file__ = old
