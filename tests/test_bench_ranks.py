"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2): the
barrier, the max over ranks of the timed region, and the whole-job value.
The layer itself is not sharded (replicas only), so this is all of the N > 1
path apart from the per-rank GPU work."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    ranks = bench.Ranks(backend="gloo")
    try:
        ranks.barrier()
        seconds = 1.0 + rank  # rank 1 is the slow one
        slowest = ranks.max(seconds)
        value = bench.aggregate(units_per_rank=1000.0, world=ranks.world, max_seconds=slowest)
        q.put((rank, ranks.world, slowest, value))
    finally:
        ranks.close()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, world, slowest, value in got:
        assert world == 2
        assert slowest == 2.0
        assert value == pytest.approx(1000.0 * 2 / 2.0)


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    r = bench.Ranks()
    assert r.world == 1 and r.rank == 0 and r.dist is None
    assert r.max(3.5) == 3.5
    r.barrier()
    assert bench.aggregate(100, 1, 0.5) == 200


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("fmt", ["int8", "fp8", "int8-smooth"])
def test_reference_arm_line_on_the_host(fmt):
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the contract's keys, for every format, on the tiny layer."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "1", "--format", fmt],
                       capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "cpu_baseline", "e2e",
                "config", "dtype"):
        assert key in line, key
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_committed_profile_tables_are_read_for_the_current_sources():
    """`roofline.traffic` comes from the committed ncu table only while the
    GEMM sources hash as they did at capture; the tensor rates are read as
    committed."""
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    for cfg, kernel, fmt in (("prefill", "gemm1_gateup", "int8"), ("decode", "gemm1_gateup", "int8"),
                             ("decode", "fused_layer", "int8"), ("prefill_fp8", "gemm1_gateup", "fp8"),
                             ("decode_fp8", "gemm1_gateup", "fp8")):
        ent = table[cfg][kernel]
        want = ent["dram_bytes_per_launch"] if ent["gemm_src_sha256_16"] == bench.gemm_source_sha(fmt) else None
        assert bench.traffic_from_profiles(cfg, kernel, fmt) == want
    assert bench.traffic_from_profiles("no_such_workload", "gemm1_gateup") is None
    f16, e4m3 = bench.tensor_rate_from_profiles("int8"), bench.tensor_rate_from_profiles("fp8")
    assert f16 > 0 and e4m3 > f16


def test_contraction_rate_program_compiles_for_sm103a(tmp_path):
    """The program behind the committed tensor rates builds with the library's
    headers (nvcc cross-compiles here; running it needs a GB300)."""
    import shutil
    import subprocess
    from w8a8_quantised_moe_gb300 import build as lib_build
    if shutil.which(lib_build.nvcc()) is None and not os.path.exists(lib_build.nvcc()):
        pytest.skip("nvcc not found")
    pkg = os.path.join(ROOT, "w8a8_quantised_moe_gb300")
    r = subprocess.run([lib_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I", os.path.join(ROOT, "include"), "-I", pkg, os.path.join(pkg, "peak_int8.cu"),
                        "-o", str(tmp_path / "peak_int8")], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
