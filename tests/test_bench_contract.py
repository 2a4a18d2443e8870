"""The JSON line of bench.py's reference arm (the fp64 oracle on the host
cores), which needs no GPU: one line with the contract's keys, and under a
two-rank launch rank 0 alone prints it."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(cmd, env=None, timeout=300):
    e = dict(os.environ)
    e.update(env or {})
    e["OMP_NUM_THREADS"] = e.get("OMP_NUM_THREADS", "4")
    return subprocess.run(cmd, cwd=ROOT, env=e, capture_output=True, text=True, timeout=timeout)


def _lines(stdout):
    return [json.loads(line) for line in stdout.splitlines() if line.strip().startswith("{")]


def _check_line(d, steps, warmup, n_gpus=1):
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s" and d["value"] > 0
    assert d["n_gpus"] == n_gpus and d["steps"] == steps and d["warmup"] == warmup
    assert d["higher_is_better"] is True and d["scaling"] in ("weak", "strong")
    assert d["vs_baseline"] is None
    assert d["dtype"] == "f64" and d["data"] == "synthetic"
    assert isinstance(d["config"], dict) and d["config"]["workload"]
    assert d["ms_per_step"] > 0
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and isinstance(cb["sample"], str) and cb["sample"]


def test_reference_arm_prints_one_contract_line():
    r = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1, r.stdout
    _check_line(lines[0], steps=2, warmup=3)


def test_bench_rejects_fewer_than_three_warmup_steps():
    r = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "2"])
    assert r.returncode != 0
    assert "--warmup must be at least 3" in r.stderr


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_under_two_ranks_prints_from_rank_0_only():
    r = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
              "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
              "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"],
             env={"OMP_NUM_THREADS": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1, r.stdout
    _check_line(lines[0], steps=2, warmup=3, n_gpus=2)


def test_cpu_baseline_reports_all_cores_and_one_thread():
    import bench
    import oracle
    from paged_kv_cache_218_gb300 import workload as W
    n_all = oracle.num_threads()
    cb = bench.cpu_baseline_obj(W.tiny(), 0.2)
    assert oracle.num_threads() == n_all  # the thread count is restored
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] == n_all
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["unit"] == "GB/s" and st["value"] > 0 and st["sample"]
