"""bench.py's host side without a GPU: the reference arm's JSON line, and the multi-rank
aggregation (slowest rank's time, whole-job throughput) over two gloo ranks on CPU."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                          env=env, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_contract_line():
    res = _run_reference({"RANK": "0"})
    assert res.returncode == 0, res.stderr
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_is_silent_on_other_ranks():
    res = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    ms = b.slowest_rank_ms(10.0 + 5.0 * rank, world, dist)      # rank 1 is the slow one
    gbs = b.job_gbs(world, 1_000_000, 100, ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "gbs": gbs}, f)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_throughput(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    assert all(g["ms"] == 15.0 for g in got)
    # every rank's 100 calls of 1 MB over the slowest rank's 15 ms
    assert all(abs(g["gbs"] - 2 * 100 * 1e6 / 15e-3 / 1e9) < 1e-9 for g in got)


def test_one_rank_keeps_its_own_time():
    b = _bench()
    assert b.slowest_rank_ms(12.5, 1, None) == 12.5
    assert b.job_gbs(1, 60_620_800, 100, 1.6) == pytest.approx(60_620_800 * 100 / 1.6e-3 / 1e9)
