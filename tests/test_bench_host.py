"""Host-side logic of bench.py, without a GPU: the reference arm's JSON line
(the float64 oracle timed on the host cores), the silence of ranks other
than 0, the traffic record's tie to the kernel sources, and the workload
table (every workload generates [N,T] inputs and names its bytes per
env-step)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env=None):
    e = dict(os.environ)
    if env:
        e.update(env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--workload", "gae_8x128", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "env-steps/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "gae_8x128"
    sys.path.insert(0, ROOT)
    import bench
    # both arms print the same config object for a workload
    assert d["config"] == bench.workload_config("gae_8x128")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_warmup_is_at_least_three():
    r = _bench("--impl", "reference", "--workload", "gae_8x128", "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    assert json.loads(r.stdout.strip().splitlines()[-1])["warmup"] == 3


def test_reference_arm_other_ranks_print_nothing():
    r = _bench("--impl", "reference", "--workload", "gae_8x128", "--steps", "1", "--warmup", "3",
               env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


@pytest.fixture()
def bench_module():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def test_traffic_record_only_for_the_recorded_sources(bench_module, monkeypatch):
    b = bench_module
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)["records"]
    key = "gae_returns@gae_returns_4096x1024"
    entry = rec[key]
    monkeypatch.setattr(b, "_csrc_hash", lambda: entry["csrc_sha"])
    assert b._ncu_traffic("gae_returns", "gae_returns_4096x1024") == entry["dram_bytes_per_launch"]
    monkeypatch.setattr(b, "_csrc_hash", lambda: "0" * 16)
    assert b._ncu_traffic("gae_returns", "gae_returns_4096x1024") is None
    monkeypatch.setattr(b, "_csrc_hash", lambda: entry["csrc_sha"])
    assert b._ncu_traffic("gae_returns", "no_such_workload") is None


def test_csrc_hash_follows_the_kernel_sources(bench_module, tmp_path, monkeypatch):
    b = bench_module
    h = b._csrc_hash()
    assert len(h) == 16 and h == b._csrc_hash()
    fake = tmp_path / "linear_recurrence_scan_gb300" / "csrc"
    fake.mkdir(parents=True)
    (fake / "a.cu").write_text("x")
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    h1 = b._csrc_hash()
    (fake / "a.cu").write_text("y")
    assert b._csrc_hash() != h1


def test_every_workload_generates_its_inputs(bench_module):
    for name, wl in bench_module.WORKLOADS.items():
        assert wl["estimators"], name
        for est, bytes_per_step, cfg in wl["estimators"]:
            assert bytes_per_step > 0 and isinstance(cfg, dict), (name, est)
        T = min(wl["T"], 256)
        batch = wl["gen"](4, T)
        shapes = {k: np.shape(v) for k, v in batch.items() if v is not None and np.ndim(v) >= 2}
        assert shapes, name
        for k, s in shapes.items():
            assert s[:2] == (4, T), (name, k, s)


def test_default_headline_is_the_largest_configuration(bench_module):
    b = bench_module
    assert b.HEADLINE == "long_rows_64x1048576"
    sizes = {n: w["N"] * w["T"] for n, w in b.WORKLOADS.items()}
    assert sizes[b.HEADLINE] == max(sizes.values())
    # every named workload is measured beside the headline, each once
    assert len(set(b.SUITE)) == len(b.SUITE) and b.HEADLINE not in b.SUITE
    assert set(b.SUITE) | {b.HEADLINE} == set(b.WORKLOADS)


def test_l2_plan_rotates_small_workloads_only(bench_module):
    b = bench_module
    for name in b.WORKLOADS:
        n_sets, set_bytes = b.l2_plan(name)
        assert set_bytes > 0
        if set_bytes > 4 * b.L2_BYTES:
            assert n_sets == 1, name
        else:
            assert n_sets * set_bytes > 129 * 1024 * 1024 or n_sets == 16, name
    assert b.l2_plan("long_rows_64x1048576")[0] == 1
    assert b.l2_plan("gae_returns_4096x1024")[0] >= 4
