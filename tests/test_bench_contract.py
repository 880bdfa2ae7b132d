"""bench.py's output contract, checked on the CPU through its reference arm
(the oracle timed on the host): one JSON line with the keys the contract
names, the reference arm's own e2e and cpu_baseline objects, and a warm-up
floor of 3."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=600):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_prints_the_contract_line():
    r = run_bench("--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_warmup_floor_is_enforced():
    r = run_bench("--impl", "reference", "--steps", "1", "--warmup", "2", timeout=120)
    assert r.returncode != 0
    assert "warmup" in r.stderr


def test_l2_flush_reads_its_buffer():
    # the flush is a full read of a buffer (no writes): it must run without a GPU too
    import torch
    import bench
    f = bench.L2Flush(torch.device("cpu"), 1 << 16)
    f()
    assert int(f.sink) == f.buf.numel()


def test_parity_check_catches_wrong_rows():
    # the bench's all-row comparison: passes within the tolerance, fails on one bad element,
    # on a mean drift, and on a non-finite output
    import numpy as np
    import torch
    import bench
    ref = np.random.default_rng(0).standard_normal((4, 8, 16)) * 0.1
    good = torch.from_numpy(ref).half()
    p = bench.parity(good, ref)
    assert p["ok"] and p["rows"] == "all" and p["n_rows"] == 32 and p["max_abs"] <= 1e-3
    bad = good.clone()
    bad[2, 5, 7] += 0.01
    assert not bench.parity(bad, ref)["ok"]
    drift = (good.double() + 6e-4).half()
    assert not bench.parity(drift, ref)["ok"]
    nan = good.clone()
    nan[0, 0, 0] = float("nan")
    assert not bench.parity(nan, ref)["ok"]


def test_dtype_label_states_the_p_rounding():
    import bench
    assert "p rounded to f16" in bench.dtype_label("tma_mma", False)
    assert "p rounded to f16" in bench.dtype_label("tcgen05+longest_first", True)
    assert "e4m3" in bench.dtype_label("tma_mma", True)
    assert "p rounded" not in bench.dtype_label("l2_prefetch", False)
