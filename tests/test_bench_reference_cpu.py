"""bench.py's reference arm (the CPU oracle timed on the host cores) prints one
JSON line with the contract's keys in every mode; it needs no GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("mode", ["train", "decode", "varlen"])
def test_reference_arm_prints_one_contract_line(mode):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--mode", mode,
           "--steps", "2", "--warmup", "3", "--ref-seq", "128"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"]


def test_stored_traffic_hash_ignores_comments_only():
    """The hash that ties profiles/traffic.json to the kernels' code changes with
    the code and not with its comments."""
    sys.path.insert(0, ROOT)
    import bench
    files = {name: "int f(int x) {  // one\n    return x + 1; /* two\n lines */\n}\n"
             for name in bench.KERNEL_SOURCES["fwd_tcgen05_bf16"] + bench.SHARED_DEVICE_SOURCES}
    h0 = bench.source_hash("fwd_tcgen05_bf16", read=files.__getitem__)
    commented = {k: v.replace("// one", "// other words") + "// trailing note\n" for k, v in files.items()}
    assert bench.source_hash("fwd_tcgen05_bf16", read=commented.__getitem__) == h0
    changed = {k: v.replace("x + 1", "x + 2") for k, v in files.items()}
    assert bench.source_hash("fwd_tcgen05_bf16", read=changed.__getitem__) != h0

