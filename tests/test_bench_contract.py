"""bench.py's output contract, checked on CPU: the reference arm (the oracle
timed on the host cores) prints one JSON line with the keys the driver
reads, and the GB300 arm refuses to run without a GPU instead of falling
back to anything on the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=300):
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_line():
    r = _run(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "0"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "routed tokens/sec per MoE layer on 1 GB300"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2
    assert d["warmup"] >= 3                      # at least three untimed steps whatever is asked
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("tiny")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gb300_arm_fails_without_gpu():
    r = _run(["--steps", "1", "--warmup", "1", "--no-cpu-baseline"])
    assert r.returncode != 0
    assert not r.stdout.strip(), "no result line without a GPU"


def test_tensor_peak_follows_the_clock_of_the_timed_region():
    sys.path.insert(0, ROOT)
    import bench
    pk = dict(hbm=6786.6, bf16=1910.8, bf16_sustained=1715.2, source="measured")
    at_max = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    capped = {"sm_mhz": 1650.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.tensor_peak_for(pk, 0.09, at_max) == ("burst", 1910.8, 1715.2)
    assert bench.tensor_peak_for(pk, 0.09, None) == ("burst", 1910.8, 1715.2)
    assert bench.tensor_peak_for(pk, 1.4, at_max) == ("sustained", 1715.2, 1910.8)
    assert bench.tensor_peak_for(pk, 0.5, capped) == ("sustained", 1715.2, 1910.8)
    low = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.tensor_peak_for(pk, 0.5, low)[0] == "sustained"


def test_expert_mma_rows():
    sys.path.insert(0, ROOT)
    import bench
    # gathered path: 128-row tiles
    assert bench.expert_mma_rows([0, 1, 128, 129, 316], 393, False) == 0 + 128 + 128 + 256 + 384
    # bank path: 316 -> one group, chunks 160 (158 rounded to 32) + 160 (156
    # rounded to 16); 393 -> 224 + 176 (169 -> 176); 250 -> 256; 33 -> 48;
    # 0 -> nothing
    assert bench.expert_mma_rows([316], 393, True) == 320
    assert bench.expert_mma_rows([393], 393, True) == 224 + 176
    assert bench.expert_mma_rows([250, 33, 0], 393, True) == 256 + 48
    # counts past c_recv are clamped
    assert bench.expert_mma_rows([500], 393, True) == 224 + 176
    # 900 rows: three groups of 304, 304, 292 -> chunks 160+144, 160+144, 160+144
    assert bench.expert_mma_rows([900], 1000, True) == 3 * 304


def test_expert_stream_bytes_match_the_traffic_records():
    """The expert products' DRAM floor (weights of the experts with rows once,
    rows in once, output once) against the full launch's algorithmic bytes
    the committed traffic records were scaled to (full workload: 384 experts
    with rows, 121,556 kept rows)."""
    sys.path.insert(0, ROOT)
    import bench
    from moe_routing_capacity_gb300 import workloads as wl
    recs = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    cfg = wl.CONFIGS["full"]
    st = {"kept": 121556}
    for name in ("gemm_expert_gateup", "gemm_expert_down"):
        got = bench.expert_stream_bytes(name, cfg, st, 384) * 1e9
        assert round(got) == recs[name]["full_algorithmic_bytes"], name
    assert bench.expert_stream_bytes("combine", cfg, st, 384) is None


def test_source_hash_follows_code_not_comments():
    """A traffic record stays valid through comment and layout edits of the
    kernel's sources, and not through a change of code."""
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) {  // the same\n  return x + 1; /* block\n comment */ }\n"
    b = "int f(int x) {\n    return x + 1;\n}\n// another comment\n"
    c = "int f(int x) { return x + 2; }"
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
