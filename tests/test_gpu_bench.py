"""The native arm of bench.py on a GPU: one JSON line with every key of the
contract, numbers that hang together, and the device results checked first.

Runs the small tiny_direct workload (8 ranks x 128 tokens), a packed-rows run
and a cached run, each as its own process, the way the benchmark is launched.
"""
import json
import os
import subprocess
import sys
import time
from types import SimpleNamespace

import pytest

import bench
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*extra):
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny_direct",
                        "--steps", "4", "--warmup", "3", *extra], capture_output=True, text=True, timeout=900,
                       cwd=ROOT)
    wall_s = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0]), wall_s


def dedup_rows(wl):
    idx, _ = W.routing(wl)
    st, lay = oracle.layout(wl, idx)
    assert st == 0
    return int(lay["num_tokens_per_rank"].sum())


def test_native_line_carries_the_whole_contract():
    d, wall_s = run_bench()
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches", "phases", "phase_replay", "launch_floor_us", "graph"):
        assert key in d, key
    wl = W.WORKLOADS["tiny_direct"]
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    args = SimpleNamespace(cached=False, copy_path=0)
    assert d["config"] == bench.run_config(wl, args, 1, dedup_rows(wl))
    # value is tokens per second of the timed steps
    assert d["value"] == pytest.approx(wl.num_ranks * wl.num_tokens / (d["ms_per_step"] * 1e-3), rel=1e-6)
    assert d["ms_per_step"] * d["steps"] < wall_s * 1e3
    # three launches of this library per step: layout, dispatch, combine
    assert d["gpu_launches"] == d["steps"] * 3

    roof = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    phase = "combine" if roof["kernel"] == "combine_kernel" else "dispatch"
    assert roof["achieved"] == pytest.approx(d["phases"][phase]["gbs"])

    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0 and cpu["sample"]

    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "tokens/s"
    # inputs in (x bf16, top-k int64, weights fp32) and the combined output back, per step
    R, T, K, H = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.hidden
    assert e2e["h2d_bytes_per_step"] == R * T * (H * 2 + K * 8 + K * 4)
    assert e2e["d2h_bytes_per_step"] == R * T * H * 2
    assert e2e["value"] != d["value"]

    clocks = d["clocks"]
    assert clocks["sm_max_mhz"] > 0 and isinstance(clocks["reasons"], list)

    for k in ("layout", "dispatch", "combine"):
        assert d["phases"][k]["us"] > 0
        assert d["phase_replay"][k]["us"] > 0
    assert d["graph"]["ms_per_step"] > 0


def test_packed_rows_and_cached_lines():
    d, _ = run_bench("--compact", "--no-e2e", "--no-cpu-baseline")
    wl = W.WORKLOADS["tiny_direct"].replace(compact=2)
    assert d["config"] == bench.run_config(wl, SimpleNamespace(cached=False, copy_path=0), 1, dedup_rows(wl))
    assert d["memory"]["recv_x_rows"] < wl.num_ranks * wl.num_ranks * wl.num_max_tokens_per_rank
    c, _ = run_bench("--cached", "--no-e2e", "--no-cpu-baseline")
    # the stored layout is replayed: two launches a step, and no layout replay
    assert c["gpu_launches"] == c["steps"] * 2
    assert "layout" not in c["phase_replay"]
