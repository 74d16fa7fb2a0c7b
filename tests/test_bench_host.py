"""Host-side pieces of bench.py, on the CPU.

- The byte counts behind every roofline fraction: bench.algorithmic_bytes works
  from the layout's counts; here the same totals are recounted from what the
  oracle actually writes and reads (receive rows that left their fill value,
  sidecar rows, distinct rows the combine lanes point at).
- The reference arm's JSON line (it runs the oracle only, so it runs here).
"""
import json
import os
import subprocess
import sys
import time
from types import SimpleNamespace

import numpy as np
import pytest

import bench
import oracle
import workloads as W
from _harness import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SMALL = {
    "direct": W.WORKLOADS["direct_zipf"].replace(num_tokens=64, num_max_tokens_per_rank=64, hidden=256),
    "hybrid_compact": W.WORKLOADS["hybrid_rowform"].replace(num_tokens=40, num_max_tokens_per_rank=48,
                                                           hidden=128, compact=True),
    "cast": W.WORKLOADS["dsv3_fp8"].replace(num_tokens=48, num_max_tokens_per_rank=48, hidden=512),
    "precast_packed": W.WORKLOADS["dsv3_fp8"].replace(num_tokens=48, num_max_tokens_per_rank=48, hidden=640,
                                                      x_dtype="fp8", sf_pack=True),
    "expanded_pad": W.WORKLOADS["expanded"].replace(num_tokens=24, num_max_tokens_per_rank=24, hidden=64,
                                                    expert_alignment=4, zero_padding=True),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_algorithmic_bytes_equal_what_the_oracle_moves(name):
    wl = SMALL[name]
    R, T, K, H = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.hidden
    idx, w, x, sf = inputs(wl)
    st, lay = oracle.layout(wl, idx)
    assert st == 0
    st, rec = oracle.dispatch(wl, lay, x, sf, idx, w, fill=0xFF)
    assert st == 0

    # rows the dispatch wrote: hidden rows (and zeroed padding) left the 0xFF fill
    rx = np.ascontiguousarray(rec["recv_x"]).view(np.uint8).reshape(rec["recv_x"].shape[0], -1)
    written = int((rx != 0xFF).any(axis=1).sum())
    md = rec["recv_src_metadata"].reshape(-1, K + 2)
    side_rows = int((md[:, 0] != -1).sum())  # a written row carries its source rank (>= 0) in field 0
    ix = idx.numpy()
    tokens_with_lane = int((ix >= 0).any(axis=-1).sum())
    rows = oracle.global_rows(wl, lay, idx)
    read_rows = int(np.unique(rows[rows >= 0]).size)  # distinct rows the combine lanes gather

    eb_in = 1 if wl.x_dtype == "fp8" else 2
    eb_out = 1 if wl.recv_dtype == "fp8" else 2
    G = H // 128
    sw = 4 * (((G + 3) // 4) if wl.sf_pack else G) if wl.recv_dtype == "fp8" else 0
    exp_dispatch = (tokens_with_lane * H * eb_in + (tokens_with_lane * sw if wl.x_dtype == "fp8" else 0)
                    + written * (H * eb_out + sw)
                    + side_rows * (K * 8 + K * 4 + (2 + K) * 4)
                    + R * T * K * 16)
    exp_combine = read_rows * H * 2 + R * T * H * 2 + R * T * K * 16

    ntpr = int(lay["num_tokens_per_rank"].sum())
    valid = int((ix >= 0).sum())
    pad = int(lay["exp_region"][-1]) - valid if (wl.expand and wl.zero_padding) else 0
    got = bench.algorithmic_bytes(wl, ntpr, valid, tokens_with_lane, pad)
    assert got["dispatch"] == exp_dispatch
    assert got["combine"] == exp_combine
    assert written == (valid if wl.expand else ntpr) + pad


def test_reference_arm_prints_one_contract_line():
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_direct", "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    wall_s = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    # the native arm's config, key for key (the tiny workload's layout gives the dedup rows)
    wl = W.WORKLOADS["tiny_direct"]
    idx, _ = W.routing(wl)
    st, lay = oracle.layout(wl, idx)
    args = SimpleNamespace(cached=False, copy_path=0)
    assert d["config"] == bench.run_config(wl, args, 1, int(lay["num_tokens_per_rank"].sum()))
    # ms_per_step is time actually measured: the timed steps fit in the run's own wall clock
    assert d["ms_per_step"] * d["steps"] < wall_s * 1e3
