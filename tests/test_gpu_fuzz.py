"""Randomised GPU-vs-oracle parity over every mode combination.

Each case draws a small configuration (ranks, scale-out split, experts per rank,
top-k, tokens, max tokens, hidden, input/receive dtypes, expanded or row form,
alignment and zero padding, compact and packed rows, packed scales, masking, the way unchanged
rows are copied) from a seeded generator, runs layout -> dispatch -> combine through the C ABI and compares
every output with the oracle: layouts, every row of the receive buffers (which
start filled with 0xFF, so untouched rows must stay 0xFF and padding rows must
become zero), the scale and sidecar rows, and the combined tokens.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_02_gb300 as ep
import oracle
import workloads as W
from _harness import GpuRun, assert_layout_equal, inputs, u16

pytestmark = pytest.mark.gpu

N_CASES = 160


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    n_so = int(rng.choice([1, 1, 2, 4]))
    n_su = int(rng.integers(1, 9))
    R = n_so * n_su
    L = int(rng.choice([1, 2, 3, 8, 16]))
    E = R * L
    K = int(rng.integers(1, min(E, 12) + 1))
    T = int(rng.choice([0, 1, 37, 255, 256, 513, 700])) if seed % 7 else int(rng.integers(0, 600))
    M = T + int(rng.choice([0, 0, 1, 50]))
    M = max(M, 1)
    kind = rng.choice(["bf16", "cast", "precast"])
    expand = bool(rng.random() < 0.35)
    x_dtype, recv = {"bf16": ("bf16", "bf16"), "cast": ("bf16", "fp8"), "precast": ("fp8", "fp8")}[kind]
    H = int(rng.integers(1, 33)) * 8 if kind == "bf16" else int(rng.integers(1, 13)) * 128
    # keep the row-form receive buffer (R*R*M rows) under ~64 MB
    row_bytes = H * (2 if recv == "bf16" else 1)
    while R * R * M * row_bytes > 64 << 20 and M > 1:
        T, M = T // 2, max(M // 2, 1)
    align = int(rng.choice([1, 2, 4, 128])) if expand else 1
    return W.Workload(
        f"fuzz{seed}", n_so, n_su, E, K, T, M, H, x_dtype=x_dtype, recv_dtype=recv, expand=expand,
        expert_alignment=align, zero_padding=expand and bool(rng.random() < 0.5),
        compact=0 if expand else int(rng.choice([0, 0, 0, 1, 2])),
        sf_pack=recv == "fp8" and bool(rng.random() < 0.4),
        routing=str(rng.choice(["gauss", "zipf"])), mask_frac=float(rng.choice([0.0, 0.1, 0.5])),
        y_kind="random", seed=seed)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_fuzz_case(seed):
    wl = draw(seed)
    idx, w, x, sf = inputs(wl)
    st, olay = oracle.layout(wl, idx)
    assert st == 0
    run = GpuRun(wl, idx, w, x, sf, num_prologue_sms=seed % 5 * 7, num_sms=(seed % 3) * 11,
                 copy_path=seed % 3).layout()
    run.recv = ep.alloc_recv(run.cfg, run.dev)
    for t in (run.recv.recv_x, run.recv.recv_sf, run.recv.recv_topk_idx, run.recv.recv_topk_weights,
              run.recv.recv_src_metadata):
        if t is not None:
            t.view(torch.uint8).fill_(0xFF)
    run.dispatch()
    y = W.expert_outputs(wl, max(ep.ep_recv_rows(run.cfg), 1), device="cuda")
    run.combine(y)
    assert run.status() == ep.EP_OK, wl
    assert_layout_equal(run.layout_np(), olay, wl.expand)

    st, orec = oracle.dispatch(wl, olay, x, sf, idx, w, fill=0xFF)
    assert st == 0
    rows = int(olay["exp_region"][-1]) if wl.expand else orec["recv_x"].shape[0]
    row_bytes = wl.hidden * (1 if wl.recv_dtype == "fp8" else 2)
    got = run.recv.recv_x[:rows].contiguous().view(torch.uint8).cpu().numpy().reshape(rows, row_bytes)
    exp = np.ascontiguousarray(orec["recv_x"][:rows]).view(np.uint8).reshape(rows, row_bytes)
    assert np.array_equal(got, exp), wl
    if wl.recv_dtype == "fp8":
        got_sf = run.recv.recv_sf[:rows].cpu().numpy().view(np.uint32)
        assert np.array_equal(got_sf, orec["recv_sf"][:rows].view(np.uint32)), wl
    # whole sidecar buffers: written rows equal, the rest still 0xFF on both sides
    K = wl.num_topk
    for name, width in (("recv_topk_idx", K), ("recv_topk_weights", K), ("recv_src_metadata", K + 2)):
        g = getattr(run.recv, name).reshape(-1, width).cpu().numpy()
        assert np.array_equal(g.view(np.uint8), orec[name].view(np.uint8)), (wl, name)

    exp = oracle.combine_gathered(oracle.global_rows(wl, olay, idx).reshape(-1, K),
                                  u16(y), w.numpy().reshape(-1, K)) if wl.num_tokens else None
    if exp is not None:
        assert np.array_equal(u16(run.out).reshape(-1, wl.hidden), exp), wl
