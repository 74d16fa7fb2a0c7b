"""Pins of the oracle's lane rows (``oracle.lane_rows``), the rows the GPU
parity checks select with.

For every parity workload (at reduced sizes) and a set of seeded random
configurations across every layout mode:
  * the recv_x rows of the lanes are exactly the rows ``oracle.dispatch``
    writes: a row is written iff it comes out the same from two dispatches
    into buffers prefilled with different bytes;
  * the sidecar rows of the lanes are exactly the sidecar rows it writes;
  * the combine computed from the gathered lane rows equals ``oracle.combine``
    bit for bit.
So the rows the tests pick are the rows the oracle's own dispatch and combine
use (PR #753 Approach: slot = row block * num_max_tokens_per_rank + running
count; PR #690 Direct Recv X: compact rows from the per-source prefix).
"""
from types import SimpleNamespace

import numpy as np
import pytest

import workloads as W


def _written(a, b):
    """Rows of two fills' outputs that are equal: the rows the dispatch wrote."""
    a = a.reshape(a.shape[0], -1).view(np.uint8)
    b = b.reshape(b.shape[0], -1).view(np.uint8)
    return np.flatnonzero((a == b).all(-1))


def _check(orc, wl, idx, w, x, sf):
    st, lay = orc.layout(wl, idx)
    assert st in (0, orc.BAD_TOPK)
    st, hid, side = orc.lane_rows(wl, lay, idx)
    assert st in (0, orc.BAD_TOPK)
    st0, r0 = orc.dispatch(wl, lay, x, sf, idx, w, fill=0x00)
    st1, r1 = orc.dispatch(wl, lay, x, sf, idx, w, fill=0xFF)
    assert st0 == st1
    written = _written(r0["recv_x"], r1["recv_x"])
    expect = np.unique(hid[hid >= 0])
    if wl.expand and wl.zero_padding:  # zeroed padding rows are written too
        pad = []
        L = wl.num_experts // wl.num_ranks
        for d in range(wl.num_ranks):
            for j in range(L):
                a = lay["exp_region"][d] + lay["exp_base"][d, j] + lay["exp_cnt"][d, j]
                pad.extend(range(a, lay["exp_region"][d] + lay["exp_base"][d, j + 1]))
        expect = np.union1d(expect, np.array(pad, np.int64))
    assert np.array_equal(written, expect)
    for k in ("recv_topk_idx", "recv_topk_weights", "recv_src_metadata"):
        assert np.array_equal(_written(r0[k], r1[k]), np.unique(side[side >= 0])), k
    # combine through the gathered lane rows = the oracle's combine
    rows = orc.recv_rows(wl)
    rng = np.random.default_rng(7)
    y = (rng.standard_normal((rows, wl.hidden)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    st, out = orc.combine(wl, lay, y, idx, w)
    flat = hid.reshape(-1, wl.num_topk)
    got = orc.combine_gathered(flat, y, np.asarray(w).reshape(-1, wl.num_topk))
    assert np.array_equal(got.reshape(out.shape), out)


SMALL = {name: wl.replace(num_tokens=min(wl.num_tokens, 24),
                          num_max_tokens_per_rank=min(wl.num_tokens, 24) + (3 if wl.num_tokens > 24 else 0),
                          hidden=min(wl.hidden, 256 if wl.hidden % 128 == 0 else wl.hidden))
         for name, wl in W.PARITY.items()}


@pytest.mark.parametrize("name", list(SMALL))
def test_lane_rows_are_the_rows_dispatch_and_combine_use(orc, name):
    wl = SMALL[name]
    idx, w = W.routing(wl)
    x, sf = W.hidden(wl)
    _check(orc, wl, idx.numpy(), w.numpy(), x, sf)


def _random_case(seed):
    rng = np.random.default_rng(seed)
    n_so = int(rng.choice([1, 1, 2, 3]))
    n_su = int(rng.integers(1, 5))
    R = n_so * n_su
    L = int(rng.integers(1, 5))
    E = R * L
    K = int(rng.integers(1, min(E, 9) + 1))
    T = int(rng.integers(0, 30))
    M = T + int(rng.integers(0, 4)) or 1
    expand = bool(rng.random() < 0.3)
    compact = 0 if expand else int(rng.choice([0, 1, 2]))
    wl = SimpleNamespace(n_so=n_so, n_su=n_su, num_ranks=R, num_experts=E, num_topk=K, num_tokens=T,
                         num_max_tokens_per_rank=M, hidden=128, x_dtype="bf16",
                         recv_dtype=str(rng.choice(["bf16", "fp8"])), expand=expand,
                         expert_alignment=int(rng.choice([1, 1, 2, 4])) if expand else 1, compact=compact,
                         zero_padding=expand and bool(rng.random() < 0.5), sf_pack=False, recv_capacity=0)
    if expand:  # no repeated expert within a token
        idx = np.stack([np.stack([rng.permutation(E)[:K] for _ in range(T)]) for _ in range(R)]) \
            if T else np.zeros((R, 0, K), np.int64)
    else:
        idx = rng.integers(0, E, size=(R, T, K))
    idx = np.where(rng.random((R, T, K)) < 0.15, -1, idx).astype(np.int64)
    w = rng.random((R, T, K)).astype(np.float32)
    x = (rng.standard_normal((R, T, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return wl, idx, w, x


@pytest.mark.parametrize("seed", range(40))
def test_lane_rows_random_configurations(orc, seed):
    wl, idx, w, x = _random_case(seed)
    _check(orc, wl, idx, w, x, None)
