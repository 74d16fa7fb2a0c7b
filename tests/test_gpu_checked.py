"""The bounds-checked build of the library (libep_get_checked.so, -DEP_CHECKED).

Every row index the kernels compute (layout slots and expanded rows, dispatch
destination rows, sidecar rows, padding rows, combine gather rows) is tested
against its buffer before the access; one outside is skipped and latched as
EP_ERR_BOUNDS. With compute-sanitizer closed on this pool this is the check that
no index leaves its buffer:

- every parity case runs through the checked build with both copy paths, must
  report no bounds error and must still match the oracle bit for bit;
- a layout corrupted on the host (a token's slots or expanded rows pushed far
  past the receive buffer) must come back as EP_ERR_BOUNDS from dispatch and
  from combine, with every other token still exact. In the compact and packed
  layouts such a slot names a row block past the last, and the check comes
  before the receive prefix sums are read with it. Only the checked build is
  given such input: its checks sit in front of every access that uses them.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_02_gb300 as ep
import oracle
import workloads as W
from _harness import (GpuRun, assert_layout_equal, compare_dispatch, inputs,
                      oracle_combine_from_device_y, random_y, u16)
from test_gpu_parity import CASES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    ep.use_checked(True)
    yield
    ep.use_checked(False)


def _paths(wl):
    # the copy path matters only for rows that travel unchanged
    return (0,) if (wl.x_dtype, wl.recv_dtype) == ("bf16", "fp8") else (1, 2)


@pytest.mark.parametrize("name,copy_path", [(n, p) for n in sorted(CASES) for p in _paths(CASES[n])])
def test_parity_case_has_no_bounds_error(name, copy_path):
    wl = CASES[name]
    idx, w, x, sf = inputs(wl)
    st, olay = oracle.layout(wl, idx)
    assert st == 0
    run = GpuRun(wl, idx, w, x, sf, copy_path=copy_path).layout()
    assert run.status() == ep.EP_OK
    assert_layout_equal(run.layout_np(), olay, wl.expand)
    run.dispatch()
    assert run.status() == ep.EP_OK
    st, orec = oracle.dispatch(wl, olay, x, sf, idx, w)
    assert st == 0
    compare_dispatch(run, olay, orec)
    y = random_y(wl, ep.ep_recv_rows(run.cfg), run.dev)
    run.combine(y)
    assert run.status() == ep.EP_OK
    assert np.array_equal(u16(run.out).reshape(-1, wl.hidden), oracle_combine_from_device_y(wl, olay, idx, w, y))


@pytest.mark.parametrize("name,copy_path", [("direct_zipf", 1), ("direct_zipf", 2), ("dsv3_fp8", 0),
                                            ("expanded", 1), ("expanded", 2),
                                            ("direct_zipf_compact", 1), ("hybrid_compact", 2),
                                            ("hybrid_packed", 1), ("dsv3_fp8_packed_rows", 0)])
def test_corrupted_layout_is_reported_not_written(name, copy_path):
    wl = W.PARITY[name]
    R, T, K = wl.num_ranks, wl.num_tokens, wl.num_topk
    idx, w, x, sf = inputs(wl)
    st, olay = oracle.layout(wl, idx)
    assert st == 0
    run = GpuRun(wl, idx, w, x, sf, copy_path=copy_path).layout()
    assert run.status() == ep.EP_OK
    # token (1, 5): every lane's row pushed ten million rows past its place
    bad_tok = 1 * T + 5
    key = "exp_pos" if wl.expand else "slot_map"
    table = getattr(run.lay, key).view(-1, K)
    assert bool((table[bad_tok] >= 0).any())
    table[bad_tok] = torch.where(table[bad_tok] >= 0, table[bad_tok] + 10_000_000, table[bad_tok])

    run.dispatch()
    assert run.status() == ep.EP_ERR_BOUNDS
    assert run.status() == ep.EP_OK  # read once, then cleared
    y = random_y(wl, ep.ep_recv_rows(run.cfg), run.dev)
    run.combine(y)
    assert run.status() == ep.EP_ERR_BOUNDS

    # the bad token's lanes were dropped; every other token is exact
    good = np.setdiff1d(np.arange(R * T), [bad_tok])
    got = u16(run.out).reshape(-1, wl.hidden)
    exp = oracle_combine_from_device_y(wl, olay, idx, w, y, tokens=good)
    assert np.array_equal(got[good], exp)
    bad_lanes = idx.numpy().reshape(-1, K)[bad_tok] >= 0
    if bad_lanes.any():  # no valid lane left: the token sums to +0
        assert np.all(got[bad_tok] == 0)
