"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The bulk-copy dispatch waits on mbarriers for its own copies; each wait has a
round limit after which the kernel drains the copies in flight, latches a
timeout bit in the workspace and returns. ep_diag_wait_timeout runs that same
sequence on an mbarrier nothing completes (a copy of real data in flight), so
the host must read EP_ERR_TIMEOUT once, the bit must clear, and the context must
still run the path bit-exactly afterwards."""
import pytest
import torch

import combine_ep_get_02_gb300 as ep
import oracle
import workloads as W
from _harness import GpuRun, compare_dispatch, inputs

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_the_context_survives():
    wl = W.PARITY["direct_zipf"]
    cfg = ep.config_of(wl)
    ws = ep.alloc_workspace(cfg, "cuda")
    src = torch.arange(4096, dtype=torch.int32, device="cuda").to(torch.uint8)
    ep.ep_diag_wait_timeout(ws, src, 4096, 64)
    assert ep.ep_check_error(ws) == ep.EP_ERR_TIMEOUT
    assert ep.ep_check_error(ws) == ep.EP_OK          # read once, then cleared
    ep.ep_diag_wait_timeout(ws, None, 0, 0)             # nothing in flight, no rounds at all
    assert ep.ep_check_error(ws) == ep.EP_ERR_TIMEOUT

    # the same context still runs layout -> bulk-copy dispatch, bit-exact
    idx, w, x, sf = inputs(wl)
    st, olay = oracle.layout(wl, idx)
    assert st == 0
    run = GpuRun(wl, idx, w, x, sf, copy_path=2).layout().dispatch()
    assert run.status() == ep.EP_OK
    st, orec = oracle.dispatch(wl, olay, x, sf, idx, w)
    assert st == 0
    compare_dispatch(run, olay, orec)


def test_wait_timeout_rejects_bad_arguments():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    src = torch.zeros(8192, dtype=torch.uint8, device="cuda")
    for args in ((src, 4112, 1), (src, 24, 1), (None, 16, 1), (src[1:], 16, 1), (src, 16, (1 << 20) + 1)):
        with pytest.raises(ep.EpError):
            ep.ep_diag_wait_timeout(ws, *args)
    with pytest.raises(ep.EpError):
        ep.ep_diag_wait_timeout(ws[1:], src, 16, 1)
