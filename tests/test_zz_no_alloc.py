"""The allocation-free layout entry point, for callers that may not allocate
device memory (for example engine plugins handed only their buffers): it must
give exactly the layout of ep_get_dispatch_layout, call after call, while its
scratch lives in a fixed array inside the library instead of a workspace; the
device's free memory must not move across its calls; and the device-detected
errors it latches in that array must reach ep_check_error_noalloc.

Kept in a file of its own that pytest collects last."""
import pytest
import torch

import combine_ep_get_02_gb300 as ep
import workloads as W
from _harness import GpuRun, assert_layout_equal, inputs

pytestmark = pytest.mark.gpu


def _poison(lay):
    for f in ("num_tokens_per_rank", "num_tokens_per_expert", "slot_map", "recv_cnt", "recv_psum",
              "exp_cnt", "exp_base", "exp_region", "exp_pos"):
        t = getattr(lay, f)
        if t is not None:
            t.fill_(-7)
    lay.is_token_in_rank.fill_(0xAB)


@pytest.mark.parametrize("name", ["direct_zipf", "hybrid_rowform", "expanded"])
def test_noalloc_layout_matches_the_workspace_entry_point(name):
    wl = W.PARITY[name]
    idx, w, x, sf = inputs(wl)
    ref = GpuRun(wl, idx, w, x, sf).layout()
    assert ref.status() == ep.EP_OK
    expect = ref.layout_np()
    assert ep.ep_workspace_bytes(ref.cfg) <= 1 << 20
    lay = ep.alloc_layout(ref.cfg, ref.dev)
    for _ in range(2):  # two calls in a row share the library's scratch
        _poison(lay)
        ep.ep_get_dispatch_layout_noalloc(ref.cfg, ref.idx, lay)
        torch.cuda.synchronize()
        got = {k: getattr(lay, k).cpu().numpy() for k in expect}
        assert_layout_equal(got, expect, wl.expand)
    # and the dispatch that consumes it gives the same rows
    ref.dispatch()
    other = ep.alloc_recv(ref.cfg, ref.dev, zero=True)
    ep.ep_dispatch(ref.cfg, lay, ref.x, ref.sf, ref.idx, ref.w, other, ref.ws)
    torch.cuda.synchronize()
    assert torch.equal(ref.recv.recv_x.view(torch.int16), other.recv_x.view(torch.int16))


def test_noalloc_allocates_nothing():
    """Free device memory (cudaMemGetInfo) is the same before and after a run of
    calls: the scratch is the library's static array, nothing is allocated."""
    wl = W.PARITY["expanded"]
    idx, w, x, sf = inputs(wl)
    cfg = ep.config_of(wl)
    lay = ep.alloc_layout(cfg, "cuda")
    idx_d = idx.to("cuda")
    ep.ep_get_dispatch_layout_noalloc(cfg, idx_d, lay)  # first call: the module is loaded
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        ep.ep_get_dispatch_layout_noalloc(cfg, idx_d, lay)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert ep.ep_check_error_noalloc() == ep.EP_OK


def test_noalloc_reports_bad_topk_values():
    """A top-k value outside [-1, E) is masked, as in the workspace entry point,
    and reported once through ep_check_error_noalloc."""
    wl = W.Workload("bad_noalloc", 1, 4, 16, 2, 30, 30, 128)
    idx, w, x, sf = inputs(wl)
    idx = idx.clone()
    idx[1, 3, 0] = 16
    ref = GpuRun(wl, idx, w, x, sf).layout()
    assert ref.status() == ep.EP_ERR_BAD_TOPK
    lay = ep.alloc_layout(ref.cfg, ref.dev)
    _poison(lay)
    ep.ep_get_dispatch_layout_noalloc(ref.cfg, ref.idx, lay)
    assert ep.ep_check_error_noalloc() == ep.EP_ERR_BAD_TOPK
    assert ep.ep_check_error_noalloc() == ep.EP_OK  # read once, then cleared
    got = {k: getattr(lay, k).cpu().numpy() for k in ref.layout_np()}
    assert_layout_equal(got, ref.layout_np(), False)


def test_noalloc_rejects_configs_beyond_its_scratch():
    # expanded: the scratch holds one int32 per (source rank, expert) after a
    # 256-byte header; 64 ranks x 4096 experts needs 1 MiB + 256 bytes
    cfg = ep.Config(1, 64, 4096, 8, 16, 16, 128, expand=1)
    assert ep.ep_workspace_bytes(cfg) > 1 << 20
    lay = ep.alloc_layout(ep.Config(1, 1, 1, 1, 0, 1, 8), "cuda")  # never written
    with pytest.raises(ep.EpError) as e:
        ep.ep_get_dispatch_layout_noalloc(cfg, torch.empty(0, dtype=torch.int64, device="cuda"), lay)
    assert e.value.status == ep.EP_ERR_WORKSPACE
    bad = ep.Config(1, 16, 250, 8, 16, 16, 128)  # experts not a multiple of the ranks
    with pytest.raises(ep.EpError) as e:
        ep.ep_get_dispatch_layout_noalloc(bad, torch.empty(0, dtype=torch.int64, device="cuda"), lay)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
