"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and the CPU oracle on the same seeded inputs, then compare."""
from __future__ import annotations

import numpy as np
import torch

import combine_ep_get_02_gb300 as ep
import oracle
import workloads as W

LAYOUT_KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "slot_map",
               "recv_cnt", "recv_psum", "recv_region")
EXPAND_KEYS = ("exp_cnt", "exp_base", "exp_region", "exp_pos")


def u16(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy().view(np.uint16) if t.dtype == torch.int16 else t.numpy()


def inputs(wl):
    idx, w = W.routing(wl)
    x, sf = W.hidden(wl)
    return idx, w, x, sf


class GpuRun:
    """One layout -> dispatch (-> combine) of a workload on the current device."""

    def __init__(self, wl, idx, w, x, sf, dev="cuda", **cfg_over):
        self.wl = wl
        self.cfg = ep.config_of(wl, **cfg_over)
        self.dev = dev
        self.idx = idx.to(dev)
        self.w = w.to(dev)
        self.x = x.to(dev)
        self.sf = None if sf is None else sf.to(dev)
        self.ws = ep.alloc_workspace(self.cfg, dev)
        self.lay = ep.alloc_layout(self.cfg, dev)
        self.recv = None
        self.out = None

    def layout(self):
        ep.ep_get_dispatch_layout(self.cfg, self.idx, self.lay, self.ws)
        return self

    def dispatch(self, zero=True):
        if self.recv is None:
            self.recv = ep.alloc_recv(self.cfg, self.dev, zero=zero)
        ep.ep_dispatch(self.cfg, self.lay, self.x, self.sf, self.idx, self.w, self.recv, self.ws)
        return self

    def combine(self, y):
        self.out = torch.empty(self.wl.num_ranks, self.wl.num_tokens, self.wl.hidden,
                               dtype=torch.bfloat16, device=self.dev)
        ep.ep_combine(self.cfg, self.lay, y, self.idx, self.w, self.out, self.ws)
        return self

    def status(self):
        return ep.ep_check_error(self.ws)

    def layout_np(self):
        d = {k: getattr(self.lay, k).cpu().numpy() for k in LAYOUT_KEYS}
        if self.wl.expand:
            d.update({k: getattr(self.lay, k).cpu().numpy() for k in EXPAND_KEYS})
        return d


def assert_layout_equal(got, exp, expand):
    keys = LAYOUT_KEYS + (EXPAND_KEYS if expand else ())
    for k in keys:
        assert got[k].shape == exp[k].shape, k
        if not np.array_equal(got[k], exp[k]):
            bad = np.argwhere(got[k] != exp[k])
            raise AssertionError(f"{k}: {len(bad)} mismatches, first at {bad[0].tolist()}: "
                                 f"got {got[k][tuple(bad[0])]} expected {exp[k][tuple(bad[0])]}")


def filled_rows(wl, olay, idx):
    """(recv_x rows, sidecar rows) the oracle fills: its lane rows, deduplicated."""
    st, hid, side = oracle.lane_rows(wl, olay, idx)
    return np.unique(hid[hid >= 0]), np.unique(side[side >= 0])


def compare_dispatch(run: GpuRun, olay, orec):
    wl = run.wl
    idx = run.idx.cpu()
    hid, side = filled_rows(wl, olay, idx)
    hid_t = torch.from_numpy(hid).to(run.dev)
    side_t = torch.from_numpy(side).to(run.dev)
    got_x = u16(run.recv.recv_x.index_select(0, hid_t))
    assert np.array_equal(got_x, orec["recv_x"][hid]), "recv_x differs"
    if wl.recv_dtype == "fp8":
        got_sf = run.recv.recv_sf.index_select(0, hid_t).cpu().numpy()
        assert np.array_equal(got_sf.view(np.uint32), orec["recv_sf"][hid].view(np.uint32)), "recv_sf differs"
    K = wl.num_topk
    for name, width in (("recv_topk_idx", K), ("recv_topk_weights", K), ("recv_src_metadata", K + 2)):
        g = getattr(run.recv, name).reshape(-1, width).index_select(0, side_t).cpu().numpy()
        e = orec[name][side]
        assert np.array_equal(g.view(np.uint8), e.view(np.uint8)), f"{name} differs"
    return hid, side


def random_y(wl, rows, dev):
    return W.expert_outputs(wl, rows, device=str(dev))


def oracle_combine_from_device_y(wl, olay, idx, w, y_dev, tokens=None):
    """Oracle combine of the listed tokens (flat s*T+t; all if None), reading
    the expert outputs the lanes need from the device tensor y_dev."""
    rows = oracle.global_rows(wl, olay, idx).reshape(-1, wl.num_topk)
    wf = (w.numpy() if hasattr(w, "numpy") else w).reshape(-1, wl.num_topk)
    if tokens is not None:
        rows = rows[tokens]
        wf = wf[tokens]
    uniq, inv = np.unique(rows[rows >= 0], return_inverse=True)
    compact = np.full(rows.shape, -1, np.int64)
    compact[rows >= 0] = inv
    ys = u16(y_dev.index_select(0, torch.from_numpy(uniq).to(y_dev.device))) if uniq.size else \
        np.zeros((0, wl.hidden), np.uint16)
    return oracle.combine_gathered(compact, ys, wf)
