"""GPU parity at the five full workload sizes, in the launch configuration the
benchmark times (all SMs, automatic prologue grid).

The whole layout is compared with the oracle element by element (it is cheap
on the CPU). Dispatch rows, their sidecars and combined outputs are compared on
a seeded sample of source tokens that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_02_gb300 as ep
import oracle
import workloads as W
from _harness import GpuRun, assert_layout_equal, inputs, oracle_combine_from_device_y, random_y, u16

pytestmark = pytest.mark.gpu

SAMPLE = 384


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_full_size(name):
    wl = W.WORKLOADS[name]
    idx, w, x, sf = inputs(wl)
    R, T, K, M, H = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.num_max_tokens_per_rank, wl.hidden
    L = wl.num_experts // R
    st, olay = oracle.layout(wl, idx)
    assert st == 0

    run = GpuRun(wl, idx, w, x, sf).layout().dispatch(zero=False)
    assert run.status() == ep.EP_OK
    assert_layout_equal(run.layout_np(), olay, wl.expand)

    rng = np.random.default_rng(1234)
    toks = np.sort(rng.choice(R * T, size=min(SAMPLE, R * T), replace=False))
    idx_np = idx.numpy().reshape(R * T, K)
    w_np = w.numpy().reshape(R * T, K)
    xv = x.reshape(R * T, H)
    xv = xv.view(torch.int16).numpy().view(np.uint16) if xv.dtype == torch.bfloat16 else xv.numpy()
    sfv = None if sf is None else sf.reshape(R * T, -1).numpy()
    recv = run.recv
    for tok in toks:
        s, t = divmod(int(tok), T)
        o = oracle.dispatch_token(wl, olay, s, t, xv[tok], None if sfv is None else sfv[tok],
                                  idx_np[tok], w_np[tok])
        for d, r in zip(o["hid_dst"], o["hid_row"]):
            g = int(olay["exp_region"][d]) + int(r) if wl.expand else int(d) * R * M + int(r)
            assert np.array_equal(u16(recv.recv_x[g]), o["hid"]), (tok, d)
            if wl.recv_dtype == "fp8":
                assert np.array_equal(recv.recv_sf[g].cpu().numpy().view(np.uint32),
                                      o["hid_sf"].view(np.uint32)), (tok, d)
        for i, (d, r) in enumerate(zip(o["meta_dst"], o["meta_row"])):
            assert recv.recv_topk_idx[d, r].cpu().numpy().tolist() == o["meta_idx"][i].tolist()
            assert np.array_equal(recv.recv_topk_weights[d, r].cpu().numpy().view(np.uint32),
                                  o["meta_w"][i].view(np.uint32))
            assert recv.recv_src_metadata[d, r].cpu().numpy().tolist() == o["meta_md"][i].tolist()

    identity = wl.y_kind == "identity" and wl.recv_dtype == "bf16"
    y = recv.recv_x if identity else random_y(wl, ep.ep_recv_rows(run.cfg), run.dev)
    run.combine(y)
    assert run.status() == ep.EP_OK
    got = u16(run.out.reshape(R * T, H)[torch.from_numpy(toks).to(run.dev)])
    exp = oracle_combine_from_device_y(wl, olay, idx, w, y, tokens=toks)
    assert np.array_equal(got, exp)

    # properties that hold at any size: every token's output is finite, and a
    # token without a valid lane gives +0
    out = run.out.float()
    assert torch.isfinite(out).all()
    none = (idx < 0).all(-1).to(run.dev)
    if none.any():
        assert (run.out[none].view(torch.int16) == 0).all()
