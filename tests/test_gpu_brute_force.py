"""GPU == oracle on every routing of tiny shapes.

Every assignment of {-1, 0..E-1} to one source's 3 tokens x 2 lanes (E = 4:
5^6 = 15,625 routings) goes through layout -> dispatch -> combine on the GPU
and through the oracle. One call carries R routings, one per source rank, so
ceil(15,625 / R) calls cover the enumeration; the layouts, every receive row,
the sidecars of the filled rows and the combined tokens must match bit for
bit, with unchanged rows moved both by register copies and by bulk copies.
Expanded layouts enumerate the routings without an expert repeated inside
a token (21^3 = 9,261), a repeat being an error there.

The oracle itself is pinned on the same enumeration against the sort-based
statement of the slot rule (PR #753, Approach: the kernel-side order equals the
post-hoc sort by source token).
"""
import itertools

import numpy as np
import pytest
import torch

import combine_ep_get_02_gb300 as ep
import oracle
import workloads as W
from _harness import assert_layout_equal, u16

pytestmark = pytest.mark.gpu

T, K, E = 3, 2, 4

SHAPES = {
    # R = 2 direct: 2 experts per rank, so lanes of one token can share a row
    "direct_r2": W.Workload("bf_direct_r2", 1, 2, E, K, T, 4, 8),
    # R = 4 direct, one expert per rank, M = T (no free rows between sources)
    "direct_r4": W.Workload("bf_direct_r4", 1, 4, E, K, T, T, 8),
    # 2 scale-out x 2 scale-up row form
    "hybrid_2x2": W.Workload("bf_hybrid_2x2", 2, 2, E, K, T, 4, 8),
    # compact receive rows
    "compact_r2": W.Workload("bf_compact_r2", 1, 2, E, K, T, 5, 8, compact=1),
    # packed receive rows (destinations back to back), direct and hybrid
    "packed_r2": W.Workload("bf_packed_r2", 1, 2, E, K, T, 5, 8, compact=2),
    "packed_hybrid_2x2": W.Workload("bf_packed_hybrid_2x2", 2, 2, E, K, T, 4, 8, compact=2),
    # fused bf16 -> FP8 cast with fp32 scales, hybrid
    "fp8_hybrid": W.Workload("bf_fp8_hybrid", 2, 2, E, K, T, T, 128, recv_dtype="fp8"),
    # expanded per-expert blocks, alignment 2, zeroed padding
    "expanded_a2": W.Workload("bf_expanded_a2", 1, 2, E, K, T, T, 8, expand=True,
                              expert_alignment=2, zero_padding=True),
}


def routings(expand):
    vals = range(-1, E)
    all_ = np.array(list(itertools.product(vals, repeat=T * K)), np.int64).reshape(-1, T, K)
    if expand:
        dup = (all_[:, :, 0] == all_[:, :, 1]) & (all_[:, :, 0] >= 0)
        all_ = all_[~dup.any(axis=1)]
    return all_


def test_enumeration_sizes():
    assert routings(False).shape == (15625, T, K)
    assert routings(True).shape == (9261, T, K)


CASES = [(name, path) for name in SHAPES for path in ((0,) if SHAPES[name].recv_dtype == "fp8" else (1, 2))]


@pytest.mark.parametrize("name,copy_path", CASES)
def test_every_routing_matches_the_oracle(name, copy_path):
    wl = SHAPES[name]
    R, M, H = wl.num_ranks, wl.num_max_tokens_per_rank, wl.hidden
    cases = routings(wl.expand)
    n_calls = -(-len(cases) // R)
    # wrap around so the last call is full; every routing appears at least once
    order = np.arange(n_calls * R) % len(cases)

    cfg = ep.config_of(wl, copy_path=copy_path)
    dev = "cuda"
    _, w = W.routing(wl)                 # fp32 weights [R, T, K]; masked lanes are skipped
    x, sf = W.hidden(wl)
    w_d, x_d = w.to(dev), x.to(dev)
    sf_d = None if sf is None else sf.to(dev)
    ws = ep.alloc_workspace(cfg, dev)
    lay = ep.alloc_layout(cfg, dev)
    recv = ep.alloc_recv(cfg, dev)
    rows_cap = max(ep.ep_recv_rows(cfg), 1)
    y = W.expert_outputs(wl.replace(y_kind="random"), rows_cap, device=dev)
    y_h = u16(y)
    out = torch.empty(R, T, H, dtype=torch.bfloat16, device=dev)
    idx_d = torch.empty(R, T, K, dtype=torch.int64, device=dev)
    row_bytes = H * (1 if wl.recv_dtype == "fp8" else 2)
    side_tensors = [("recv_topk_idx", K), ("recv_topk_weights", K), ("recv_src_metadata", K + 2)]

    for c in range(n_calls):
        idx = torch.from_numpy(cases[order[c * R:(c + 1) * R]].copy())
        idx_d.copy_(idx)
        for t in (recv.recv_x, recv.recv_sf, recv.recv_topk_idx, recv.recv_topk_weights,
                  recv.recv_src_metadata):
            if t is not None:
                t.view(torch.uint8).fill_(0xFF)
        ep.ep_get_dispatch_layout(cfg, idx_d, lay, ws)
        ep.ep_dispatch(cfg, lay, x_d, sf_d, idx_d, w_d, recv, ws)
        ep.ep_combine(cfg, lay, y, idx_d, w_d, out, ws)
        assert ep.ep_check_error(ws) == ep.EP_OK, (name, c)

        st, olay = oracle.layout(wl, idx)
        assert st == 0
        got = {k: getattr(lay, k).cpu().numpy() for k in
               ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "slot_map",
                "recv_cnt", "recv_psum", "recv_region")}
        if wl.expand:
            got.update({k: getattr(lay, k).cpu().numpy() for k in
                        ("exp_cnt", "exp_base", "exp_region", "exp_pos")})
        assert_layout_equal(got, olay, wl.expand)

        st, orec = oracle.dispatch(wl, olay, x, sf, idx, w, fill=0xFF)
        assert st == 0
        rows = int(olay["exp_region"][-1]) if wl.expand else orec["recv_x"].shape[0]
        g = recv.recv_x[:rows].contiguous().view(torch.uint8).cpu().numpy().reshape(rows, row_bytes)
        e = np.ascontiguousarray(orec["recv_x"][:rows]).view(np.uint8).reshape(rows, row_bytes)
        assert np.array_equal(g, e), (name, c)
        if wl.recv_dtype == "fp8":
            assert np.array_equal(recv.recv_sf[:rows].cpu().numpy().view(np.uint32),
                                  orec["recv_sf"][:rows].view(np.uint32)), (name, c)
        # whole sidecar buffers: written rows equal, the rest still 0xFF on both sides
        for key, width in side_tensors:
            gs = getattr(recv, key).reshape(-1, width).cpu().numpy().view(np.uint8)
            es = orec[key].view(np.uint8)
            assert np.array_equal(gs, es), (name, c, key)

        exp = oracle.combine_gathered(oracle.global_rows(wl, olay, idx).reshape(-1, K), y_h,
                                      w.numpy().reshape(-1, K))
        assert np.array_equal(u16(out).reshape(-1, H), exp), (name, c)
