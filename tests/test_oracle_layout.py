"""Pins of the oracle's dispatch layout (slots, counts, expanded positions).

Sources: PR #753 (Motivation, Approach, "Direct vs hybrid dispatch"): slot =
row_base_idx * num_max_tokens_per_rank + the sender's running count of
deduplicated entries to that destination in token order; direct row base =
the source rank; hybrid row form: segment = source scale-up rank, offset =
source scale-out rank * num_max_tokens_per_rank + row-local slot; the
kernel-side order equals the post-hoc sort by source token (source rank, then
token). PR #544 title: a token counts once per destination rank.

The checks restate the rule in other forms than the oracle's running counter:
hand-worked examples, a set-membership count over earlier tokens, a sort of the
received entries, and brute force over every routing of a tiny case.
"""
import itertools
from types import SimpleNamespace

import numpy as np
import pytest


def wl_of(n_so, n_su, E, K, T, M=None, H=128, expand=False, align=1):
    return SimpleNamespace(n_so=n_so, n_su=n_su, num_ranks=n_so * n_su, num_experts=E, num_topk=K,
                           num_tokens=T, num_max_tokens_per_rank=M if M is not None else T,
                           hidden=H, x_dtype="bf16", recv_dtype="bf16", expand=expand,
                           expert_alignment=align)


HAND_IDX = np.array([[[0, 3], [1, 0], [2, -1]],
                     [[3, 2], [0, -1], [-1, -1]]], np.int64)


def test_hand_worked_direct(orc):
    # R=2 direct, E=4 (2 experts per rank), K=2, T=M=3.
    # source 0: t0 -> d0 (e0), d1 (e3) ; t1 -> d0 (e1, e0 shares the row) ; t2 -> d1 (e2)
    # source 1 (row base 1*3): t0 -> d1 (e3, e2 shares) ; t1 -> d0 (e0)
    st, lay = orc.layout(wl_of(1, 2, 4, 2, 3), HAND_IDX)
    assert st == 0
    assert lay["slot_map"].tolist() == [[[0, 0], [1, 1], [1, -1]],
                                        [[3, 3], [3, -1], [-1, -1]]]
    assert lay["num_tokens_per_rank"].tolist() == [[2, 2], [1, 1]]
    assert lay["num_tokens_per_expert"].tolist() == [[2, 1, 1, 1], [1, 0, 1, 1]]
    assert lay["is_token_in_rank"].tolist() == [[[1, 1], [1, 0], [0, 1]],
                                                [[0, 1], [1, 0], [0, 0]]]
    assert lay["recv_cnt"].tolist() == [[2, 1], [2, 1]]
    assert lay["recv_psum"].tolist() == [[2, 3], [2, 3]]


def test_hand_worked_hybrid_row_bases(orc):
    # 2 scale-out x 2 scale-up; rank r = so*2 + su. Row block of a source inside a
    # destination region = su*n_so + so: r0 -> 0, r1 -> 2, r2 -> 1, r3 -> 3 (M=2 rows each).
    idx = np.array([[[0], [1]], [[0], [-1]], [[1], [0]], [[0], [0]]], np.int64)  # E=4: d = e
    st, lay = orc.layout(wl_of(2, 2, 4, 1, 2), idx)
    assert st == 0
    # r0: t0 -> d0 row 0, t1 -> d1 row 0 (its first entry to d1); r1 (block 2): row 4;
    # r2 (block 1): t0 -> d1 row 2, t1 -> d0 row 2; r3 (block 3): rows 6, 7 of d0
    assert lay["slot_map"][:, :, 0].tolist() == [[0, 0], [4, -1], [2, 2], [6, 7]]
    # prefix sums of the per-source counts in row-block order (r0, r2, r1, r3)
    assert lay["recv_cnt"][0].tolist() == [1, 1, 1, 2]
    assert lay["recv_psum"][0].tolist() == [1, 2, 3, 5]


def test_hand_worked_expanded(orc):
    # same routing as the direct example, expanded: per destination, per local
    # expert, lanes in (source, token) order.
    #   e0: (s0,t0), (s0,t1), (s1,t1) -> 0,1,2 ; e1: (s0,t1) -> 3   (d0 blocks [0,3,4])
    #   e2: (s0,t2), (s1,t0) -> 0,1 ; e3: (s0,t0), (s1,t0) -> 2,3    (d1 blocks [0,2,4])
    st, lay = orc.layout(wl_of(1, 2, 4, 2, 3, expand=True), HAND_IDX)
    assert st == 0
    assert lay["exp_cnt"].tolist() == [[3, 1], [2, 2]]
    assert lay["exp_base"].tolist() == [[0, 3, 4], [0, 2, 4]]
    assert lay["exp_region"].tolist() == [0, 4, 8]
    assert lay["exp_pos"].tolist() == [[[0, 2], [3, 1], [0, -1]],
                                       [[3, 1], [2, -1], [-1, -1]]]
    # alignment 4 pads every block to a multiple of 4 rows
    st, lay = orc.layout(wl_of(1, 2, 4, 2, 3, expand=True, align=4), HAND_IDX)
    assert lay["exp_base"].tolist() == [[0, 4, 8], [0, 4, 8]]
    assert lay["exp_region"].tolist() == [0, 8, 16]
    assert lay["exp_pos"].tolist() == [[[0, 4], [4, 1], [0, -1]],
                                       [[5, 1], [2, -1], [-1, -1]]]


def row_block(wl, s):
    if wl.n_so == 1:
        return s
    return (s % wl.n_su) * wl.n_so + s // wl.n_su


def dst_sets(wl, idx):
    """D(s,t): the set of destination ranks of the valid lanes."""
    L = wl.num_experts // wl.num_ranks
    R, T, K = idx.shape
    return [[{int(e) // L for e in idx[s, t] if e >= 0} for t in range(T)] for s in range(R)]


def expected_slots_by_counting(wl, idx):
    """slot(s,t,k) = row_block(s)*M + |{t' < t : d in D(s,t')}|, d = destination of lane k."""
    L = wl.num_experts // wl.num_ranks
    R, T, K = idx.shape
    D = dst_sets(wl, idx)
    out = np.full((R, T, K), -1, np.int64)
    for s in range(R):
        for t in range(T):
            for k in range(K):
                e = idx[s, t, k]
                if e < 0:
                    continue
                d = int(e) // L
                out[s, t, k] = row_block(wl, s) * wl.num_max_tokens_per_rank + \
                    sum(1 for tp in range(t) if d in D[s][tp])
    return out


def expected_slots_by_sorting(wl, idx):
    """The post-hoc-sort view: sort each destination's entries by (source, token);
    within a source, the i-th entry sits at row_block(source)*M + i."""
    L = wl.num_experts // wl.num_ranks
    R, T, K = idx.shape
    entries = {d: sorted({(s, t) for s in range(R) for t in range(T)
                          for e in idx[s, t] if e >= 0 and int(e) // L == d}) for d in range(R)}
    row = {}
    for d, lst in entries.items():
        for s, grp in itertools.groupby(lst, key=lambda st: st[0]):
            for i, (_, t) in enumerate(grp):
                row[(s, t, d)] = row_block(wl, s) * wl.num_max_tokens_per_rank + i
    out = np.full((R, T, K), -1, np.int64)
    for s in range(R):
        for t in range(T):
            for k in range(K):
                if idx[s, t, k] >= 0:
                    out[s, t, k] = row[(s, t, int(idx[s, t, k]) // L)]
    return out


def random_idx(rng, wl, mask_frac=0.1):
    R, T, K, E = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.num_experts
    idx = np.stack([[rng.choice(E, K, replace=False) for _ in range(T)] for _ in range(R)]).astype(np.int64)
    idx[rng.random(idx.shape) < mask_frac] = -1
    return idx


@pytest.mark.parametrize("shape", [(1, 4, 16, 3, 9, 9), (2, 2, 8, 4, 7, 11), (1, 8, 32, 4, 12, 12),
                                   (4, 2, 16, 2, 5, 5), (1, 3, 3, 3, 6, 6)])
def test_slots_match_counting_and_sorting(orc, shape):
    n_so, n_su, E, K, T, M = shape
    wl = wl_of(n_so, n_su, E, K, T, M)
    rng = np.random.default_rng(hash(shape) & 0xFFFF)
    for _ in range(5):
        idx = random_idx(rng, wl)
        st, lay = orc.layout(wl, idx)
        assert st == 0
        a = expected_slots_by_counting(wl, idx)
        b = expected_slots_by_sorting(wl, idx)
        assert np.array_equal(a, b)
        assert np.array_equal(lay["slot_map"], a)


def check_invariants(wl, idx, lay):
    R, T, K = idx.shape
    L = wl.num_experts // R
    M = wl.num_max_tokens_per_rank
    D = dst_sets(wl, idx)
    ntpr, itir, slot = lay["num_tokens_per_rank"], lay["is_token_in_rank"], lay["slot_map"]
    for s in range(R):
        assert ntpr[s].sum() == sum(len(D[s][t]) for t in range(T))
        assert lay["num_tokens_per_expert"][s].sum() == int((idx[s] >= 0).sum())
        for t in range(T):
            assert itir[s, t].sum() == len(D[s][t])
            assert {d for d in range(R) if itir[s, t, d]} == D[s][t]
        # the filled rows of (s, d) are exactly [row_block*M, row_block*M + count)
        for d in range(R):
            rows = sorted({int(slot[s, t, k]) for t in range(T) for k in range(K)
                           if idx[s, t, k] >= 0 and int(idx[s, t, k]) // L == d})
            base = row_block(wl, s) * M
            assert rows == list(range(base, base + int(ntpr[s, d])))
            assert ntpr[s, d] <= M
    assert np.array_equal(lay["recv_cnt"], ntpr.T)
    assert np.array_equal(lay["recv_psum"][:, -1], ntpr.sum(0))
    assert np.all(np.diff(lay["recv_psum"], axis=1) >= 0)
    # lanes of one token to one destination share one row; masked lanes are -1
    assert np.all((slot < 0) == (idx < 0))
    if wl.expand:
        for d in range(R):
            n_in = int(((idx >= 0) & (idx // L == d)).sum())
            assert lay["exp_cnt"][d].sum() == n_in


@pytest.mark.parametrize("shape", [(1, 2, 4, 2), (2, 2, 4, 2), (1, 4, 4, 2)])
def test_brute_force_every_routing_of_source0(orc, shape):
    """Every assignment of {-1, 0..E-1} to source 0's 3 tokens x 2 lanes (5^6 cases),
    the other sources fixed: oracle == sort-based rule, and all invariants hold."""
    n_so, n_su, E, K = shape
    T = 3
    wl = wl_of(n_so, n_su, E, K, T)
    R = wl.num_ranks
    rng = np.random.default_rng(7)
    base = rng.integers(-1, E, (R, T, K)).astype(np.int64)
    vals = list(range(-1, E))
    n = 0
    for combo in itertools.product(vals, repeat=T * K):
        idx = base.copy()
        idx[0] = np.array(combo, np.int64).reshape(T, K)
        st, lay = orc.layout(wl, idx)
        assert st == 0
        exp = expected_slots_by_sorting(wl, idx)
        assert np.array_equal(lay["slot_map"], exp), (combo,)
        if n % 97 == 0:
            check_invariants(wl, idx, lay)
        n += 1
    assert n == len(vals) ** (T * K)


@pytest.mark.parametrize("shape", [(1, 16, 256, 8, 40, 40), (4, 8, 256, 8, 30, 32), (1, 8, 64, 6, 33, 50)])
def test_invariants_generated_routing(orc, shape):
    import workloads as W
    n_so, n_su, E, K, T, M = shape
    wl = W.Workload("t", n_so, n_su, E, K, T, M, 128, routing="zipf", mask_frac=0.05)
    idx, _ = W.routing(wl)
    idx = idx.numpy()
    st, lay = orc.layout(wl, idx)
    assert st == 0
    check_invariants(wl, idx, lay)
    assert np.array_equal(lay["slot_map"], expected_slots_by_sorting(wl, idx))


def test_hybrid_is_a_fixed_permutation_of_direct(orc):
    rng = np.random.default_rng(3)
    hyb = wl_of(4, 2, 32, 4, 20, 24)
    dire = wl_of(1, 8, 32, 4, 20, 24)
    M = 24
    for _ in range(5):
        idx = random_idx(rng, hyb)
        _, lh = orc.layout(hyb, idx)
        _, ld = orc.layout(dire, idx)
        s = np.arange(8)[:, None, None]
        rb = np.array([row_block(hyb, r) for r in range(8)])[:, None, None]
        expect = np.where(ld["slot_map"] >= 0, ld["slot_map"] - s * M + rb * M, -1)
        assert np.array_equal(lh["slot_map"], expect)
        assert np.array_equal(lh["num_tokens_per_rank"], ld["num_tokens_per_rank"])


def expected_positions_by_sorting(wl, idx):
    R, T, K = idx.shape
    L = wl.num_experts // R
    A = wl.expert_alignment
    cnt = np.zeros(wl.num_experts, np.int64)
    for e in idx[idx >= 0]:
        cnt[e] += 1
    pos = np.full((R, T, K), -1, np.int64)
    for e in range(wl.num_experts):
        d, j = divmod(e, L)
        start = sum(-(-cnt[d * L + jj] // A) * A for jj in range(j))
        lanes = sorted((s, t, k) for s in range(R) for t in range(T) for k in range(K) if idx[s, t, k] == e)
        for i, (s, t, k) in enumerate(lanes):
            pos[s, t, k] = start + i
    return pos


@pytest.mark.parametrize("align", [1, 4, 128])
def test_expanded_positions_by_sorting(orc, align):
    rng = np.random.default_rng(align)
    wl = wl_of(1, 4, 16, 3, 21, 25, expand=True, align=align)
    for _ in range(4):
        idx = random_idx(rng, wl, 0.15)
        st, lay = orc.layout(wl, idx)
        assert st == 0
        assert np.array_equal(lay["exp_pos"], expected_positions_by_sorting(wl, idx))
        check_invariants(wl, idx, lay)
        L = wl.num_experts // wl.num_ranks
        # blocks are aligned and regions are concatenated in rank order
        assert np.all(lay["exp_base"] % align == 0)
        assert lay["exp_region"][-1] == lay["exp_base"][:, -1].sum()
        assert lay["exp_region"][-1] <= orc.recv_rows(wl)
        # every position is unique inside its destination region
        d = np.where(idx >= 0, idx // L, -1)
        glob = lay["exp_region"][np.maximum(d, 0)] + lay["exp_pos"]
        g = glob[idx >= 0]
        assert len(np.unique(g)) == g.size


def test_errors(orc):
    wl = wl_of(1, 2, 4, 2, 3)
    bad = HAND_IDX.copy()
    bad[0, 1, 0] = 4  # >= E
    assert orc.layout(wl, bad)[0] == orc.BAD_TOPK
    bad = HAND_IDX.copy()
    bad[1, 2, 1] = -2
    st, lay = orc.layout(wl, bad)
    assert st == orc.BAD_TOPK and lay["slot_map"][1, 2, 1] == -1
    dup = HAND_IDX.copy()
    dup[0, 0] = [1, 1]  # repeated expert: fine in the row form, an error when expanded
    assert orc.layout(wl, dup)[0] == 0
    assert orc.layout(wl_of(1, 2, 4, 2, 3, expand=True), dup)[0] == orc.BAD_TOPK
    assert orc.layout(wl_of(1, 2, 4, 2, 3, M=2), HAND_IDX)[0] == orc.INVALID  # T > M
    assert orc.layout(wl_of(1, 3, 4, 2, 3), np.zeros((3, 3, 2), np.int64))[0] == orc.INVALID  # E % R
    w = wl_of(1, 2, 4, 2, 3)
    w.x_dtype, w.recv_dtype = "fp8", "bf16"
    assert orc.layout(w, HAND_IDX)[0] == orc.UNSUPPORTED


def test_empty_and_single_token(orc):
    wl = wl_of(1, 4, 8, 2, 0, 4)
    st, lay = orc.layout(wl, np.zeros((4, 0, 2), np.int64))
    assert st == 0 and lay["num_tokens_per_rank"].sum() == 0 and np.all(lay["recv_psum"] == 0)
    wl = wl_of(1, 4, 8, 2, 1, 4)
    idx = np.array([[[7, 6]], [[0, -1]], [[-1, -1]], [[2, 5]]], np.int64)
    st, lay = orc.layout(wl, idx)
    # direct: source s owns rows [s*M, s*M + M) of every destination region
    assert lay["slot_map"][:, 0].tolist() == [[0, 0], [4, -1], [-1, -1], [12, 12]]


def test_golden_fixtures_reproduce(orc):
    """The stored fixtures (written by tests/golden/make_golden.py from the
    oracle) still come out of the oracle unchanged."""
    import glob
    import json
    import os
    paths = sorted(glob.glob(os.path.join(os.path.dirname(__file__), "golden", "*.json")))
    assert len(paths) >= 3
    for p in paths:
        doc = json.load(open(p))
        c = doc["config"]
        wl = wl_of(c["n_so"], c["n_su"], c["num_experts"], c["num_topk"], c["num_tokens"],
                   c["num_max_tokens_per_rank"], expand=c["expand"], align=c["expert_alignment"])
        idx = np.array(doc["topk_idx"], np.int64)
        st, lay = orc.layout(wl, idx)
        assert st == 0
        for k, v in lay.items():
            assert np.array_equal(v, np.array(doc[k], v.dtype)), (p, k)
        assert np.array_equal(lay["slot_map"], expected_slots_by_sorting(wl, idx))
