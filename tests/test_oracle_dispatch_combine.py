"""Pins of the oracle's dispatch rows and combine reduction.

Dispatch (PR #753 Approach; PR #690 review of the copy epilogue): every
deduplicated (token, destination) entry receives the token's hidden row
unchanged (bf16 copy), or its FP8 cast with per-128-column scales; pre-cast FP8
rows and their scales travel verbatim; the sidecar rows carry the routing and
the source metadata.

Combine: combine(dispatch(x)) with identity experts equals the weight sum
times x (to one bf16 ulp); a single lane with weight 1 returns x exactly;
power-of-two weights are exact; zero expert outputs give +0.
"""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import workloads as W


def small(name, **kw):
    return W.PARITY[name].replace(**kw)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def dedup_entries(wl, idx, slot):
    """(s, t, d, row) of every deduplicated entry: the first lane per destination."""
    L = wl.num_experts // wl.num_ranks
    R, T, K = idx.shape
    out = []
    for s in range(R):
        for t in range(T):
            seen = set()
            for k in range(K):
                e = idx[s, t, k]
                if e < 0:
                    continue
                d = int(e) // L
                if d in seen:
                    continue
                seen.add(d)
                out.append((s, t, d, int(slot[s, t, k])))
    return out


@pytest.mark.parametrize("name", ["tiny_direct", "hybrid_rowform"])
def test_bf16_rows_are_the_source_rows(orc, name):
    wl = small(name, num_tokens=40, num_max_tokens_per_rank=48, hidden=256)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    st, lay = orc.layout(wl, idx)
    st2, rec = orc.dispatch(wl, lay, x, None, idx, w)
    assert st == 0 and st2 == 0
    R, M, K = wl.num_ranks, wl.num_max_tokens_per_rank, wl.num_topk
    L = wl.num_experts // R
    xb = _bits(x)
    idx = idx.numpy()
    w = w.numpy()
    ents = dedup_entries(wl, idx, lay["slot_map"])
    filled = np.zeros(rec["recv_x"].shape[0], bool)
    for s, t, d, row in ents:
        g = d * R * M + row
        filled[g] = True
        assert np.array_equal(rec["recv_x"][g], xb[s, t])
        # sidecars: destination-local expert index / weight on lanes to d, else -1 / 0
        on = (idx[s, t] >= 0) & (idx[s, t] // L == d)
        assert rec["recv_topk_idx"][g].tolist() == np.where(on, idx[s, t] - d * L, -1).tolist()
        assert rec["recv_topk_weights"][g].tolist() == np.where(on, w[s, t], 0.0).astype(np.float32).tolist()
        assert rec["recv_src_metadata"][g].tolist() == [s, t] + [-1] * K
    assert not rec["recv_x"][~filled].any()
    assert filled.sum() == lay["num_tokens_per_rank"].sum()


def test_precast_fp8_rows_and_scales_are_verbatim(orc):
    wl = small("dsv3_fp8_precast", num_tokens=20, num_max_tokens_per_rank=20, hidden=512)
    idx, w = W.routing(wl)
    x, sf = W.hidden(wl)
    _, lay = orc.layout(wl, idx)
    st, rec = orc.dispatch(wl, lay, x, sf, idx, w)
    assert st == 0
    R, M = wl.num_ranks, wl.num_max_tokens_per_rank
    for s, t, d, row in dedup_entries(wl, idx.numpy(), lay["slot_map"]):
        g = d * R * M + row
        assert np.array_equal(rec["recv_x"][g], x[s, t].numpy())
        assert np.array_equal(rec["recv_sf"][g], sf[s, t].numpy())


def test_fused_cast_rows(orc):
    wl = small("dsv3_fp8", num_tokens=12, num_max_tokens_per_rank=16, hidden=1152)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    _, lay = orc.layout(wl, idx)
    st, rec = orc.dispatch(wl, lay, x, None, idx, w)
    assert st == 0
    R, M = wl.num_ranks, wl.num_max_tokens_per_rank
    xb = _bits(x)
    for s, t, d, row in dedup_entries(wl, idx.numpy(), lay["slot_map"]):
        g = d * R * M + row
        q, sf = orc.cast_row_fp8(xb[s, t])
        assert np.array_equal(rec["recv_x"][g], q)
        assert np.array_equal(rec["recv_sf"][g], sf)
        # dequantised row within the e4m3 rounding bound of the source row
        xf = orc.bf16_to_f32(xb[s, t]).astype(np.float64)
        deq = orc.e4m3_to_f32(q).astype(np.float64) * np.repeat(sf, 128)
        assert np.all(np.abs(deq - xf) <= (2 ** -4 + 1e-6) * np.abs(xf) + 2 ** -10 * np.repeat(sf, 128) * 1.0001)


def test_expanded_rows_and_metadata(orc):
    wl = small("expanded", num_tokens=24, num_max_tokens_per_rank=24, hidden=256, expert_alignment=4)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    st, lay = orc.layout(wl, idx)
    st2, rec = orc.dispatch(wl, lay, x, None, idx, w)
    assert st == 0 and st2 == 0
    R, M, K = wl.num_ranks, wl.num_max_tokens_per_rank, wl.num_topk
    L = wl.num_experts // R
    xb = _bits(x)
    idx = idx.numpy()
    pos, region = lay["exp_pos"], lay["exp_region"]
    n = 0
    for s in range(R):
        for t in range(wl.num_tokens):
            for k in range(K):
                e = idx[s, t, k]
                if e < 0:
                    continue
                d = e // L
                assert np.array_equal(rec["recv_x"][region[d] + pos[s, t, k]], xb[s, t])
                n += 1
    assert n == int(lay["exp_cnt"].sum())
    for s, t, d, row in dedup_entries(wl, idx, lay["slot_map"]):
        on = (idx[s, t] >= 0) & (idx[s, t] // L == d)
        assert rec["recv_src_metadata"][d * R * M + row].tolist() == [s, t] + np.where(on, pos[s, t], -1).tolist()


# ---- combine -------------------------------------------------------------

def _ulp_bf16(v):
    """bf16 spacing at |v| (binary64)."""
    v = np.abs(v)
    e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    return np.where(v > 0, 2.0 ** (e - 7), 2.0 ** -133)


@pytest.mark.parametrize("name", ["tiny_direct", "hybrid_rowform", "expanded"])
def test_identity_experts_give_weight_sum_times_x(orc, name):
    wl = small(name, num_tokens=30, num_max_tokens_per_rank=32, hidden=256)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    _, lay = orc.layout(wl, idx)
    _, rec = orc.dispatch(wl, lay, x, None, idx, w)
    st, out = orc.combine(wl, lay, rec["recv_x"], idx, w)
    assert st == 0
    xf = orc.bf16_to_f32(_bits(x)).astype(np.float64)
    wsum = np.where(idx.numpy() >= 0, w.numpy().astype(np.float64), 0).sum(-1)
    closed = wsum[..., None] * xf
    got = orc.bf16_to_f32(out).astype(np.float64)
    assert np.all(np.abs(got - closed) <= _ulp_bf16(closed))


def test_single_lane_unit_weight_returns_x(orc):
    wl = small("tiny_direct", num_topk=1, num_tokens=50, num_max_tokens_per_rank=50, hidden=384)
    idx, _ = W.routing(wl)
    w = torch.ones_like(idx, dtype=torch.float32)
    x, _ = W.hidden(wl)
    _, lay = orc.layout(wl, idx)
    _, rec = orc.dispatch(wl, lay, x, None, idx, w)
    _, out = orc.combine(wl, lay, rec["recv_x"], idx, w)
    assert np.array_equal(out, _bits(x))


def test_power_of_two_weights_are_exact(orc):
    wl = small("direct_zipf", num_tokens=25, num_max_tokens_per_rank=25, hidden=256)
    idx, _ = W.routing(wl)
    K = wl.num_topk
    w = torch.tensor([2.0 ** -(k + 1) for k in range(K)], dtype=torch.float32).expand_as(idx).contiguous()
    w = w.masked_fill(idx < 0, 0.0)
    x, _ = W.hidden(wl)
    _, lay = orc.layout(wl, idx)
    _, rec = orc.dispatch(wl, lay, x, None, idx, w)
    _, out = orc.combine(wl, lay, rec["recv_x"], idx, w)
    # bf16 x has 8 significant bits; the weighted sum spans < 24 bits: exact in fp32
    exact = (w.double().sum(-1, keepdim=True) * x.double()).float()
    assert np.array_equal(out, _bits(exact.to(torch.bfloat16)))


def test_zero_outputs_give_positive_zero(orc):
    wl = small("direct_zipf", num_tokens=10, num_max_tokens_per_rank=10, hidden=128)
    idx, w = W.routing(wl)
    _, lay = orc.layout(wl, idx)
    y = np.zeros((orc.recv_rows(wl), wl.hidden), np.uint16)
    _, out = orc.combine(wl, lay, y, idx, w)
    assert np.all(out == 0)  # +0, never -0


def test_combine_token_hand_worked(orc):
    one, three = orc.f32_to_bf16(np.array([1.0, 3.0], np.float32))
    rows = [np.full(4, one, np.uint16), None, np.full(4, three, np.uint16)]
    out = orc.combine_token(rows, np.array([0.5, 7.0, 0.25], np.float32))
    # 0.5*1 + 0.25*3 = 1.25 (the masked lane's weight is ignored) -> bf16 0x3FA0
    assert out.tolist() == [0x3FA0] * 4
    assert orc.combine_token([None, None], np.array([1.0, 1.0], np.float32)).size == 0


def test_combine_is_a_fused_chain_in_lane_order(orc):
    # y = [1, 1, 2^-24], w = [1, 2^-8, 1 + 2^-23]. In lane order with fused
    # multiply-adds: acc = 1, then 1 + 2^-8 (exact), then the exact sum
    # 1 + 2^-8 + 2^-24 + 2^-47 rounds up to 1 + 2^-8 + 2^-23 in binary32, which is
    # above the bf16 tie at 1 + 2^-8, so the result is 1 + 2^-7 (0x3F81).
    # Rounding the last product first (2^-24), or summing in reverse lane order,
    # lands exactly on the tie instead and gives 1.0 (0x3F80).
    y = orc.f32_to_bf16(np.array([1.0, 1.0, 2.0 ** -24], np.float32))
    w = np.array([1.0, 2.0 ** -8, 1 + 2.0 ** -23], np.float32)
    out = orc.combine_token([np.array([v], np.uint16) for v in y], w)
    assert out.tolist() == [0x3F81]
    rev = orc.combine_token([np.array([v], np.uint16) for v in y[::-1]], w[::-1].copy())
    assert rev.tolist() == [0x3F80]


# ---- compact receive rows (PR #690, Direct Recv X) ---------------------------

def _row_block(wl, s):
    return s if wl.n_so == 1 else (s % wl.n_su) * wl.n_so + s // wl.n_su


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("name", ["direct_zipf_compact", "hybrid_compact"])
def test_compact_rows_pack_each_destination_in_row_block_order(orc, name, mode):
    """Each destination's entries, sorted by (source row block, token), occupy
    consecutive rows: from the start of the destination's R*M-row window
    (compact, PR #690 Direct Recv X), or right after everything the
    destinations before it receive (packed: destinations back to back)."""
    wl = W.PARITY[name].replace(num_tokens=23, num_max_tokens_per_rank=29, hidden=128, compact=mode)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    st, lay = orc.layout(wl, idx)
    assert st == 0
    R, T, K, M = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.num_max_tokens_per_rank
    L = wl.num_experts // R
    idx_np = idx.numpy()
    xb = _bits(x)
    expect = {}
    base = 0
    for d in range(R):
        ents = sorted({(_row_block(wl, s), t, s) for s in range(R) for t in range(T)
                       for e in idx_np[s, t] if e >= 0 and e // L == d})
        start = d * R * M if mode == 1 else base
        for i, (_, t, s) in enumerate(ents):
            expect[(s, t, d)] = start + i
        assert len(ents) == lay["recv_cnt"][d].sum()
        assert lay["recv_region"][d] == base
        base += len(ents)
    assert lay["recv_region"][R] == base
    got = {}
    for s in range(R):
        for t in range(T):
            o = orc.dispatch_token(wl, lay, s, t, xb[s, t], None, idx_np[s, t], w.numpy()[s, t])
            for dd, r in zip(o["meta_dst"], o["meta_row"]):
                got[(s, t, int(dd))] = int(r)
            assert sorted(zip(o["hid_dst"].tolist(), o["hid_row"].tolist())) == \
                sorted(zip(o["meta_dst"].tolist(), o["meta_row"].tolist()))
    assert got == expect
    if mode == 2:
        # the packed buffer holds R*T*min(K, R) rows: every token has at most
        # min(K, R) distinct destinations
        assert orc.recv_rows(wl) == R * T * min(K, R) >= base


@pytest.mark.parametrize("name", ["direct_zipf_compact", "hybrid_compact"])
def test_compact_packed_and_row_form_give_the_same_combine(orc, name):
    wl = W.PARITY[name].replace(num_tokens=40, num_max_tokens_per_rank=48, hidden=256)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    outs = []
    R, M, K = wl.num_ranks, wl.num_max_tokens_per_rank, wl.num_topk
    for mode in (0, 1, 2):
        v = wl.replace(compact=mode)
        _, lay = orc.layout(v, idx)
        st, rec = orc.dispatch(v, lay, x, None, idx, w)
        assert st == 0
        st, out = orc.combine(v, lay, rec["recv_x"], idx, w)
        assert st == 0
        outs.append(out)
        md = rec["recv_src_metadata"]
        if mode == 1:
            # filled rows of destination d are exactly the first sum_s recv_cnt[d][s] of its window
            md = md.reshape(R, R * M, -1)
            for d in range(R):
                n = int(lay["recv_cnt"][d].sum())
                assert np.all(md[d, :n, 0] >= 0) and not md[d, n:].any()
        if mode == 2:
            # packed: the first recv_region[R] rows are filled, destination by destination
            n = int(lay["recv_region"][R])
            assert md.shape == (R * wl.num_tokens * min(K, R), K + 2)
            assert np.all(md[:n, 0] >= 0) and not md[n:].any()
            for d in range(R):
                a, b = lay["recv_region"][d], lay["recv_region"][d + 1]
                assert np.all(rec["recv_topk_idx"][a:b].max(-1) >= 0)  # a lane of d on every row
                assert b - a == lay["recv_cnt"][d].sum()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_packed_capacity_overflow_is_reported_not_silent(orc):
    """Packed rows past a caller's capacity are not written and the call
    reports OVERFLOW (PR #690 review: a payload is never dropped silently); the
    rows below the capacity are those of the full-capacity dispatch, and
    combine leaves the lanes it cannot read out of the sum, reporting it."""
    wl = W.PARITY["hybrid_packed"].replace(num_tokens=20, num_max_tokens_per_rank=20, hidden=128)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    _, lay = orc.layout(wl, idx)
    total = int(lay["recv_region"][-1])
    st, full = orc.dispatch(wl, lay, x, None, idx, w, fill=0xAB)
    assert st == 0
    cap = total - 7
    small_wl = wl.replace(recv_capacity=cap)
    assert orc.recv_rows(small_wl) == cap and orc.sidecar_rows(small_wl) == cap
    st, part = orc.dispatch(small_wl, lay, x, None, idx, w, fill=0xAB)
    assert st == orc.OVERFLOW
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_metadata"):
        assert np.array_equal(part[k], full[k][:cap]), k
    st, hid, side = orc.lane_rows(small_wl, lay, idx)
    assert st == orc.OVERFLOW
    st0, hid0, _ = orc.lane_rows(wl, lay, idx)
    assert st0 == 0 and np.array_equal(hid, np.where(hid0 < cap, hid0, -1))
    y = np.arange(total * wl.hidden, dtype=np.uint32).reshape(total, wl.hidden).astype(np.uint16) & 0x3FFF
    st, out_full = orc.combine(wl.replace(recv_capacity=total), lay, y, idx, w)
    assert st == 0
    st, out_part = orc.combine(small_wl, lay, y[:cap], idx, w)
    assert st == orc.OVERFLOW
    lost = (hid0 >= cap).any(-1)  # tokens with a lane past the capacity
    assert lost.any() and np.array_equal(out_part[~lost], out_full[~lost])
    assert orc.combine(wl.replace(recv_capacity=3), lay, y, idx, w)[0] == orc.OVERFLOW


def test_zero_padding_of_aligned_expanded_blocks(orc):
    """Expanded blocks padded to the alignment: rows between an expert's lanes
    and the next block start are zero with zero padding, untouched without."""
    wl = W.PARITY["expanded_a128_zero"].replace(num_tokens=20, num_max_tokens_per_rank=20, hidden=128,
                                                expert_alignment=8)
    idx, w = W.routing(wl)
    x, _ = W.hidden(wl)
    _, lay = orc.layout(wl, idx)
    R, L = wl.num_ranks, wl.num_experts // wl.num_ranks
    pad = []
    for d in range(R):
        for j in range(L):
            a = lay["exp_region"][d] + lay["exp_base"][d, j] + lay["exp_cnt"][d, j]
            b = lay["exp_region"][d] + lay["exp_base"][d, j + 1]
            assert b - a < wl.expert_alignment and (b - lay["exp_region"][d]) % wl.expert_alignment == 0
            pad.extend(range(a, b))
    assert pad
    st, rec = orc.dispatch(wl, lay, x, None, idx, w, fill=0xFF)
    assert st == 0 and not rec["recv_x"][pad].any()
    st, rec = orc.dispatch(wl.replace(zero_padding=False), lay, x, None, idx, w, fill=0xFF)
    assert np.all(rec["recv_x"][pad] == 0xFFFF)
