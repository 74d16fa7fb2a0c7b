"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element
by element, on seeded inputs of every workload at reduced sizes (several
256-token blocks, a ragged tail, full hidden widths).

Bar: layouts, slots, receive rows, sidecars and FP8 casts bit-exact; combine
bit-exact as well (the oracle and the kernel take the same fused multiply-adds
in the same lane order), which is inside the one-bf16-ulp tolerance.
"""
import numpy as np
import pytest
import torch

import combine_ep_get_02_gb300 as ep
import oracle
import workloads as W
from _harness import (GpuRun, assert_layout_equal, compare_dispatch, inputs,
                      oracle_combine_from_device_y, random_y, u16)

pytestmark = pytest.mark.gpu

EXTRA = {
    # direct with M > T, K=1 and E = R (one expert per rank)
    "direct_k1_l1": W.Workload("direct_k1_l1", 1, 16, 16, 1, 200, 256, 512),
    # K above 8 (wide lane path) with masking
    "direct_k12": W.Workload("direct_k12", 1, 8, 64, 12, 257, 260, 256, mask_frac=0.1),
    "direct_k32": W.Workload("direct_k32", 1, 4, 64, 32, 70, 70, 128, mask_frac=0.05),
    # FP8 cast on a width that is not a multiple of 512 columns, heavy masking
    "cast_h1152": W.Workload("cast_h1152", 1, 8, 64, 6, 513, 520, 1152, recv_dtype="fp8",
                             mask_frac=0.3, routing="zipf"),
    # hybrid + expanded + alignment, FP8 cast in the expanded layout
    "hybrid_expand_a128": W.Workload("hybrid_expand_a128", 2, 4, 64, 4, 300, 300, 256,
                                     expand=True, expert_alignment=128, routing="zipf",
                                     y_kind="random"),
    "expand_fp8": W.Workload("expand_fp8", 1, 8, 32, 4, 260, 260, 512, recv_dtype="fp8",
                             expand=True, expert_alignment=4, routing="hot", y_kind="random"),
    # odd sizes: R not a multiple of 4, tiny hidden
    "odd_r6": W.Workload("odd_r6", 3, 2, 18, 3, 33, 40, 8, mask_frac=0.2),
    # one token per rank
    "one_token": W.Workload("one_token", 1, 16, 256, 8, 1, 4, 7168, y_kind="random"),
    # bf16 rows wider than one shared-memory stage of the bulk-copy dispatch (two pieces, the
    # second shorter), row form and expanded with zeroed padding
    "wide_rows": W.Workload("wide_rows", 1, 8, 64, 6, 150, 160, 12296, mask_frac=0.1),
    "wide_expand": W.Workload("wide_expand", 1, 4, 16, 4, 70, 70, 8200, expand=True,
                              expert_alignment=4, zero_padding=True, y_kind="random"),
    # the library's limits: 64 ranks, 4096 experts, top-32; hidden 16384 with FP8 (128 scale
    # groups, 32 packed scale words)
    "max_ranks_experts": W.Workload("max_ranks_experts", 1, 64, 4096, 32, 40, 48, 128, mask_frac=0.1,
                                    routing="zipf"),
    "max_expand": W.Workload("max_expand", 4, 16, 4096, 32, 30, 30, 256, expand=True, expert_alignment=8,
                             zero_padding=True, y_kind="random"),
    "max_hidden_fp8": W.Workload("max_hidden_fp8", 1, 4, 16, 4, 40, 40, 16384, recv_dtype="fp8",
                                 routing="zipf"),
    "max_hidden_packed": W.Workload("max_hidden_packed", 2, 2, 16, 4, 40, 40, 16384, recv_dtype="fp8",
                                    sf_pack=True),
    "max_hidden_precast_packed": W.Workload("max_hidden_precast_packed", 1, 4, 16, 4, 40, 40, 16384,
                                            x_dtype="fp8", recv_dtype="fp8", sf_pack=True),
    # the general layout kernel with top-k <= 8: expanded with more experts than the register
    # kernel's per-(round, warp) expert tables hold in shared memory, and more than four rounds
    # of 256 tokens per CTA (row form and expanded)
    "expand_many_experts": W.Workload("expand_many_experts", 1, 4, 4096, 8, 40, 40, 128, expand=True,
                                      expert_alignment=2, routing="zipf", y_kind="random"),
    "long_tokens": W.Workload("long_tokens", 1, 2, 16, 8, 8500, 8500, 64, mask_frac=0.05),
    "long_tokens_expand": W.Workload("long_tokens_expand", 1, 2, 16, 4, 8500, 8500, 64, expand=True,
                                     expert_alignment=4, zero_padding=True, y_kind="random"),
    # the register layout kernel with two and four rounds of 256 tokens per CTA (8 CTAs a source)
    "rounds4_rows": W.Workload("rounds4_rows", 1, 2, 16, 8, 7000, 7000, 64, mask_frac=0.05),
    "rounds2_expand": W.Workload("rounds2_expand", 1, 2, 16, 4, 3000, 3000, 64, expand=True, y_kind="random"),
    "rounds4_expand": W.Workload("rounds4_expand", 1, 2, 32, 8, 7000, 7000, 64, expand=True,
                                 expert_alignment=2, zero_padding=True, routing="zipf", y_kind="random"),
}

CASES = dict(W.PARITY)
CASES.update(EXTRA)


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    wl = CASES[request.param]
    idx, w, x, sf = inputs(wl)
    st, olay = oracle.layout(wl, idx)
    assert st == 0
    return wl, idx, w, x, sf, olay


def test_layout(case):
    wl, idx, w, x, sf, olay = case
    run = GpuRun(wl, idx, w, x, sf).layout()
    assert run.status() == ep.EP_OK
    assert_layout_equal(run.layout_np(), olay, wl.expand)


@pytest.mark.parametrize("copy_path", [1, 2])
def test_dispatch(case, copy_path):
    """Both ways of moving unchanged rows (register copies, bulk copies through
    shared memory); the fused cast ignores the setting."""
    wl, idx, w, x, sf, olay = case
    run = GpuRun(wl, idx, w, x, sf, copy_path=copy_path).layout().dispatch()
    assert run.status() == ep.EP_OK
    st, orec = oracle.dispatch(wl, olay, x, sf, idx, w)
    assert st == 0
    compare_dispatch(run, olay, orec)


def test_combine(case):
    wl, idx, w, x, sf, olay = case
    run = GpuRun(wl, idx, w, x, sf).layout()
    if wl.y_kind == "identity" and wl.recv_dtype == "bf16":
        run.dispatch()
        y = run.recv.recv_x
    else:
        y = random_y(wl, ep.ep_recv_rows(run.cfg), run.dev)
    run.combine(y)
    assert run.status() == ep.EP_OK
    got = u16(run.out).reshape(-1, wl.hidden)
    exp = oracle_combine_from_device_y(wl, olay, idx, w, y)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        raise AssertionError(f"{len(bad)} combine mismatches; first {bad[0].tolist()}: "
                             f"{got[tuple(bad[0])]:#06x} vs {exp[tuple(bad[0])]:#06x}")


def test_identity_combine_of_dispatch_is_weight_sum_times_x():
    """combine(dispatch(x)) with identity experts = (sum of weights) * x, within
    one bf16 ulp (closed form, independent of the oracle)."""
    wl = W.PARITY["direct_zipf"]
    idx, w, x, sf = inputs(wl)
    run = GpuRun(wl, idx, w, x, sf).layout().dispatch()
    run.combine(run.recv.recv_x)
    got = run.out.float().cpu().double()
    wsum = torch.where(idx >= 0, w.double(), torch.zeros((), dtype=torch.float64)).sum(-1, keepdim=True)
    closed = wsum * x.double()
    ulp = torch.where(closed != 0, 2.0 ** (torch.floor(torch.log2(closed.abs().clamp_min(1e-30))) - 7),
                      torch.full_like(closed, 2.0 ** -133))
    assert torch.all((got - closed).abs() <= ulp)


@pytest.mark.parametrize("name", ["direct_zipf", "hybrid_rowform", "expanded"])
def test_grid_sizes_do_not_change_results(name):
    """Slots are a pure function of topk_idx: outputs are identical for every
    prologue grid and every dispatch/combine grid (PR #753 Approach, New API)."""
    wl = W.PARITY[name]
    idx, w, x, sf = inputs(wl)
    ref = None
    for pro, sms in ((0, 0), (1, 1), (7, 13), (64, 3), (3, 152)):
        run = GpuRun(wl, idx, w, x, sf, num_prologue_sms=pro, num_sms=sms).layout().dispatch()
        y = run.recv.recv_x if not wl.expand else random_y(wl, ep.ep_recv_rows(run.cfg), run.dev)
        run.combine(y)
        assert run.status() == ep.EP_OK
        lay = run.layout_np()
        rx = u16(run.recv.recv_x)
        md = run.recv.recv_src_metadata.cpu().numpy()
        out = u16(run.out)
        if ref is None:
            ref = (lay, rx, md, out)
            continue
        assert_layout_equal(lay, ref[0], wl.expand)
        assert np.array_equal(rx, ref[1])
        assert np.array_equal(md, ref[2])
        assert np.array_equal(out, ref[3])


def test_repeated_runs_bitwise_equal():
    wl = W.PARITY["dsv3_fp8"]
    idx, w, x, sf = inputs(wl)
    run = GpuRun(wl, idx, w, x, sf).layout().dispatch()
    y = random_y(wl, ep.ep_recv_rows(run.cfg), run.dev)
    run.combine(y)
    first = (u16(run.recv.recv_x), run.recv.recv_sf.cpu().numpy(), u16(run.out))
    for _ in range(3):
        run.layout().dispatch().combine(y)
        assert np.array_equal(u16(run.recv.recv_x), first[0])
        assert np.array_equal(run.recv.recv_sf.cpu().numpy(), first[1])
        assert np.array_equal(u16(run.out), first[2])


def test_slots_do_not_depend_on_x_or_weights():
    wl = W.PARITY["direct_zipf"]
    idx, w, x, sf = inputs(wl)
    a = GpuRun(wl, idx, w, x, sf).layout().layout_np()
    x2 = torch.randn(x.shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    b = GpuRun(wl, idx, torch.rand_like(w), x2, sf).layout().layout_np()
    assert_layout_equal(a, b, False)


def test_empty_ranks():
    wl = W.Workload("empty", 1, 8, 32, 4, 0, 16, 256)
    idx = torch.zeros(8, 0, 4, dtype=torch.int64)
    w = torch.zeros(8, 0, 4)
    x = torch.zeros(8, 0, 256, dtype=torch.bfloat16)
    run = GpuRun(wl, idx, w, x, None).layout().dispatch()
    run.combine(run.recv.recv_x)
    assert run.status() == ep.EP_OK
    lay = run.layout_np()
    assert not lay["num_tokens_per_rank"].any() and not lay["recv_psum"].any()
    assert not lay["num_tokens_per_expert"].any()


def test_all_lanes_masked():
    wl = W.Workload("masked", 1, 4, 16, 3, 40, 40, 128)
    idx = torch.full((4, 40, 3), -1, dtype=torch.int64)
    w = torch.zeros(4, 40, 3)
    x = torch.randn(4, 40, 128).to(torch.bfloat16)
    run = GpuRun(wl, idx, w, x, None).layout().dispatch()
    run.combine(run.recv.recv_x)
    assert run.status() == ep.EP_OK
    assert (run.lay.slot_map == -1).all()
    assert not u16(run.out).any()  # +0 everywhere
    assert not u16(run.recv.recv_x).any()  # nothing written (buffer was zeroed)


def test_bad_topk_is_reported_not_written():
    wl = W.Workload("bad", 1, 4, 16, 2, 30, 30, 128)
    idx, w, x, sf = inputs(wl)
    idx = idx.clone()
    idx[1, 3, 0] = 16      # >= E
    idx[2, 7, 1] = -5      # < -1
    run = GpuRun(wl, idx, w, x, sf).layout().dispatch()
    run.combine(run.recv.recv_x)
    assert run.status() == ep.EP_ERR_BAD_TOPK
    assert run.status() == ep.EP_OK  # the status is cleared once read
    # the bad lanes are masked, everything else matches the oracle
    st, olay = oracle.layout(wl, idx)
    assert st == oracle.BAD_TOPK
    assert_layout_equal(run.layout_np(), olay, False)


def test_expanded_repeated_expert_is_reported():
    wl = W.Workload("dup", 1, 4, 16, 3, 20, 20, 128, expand=True)
    idx, w, x, sf = inputs(wl)
    idx = idx.clone()
    idx[0, 2, 2] = idx[0, 2, 0]
    run = GpuRun(wl, idx, w, x, sf).layout().dispatch()
    assert run.status() == ep.EP_ERR_BAD_TOPK
    st, olay = oracle.layout(wl, idx)
    assert_layout_equal(run.layout_np(), olay, True)


def _non_nan_slices(first, n):
    """Slices of [first, first+n) that hold no NaN bit pattern."""
    out, lo = [], first
    for nan_lo, nan_hi in ((0x7F800001, 0x80000000), (0xFF800001, 0x100000000)):
        if nan_hi <= first or nan_lo >= first + n:
            continue
        if nan_lo > lo:
            out.append(slice(lo - first, nan_lo - first))
        lo = max(lo, nan_hi)
    if lo < first + n:
        out.append(slice(lo - first, n))
    return out


@pytest.mark.parametrize("kind", ["e4m3", "bf16"])
def test_device_conversions_match_oracle_on_every_float(kind):
    """The kernels' fp32->e4m3 (RNE, satfinite) and fp32->bf16 (RNE) conversions
    against the oracle's converters (written from the format definitions) on all
    2^32 binary32 bit patterns (NaN inputs excluded: outside the contract)."""
    import concurrent.futures
    chunk = 1 << 28
    firsts = list(range(0, 1 << 32, chunk))
    conv = oracle.e4m3_of_bits if kind == "e4m3" else oracle.bf16_of_bits
    diag = ep.ep_diag_e4m3_of_bits if kind == "e4m3" else ep.ep_diag_bf16_of_bits
    dt = torch.uint8 if kind == "e4m3" else torch.int16
    buf = torch.empty(chunk, dtype=dt, device="cuda")
    with concurrent.futures.ThreadPoolExecutor(4) as ex:  # the oracle call releases the GIL
        futs = {f: ex.submit(conv, f, chunk) for f in firsts}
        for first in firsts:
            diag(first, buf)
            got = buf.cpu().numpy()
            exp = futs.pop(first).result()
            got = got.view(exp.dtype)
            for sl in _non_nan_slices(first, chunk):
                assert np.array_equal(got[sl], exp[sl]), (hex(first), sl)


@pytest.mark.parametrize("name,x_dtype,recv", [("expanded_a128_zero", "bf16", "bf16"),
                                               ("expanded_a128_zero", "bf16", "fp8"),
                                               ("expanded_a128_zero", "fp8", "fp8")])
def test_zero_padding_rows(name, x_dtype, recv):
    """Expanded blocks aligned to 128 rows: with zero padding every row of every
    region is either a lane's row or zero (PR #753 Compatibility: kDoZeroPadding,
    kExpertAlignment); checked over the whole used buffer, prefilled with 0xFF."""
    wl = W.PARITY[name].replace(x_dtype=x_dtype, recv_dtype=recv, hidden=512)
    idx, w, x, sf = inputs(wl)
    st, olay = oracle.layout(wl, idx)
    run = GpuRun(wl, idx, w, x, sf).layout()
    run.recv = ep.alloc_recv(run.cfg, run.dev)
    run.recv.recv_x.view(torch.uint8).fill_(0xFF)
    if run.recv.recv_sf is not None:
        run.recv.recv_sf.view(torch.uint8).fill_(0xFF)
    run.dispatch()
    assert run.status() == ep.EP_OK
    st, orec = oracle.dispatch(wl, olay, x, sf, idx, w, fill=0xFF)
    used = int(olay["exp_region"][-1])
    assert used % 128 == 0 and used > int(olay["exp_cnt"].sum())
    got = run.recv.recv_x[:used].contiguous().view(torch.uint8).cpu().numpy()
    assert np.array_equal(got, orec["recv_x"][:used].view(np.uint8))
    if recv == "fp8":
        assert np.array_equal(run.recv.recv_sf[:used].cpu().numpy().view(np.uint32),
                              orec["recv_sf"][:used].view(np.uint32))


def test_cached_redispatch_replays_the_stored_layout():
    """Cached mode: a second dispatch with new activations reuses the stored
    layout (no prologue) and lands every row where the oracle puts it."""
    wl = W.PARITY["dsv3_fp8"]
    idx, w, x, sf = inputs(wl)
    st, olay = oracle.layout(wl, idx)
    run = GpuRun(wl, idx, w, x, sf).layout().dispatch()
    x2 = torch.randn(x.shape, generator=torch.Generator().manual_seed(77)).to(torch.bfloat16)
    run.x = x2.to(run.dev)
    run.dispatch()  # layout not recomputed
    assert run.status() == ep.EP_OK
    st, orec = oracle.dispatch(wl, olay, x2, sf, idx, w)
    compare_dispatch(run, olay, orec)


@pytest.mark.parametrize("name", ["direct_zipf", "hybrid_rowform", "dsv3_fp8", "dsv3_fp8_precast"])
def test_atomic_slots_plus_sort_equal_the_deterministic_dispatch(name):
    """PR #753 Motivation/Approach: racing atomicAdd slots followed by the
    post-hoc sort by source token give exactly the kernel-side deterministic
    placement (every receive tensor, bit for bit)."""
    wl = W.PARITY[name]
    idx, w, x, sf = inputs(wl)
    det = GpuRun(wl, idx, w, x, sf).layout().dispatch()
    racy = ep.alloc_recv(det.cfg, det.dev, zero=True)
    counters = torch.full((wl.num_ranks, wl.num_ranks), 7, dtype=torch.int32, device=det.dev)
    ep.ep_dispatch_atomic(det.cfg, det.x, det.sf, det.idx, det.w, racy, counters, det.ws)
    assert torch.equal(counters, det.lay.num_tokens_per_rank)
    srt = ep.alloc_recv(det.cfg, det.dev, zero=True)
    ep.ep_deterministic_sort(det.cfg, racy, counters, srt)
    torch.cuda.synchronize()
    for f in ("recv_x", "recv_sf", "recv_topk_idx", "recv_topk_weights", "recv_src_metadata"):
        a, b = getattr(det.recv, f), getattr(srt, f)
        if a is None:
            continue
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f


@pytest.mark.parametrize("name", ["dsv3_fp8", "expanded", "hybrid_compact", "hybrid_packed"])
def test_cuda_graph_replay_equals_eager(name):
    """layout -> dispatch -> combine captured once in a CUDA graph and replayed
    gives the eager results bit for bit (the workspace counter returns to zero
    inside every replay)."""
    wl = W.PARITY[name]
    idx, w, x, sf = inputs(wl)
    eager = GpuRun(wl, idx, w, x, sf).layout().dispatch()
    y = eager.recv.recv_x if (wl.recv_dtype == "bf16" and not wl.expand) else \
        random_y(wl, ep.ep_recv_rows(eager.cfg), eager.dev)
    eager.combine(y)
    assert eager.status() == ep.EP_OK
    run = GpuRun(wl, idx, w, x, sf)
    run.recv = ep.alloc_recv(run.cfg, run.dev, zero=True)
    run.out = torch.empty_like(eager.out)
    y2 = run.recv.recv_x if (wl.recv_dtype == "bf16" and not wl.expand) else y
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        ep.ep_get_dispatch_layout(run.cfg, run.idx, run.lay, run.ws, s)  # first call outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            ep.ep_get_dispatch_layout(run.cfg, run.idx, run.lay, run.ws, s)
            ep.ep_dispatch(run.cfg, run.lay, run.x, run.sf, run.idx, run.w, run.recv, run.ws, s)
            ep.ep_combine(run.cfg, run.lay, y2, run.idx, run.w, run.out, run.ws, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert run.status() == ep.EP_OK
    assert_layout_equal(run.layout_np(), eager.layout_np(), wl.expand)
    assert torch.equal(run.recv.recv_x.view(torch.uint8), eager.recv.recv_x.view(torch.uint8))
    assert torch.equal(run.out.view(torch.int16), eager.out.view(torch.int16))


@pytest.mark.parametrize("name", ["hybrid_packed", "dsv3_fp8_packed_rows"])
def test_packed_capacity_overflow_is_reported(name):
    """Packed receive rows in a buffer smaller than what arrives: the entries
    past the capacity are not written and dispatch reports EP_ERR_OVERFLOW
    (PR #690 review: a payload is never dropped silently); every row below the
    capacity is the oracle's, and combine, which cannot read the lost lanes,
    reports the same and sums the rest exactly as the oracle does."""
    base = W.PARITY[name]
    idx, w, x, sf = inputs(base)
    st, olay = oracle.layout(base, idx)
    total = int(olay["recv_region"][-1])
    wl = base.replace(recv_capacity=total - 37)
    cap = total - 37
    run = GpuRun(wl, idx, w, x, sf).layout()
    assert run.status() == ep.EP_OK
    assert int(run.lay.recv_region[-1]) == total
    run.recv = ep.alloc_recv(run.cfg, run.dev)
    assert run.recv.recv_x.shape[0] == cap
    for t in (run.recv.recv_x, run.recv.recv_sf, run.recv.recv_topk_idx, run.recv.recv_topk_weights,
              run.recv.recv_src_metadata):
        if t is not None:
            t.view(torch.uint8).fill_(0xFF)
    run.dispatch()
    assert run.status() == ep.EP_ERR_OVERFLOW
    assert run.status() == ep.EP_OK
    st, orec = oracle.dispatch(wl, olay, x, sf, idx, w, fill=0xFF)
    assert st == oracle.OVERFLOW
    row_bytes = wl.hidden * (1 if wl.recv_dtype == "fp8" else 2)
    got = run.recv.recv_x.contiguous().view(torch.uint8).cpu().numpy().reshape(cap, row_bytes)
    assert np.array_equal(got, np.ascontiguousarray(orec["recv_x"]).view(np.uint8).reshape(cap, row_bytes))
    for k in ("recv_topk_idx", "recv_topk_weights", "recv_src_metadata"):
        g = getattr(run.recv, k).cpu().numpy()
        assert np.array_equal(g.view(np.uint8), orec[k].view(np.uint8)), k
    y = random_y(wl, cap, run.dev)
    run.combine(y)
    assert run.status() == ep.EP_ERR_OVERFLOW
    st, o_out = oracle.combine(wl, olay, u16(y), idx, w)
    assert st == oracle.OVERFLOW
    assert np.array_equal(u16(run.out), o_out)


def test_work_queues_return_to_zero():
    """Dispatch and combine warps take their tokens from counters in the
    workspace header; after every launch, whatever the grid, the last warp to
    leave has put them back to zero (and the results never depend on the grid)."""
    wl = W.PARITY["direct_zipf"]
    idx, w, x, sf = inputs(wl)
    ref = None
    for sms, path in ((0, 1), (1, 2), (5, 1), (152, 2), (0, 2)):
        run = GpuRun(wl, idx, w, x, sf, num_sms=sms, copy_path=path).layout().dispatch()
        run.combine(run.recv.recv_x)
        assert run.status() == ep.EP_OK
        header = run.ws[:256].cpu().numpy()
        assert not header[4:40].any(), header[:40]
        got = (u16(run.recv.recv_x), u16(run.out))
        if ref is None:
            ref = got
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
