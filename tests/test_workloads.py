"""The seeded input recipe (workloads.py) holds the properties the benchmark and
the parity tests rely on: routing shape and weights, masking rate, Zipf skew,
the hot-expert share, the expected deduplicated fan-out of uniform routing, and
the ranges of the pre-cast FP8 inputs. Draws are reproducible."""
import math

import numpy as np
import pytest
import torch

import workloads as W


def small(name, **kw):
    return W.WORKLOADS[name].replace(**kw)


def test_draws_are_reproducible():
    wl = small("direct_zipf", num_tokens=64, num_max_tokens_per_rank=64, hidden=256)
    a, b = W.routing(wl), W.routing(wl)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(W.hidden(wl)[0].view(torch.int16), W.hidden(wl)[0].view(torch.int16))
    other = W.routing(wl.replace(seed=1))[0]
    assert not torch.equal(a[0], other)


@pytest.mark.parametrize("name", ["tiny_direct", "direct_zipf", "dsv3_fp8", "hybrid_rowform", "expanded"])
def test_routing_shape_distinct_experts_and_softmax_weights(name):
    wl = small(name, num_tokens=min(W.WORKLOADS[name].num_tokens, 128),
               num_max_tokens_per_rank=min(W.WORKLOADS[name].num_tokens, 128))
    idx, w = W.routing(wl)
    R, T, K, E = wl.num_ranks, wl.num_tokens, wl.num_topk, wl.num_experts
    assert idx.shape == (R, T, K) and w.shape == (R, T, K)
    assert idx.dtype == torch.int64 and w.dtype == torch.float32
    ix, wv = idx.numpy(), w.numpy().astype(np.float64)
    valid = ix >= 0
    assert np.all((ix >= -1) & (ix < E))
    assert np.all(wv[~valid] == 0.0) and np.all(wv[valid] > 0.0)
    for row in ix.reshape(-1, K):  # the selected experts of a token are distinct
        v = row[row >= 0]
        assert len(set(v.tolist())) == v.size
    if wl.mask_frac == 0:
        assert valid.all()
        assert np.allclose(wv.sum(-1), 1.0, atol=1e-6)  # softmax over the K selected logits


def test_masking_rate():
    wl = small("direct_zipf", num_tokens=1024, num_max_tokens_per_rank=1024, hidden=256)
    idx, _ = W.routing(wl)
    frac = float((idx < 0).float().mean())
    assert abs(frac - wl.mask_frac) < 0.003  # 131k lanes: a few standard deviations


def test_uniform_routing_fan_out_matches_the_closed_form():
    # expected distinct destination ranks of K distinct experts out of E, L per rank:
    # R * (1 - C(E - L, K) / C(E, K))
    wl = small("dsv3_fp8", num_tokens=1024, num_max_tokens_per_rank=1024, hidden=128)
    R, E, K = wl.num_ranks, wl.num_experts, wl.num_topk
    L = E // R
    expect = R * (1 - math.comb(E - L, K) / math.comb(E, K))
    d = (W.routing(wl)[0].numpy() // L).reshape(-1, K)
    got = np.mean([len(set(r.tolist())) for r in d])
    assert abs(got - expect) / expect < 0.01


def test_zipf_bias_skews_expert_popularity():
    wl = small("direct_zipf", num_tokens=1024, num_max_tokens_per_rank=1024, hidden=128, mask_frac=0.0)
    idx = W.routing(wl)[0].numpy().ravel()
    counts = np.bincount(idx, minlength=wl.num_experts)
    share_top = np.sort(counts)[::-1][: wl.num_experts // 10].sum() / counts.sum()
    assert share_top > 0.3  # the top tenth of the experts take far more than a tenth of the lanes
    gauss = small("dsv3_fp8", num_tokens=1024, num_max_tokens_per_rank=1024, hidden=128)
    c2 = np.bincount(W.routing(gauss)[0].numpy().ravel(), minlength=gauss.num_experts)
    assert np.sort(c2)[::-1][: gauss.num_experts // 10].sum() / c2.sum() < 0.15


def test_hot_experts_take_the_requested_share():
    wl = W.WORKLOADS["expanded"]
    idx = W.routing(wl)[0].numpy().ravel()
    counts = np.bincount(idx, minlength=wl.num_experts)
    n_hot = math.ceil(wl.hot_expert_frac * wl.num_experts)
    share = np.sort(counts)[::-1][:n_hot].sum() / counts.sum()
    assert n_hot == 26
    assert abs(share - wl.hot_traffic) <= 0.005


def test_precast_inputs_are_finite_codes_and_scales_in_range():
    wl = small("dsv3_fp8", num_tokens=16, num_max_tokens_per_rank=16, hidden=1024, x_dtype="fp8")
    x, sf = W.hidden(wl)
    codes = x.numpy()
    assert not np.any((codes & 0x7F) == 0x7F)  # no NaN code
    s = sf.numpy()
    assert s.shape == (wl.num_ranks, wl.num_tokens, wl.hidden // 128)
    assert np.all((s >= 1e-3) & (s < 1.1e-2))
    packed = small("dsv3_fp8", num_tokens=16, num_max_tokens_per_rank=16, hidden=1152, x_dtype="fp8",
                   sf_pack=True)
    _, words = W.hidden(packed)
    b = words.numpy().view(np.uint8).reshape(packed.num_ranks, packed.num_tokens, -1)
    G = packed.hidden // 128
    assert np.all((b[..., :G] >= 100) & (b[..., :G] <= 140)) and not b[..., G:].any()
