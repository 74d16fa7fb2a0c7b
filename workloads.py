"""Seeded synthetic inputs for the MoE dispatch / combine workloads.

This module draws the inputs that both the CUDA path and the CPU oracle
consume: routing (``topk_idx``, ``topk_weights``), hidden states ``x`` (bf16,
or pre-cast FP8-e4m3 codes with fp32 per-128-column scales) and expert outputs
``y``. It holds none of the method's arithmetic (no layout, no slots, no cast,
no reduction); everything is drawn with ``torch.Generator`` from a fixed seed.

Recipe (shared by every workload):
  * draw order: router logits, per-expert bias permutation (if any), lane mask,
    hidden states;
  * routing = top-K of N(0,1) logits plus a per-expert bias; the K selected
    lanes come out in descending score order;
  * weights = fp32 softmax over the K selected scores; masked lanes get
    ``topk_idx = -1`` and weight 0.0;
  * ``x`` = bf16(N(0,1));
  * expert outputs ``y`` come from a second generator (seed, stream 1) so they
    do not disturb the routing/hidden draws, and may be drawn on the device.

The five workloads mirror the DeepEP dispatch/combine shapes:
tiny direct (8 ranks x 4 experts), direct with Zipf-skewed routing and 2%
masked lanes, DeepSeek-V3-shaped FP8 dispatch, hybrid row form (4 scale-out x
8 scale-up), and the expanded per-expert layout with heavy skew.
"""
from __future__ import annotations

import dataclasses
import math

import torch

__all__ = ["Workload", "WORKLOADS", "PARITY", "routing", "hidden", "expert_outputs"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_so: int                     # scale-out ranks (1 = direct)
    n_su: int                     # scale-up ranks
    num_experts: int
    num_topk: int
    num_tokens: int               # tokens per logical rank
    num_max_tokens_per_rank: int
    hidden: int
    x_dtype: str = "bf16"         # "bf16" | "fp8" (pre-cast codes + fp32 scales)
    recv_dtype: str = "bf16"      # "bf16" | "fp8" (fused cast when x is bf16)
    expand: bool = False
    expert_alignment: int = 1
    compact: int = 0              # receive rows (row form only): 0 at their slots; 1 compact,
                                  # packed from the start of each destination's window; 2 packed,
                                  # destinations back to back
    recv_capacity: int = 0        # packed receive rows: rows of the receive tensors (0 = the bound)
    zero_padding: bool = False    # zero the alignment padding rows (expanded only)
    sf_pack: bool = False         # packed power-of-two scales, 4 per 32-bit word
    routing: str = "gauss"        # "gauss" | "zipf" | "hot"
    zipf_s: float = 1.1
    mask_frac: float = 0.0
    hot_expert_frac: float = 0.05
    hot_traffic: float = 0.30
    y_kind: str = "identity"      # "identity" (y = recv_x) | "random"
    seed: int = 0

    @property
    def num_ranks(self) -> int:
        return self.n_so * self.n_su

    @property
    def num_local_experts(self) -> int:
        return self.num_experts // self.num_ranks

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # 8 logical ranks x 4 experts, 128 tokens/rank, hidden 1024, top-4, identity experts.
    "tiny_direct": Workload("tiny_direct", 1, 8, 32, 4, 128, 128, 1024),
    # 16 ranks, 256 experts, top-8, 1024 tokens/rank, hidden 7168, Zipf(1.1) bias, 2% masked.
    "direct_zipf": Workload("direct_zipf", 1, 16, 256, 8, 1024, 1024, 7168,
                            routing="zipf", mask_frac=0.02, y_kind="random"),
    # DeepSeek-V3 shape: 16 ranks, 256 experts, top-8, 4096 tokens/rank, hidden 7168,
    # bf16 x cast to FP8-e4m3 with 56 fp32 scales per token inside dispatch.
    "dsv3_fp8": Workload("dsv3_fp8", 1, 16, 256, 8, 4096, 4096, 7168,
                         recv_dtype="fp8", y_kind="random"),
    # Hybrid: 4 scale-out x 8 scale-up = 32 ranks, 256 experts, top-8, 2048 tokens/rank.
    "hybrid_rowform": Workload("hybrid_rowform", 4, 8, 256, 8, 2048, 2048, 4096,
                               routing="zipf"),
    # Expanded per-expert layout: 64 ranks, 512 experts, 512 tokens/rank, 30% of
    # lanes to 5% of the experts.
    "expanded": Workload("expanded", 1, 64, 512, 8, 512, 512, 2048, expand=True,
                         routing="hot", y_kind="random"),
}

# Reduced sizes for element-by-element parity: several 256-token blocks with a
# ragged tail, full hidden widths where the row loop matters.
PARITY = {
    "tiny_direct": WORKLOADS["tiny_direct"],
    "direct_zipf": WORKLOADS["direct_zipf"].replace(num_tokens=300, num_max_tokens_per_rank=300),
    "dsv3_fp8": WORKLOADS["dsv3_fp8"].replace(num_tokens=288, num_max_tokens_per_rank=288),
    "dsv3_fp8_precast": WORKLOADS["dsv3_fp8"].replace(
        name="dsv3_fp8_precast", x_dtype="fp8", num_tokens=288, num_max_tokens_per_rank=288),
    "hybrid_rowform": WORKLOADS["hybrid_rowform"].replace(num_tokens=300, num_max_tokens_per_rank=300),
    "expanded": WORKLOADS["expanded"].replace(num_tokens=100, num_max_tokens_per_rank=100),
    # compact receive rows (each destination's rows packed from row 0)
    "direct_zipf_compact": WORKLOADS["direct_zipf"].replace(
        name="direct_zipf_compact", compact=1, num_tokens=300, num_max_tokens_per_rank=320),
    "hybrid_compact": WORKLOADS["hybrid_rowform"].replace(
        name="hybrid_compact", compact=1, num_tokens=300, num_max_tokens_per_rank=300),
    # packed receive rows (destinations back to back in a buffer of R*T*min(K,R) rows)
    "direct_zipf_packed": WORKLOADS["direct_zipf"].replace(
        name="direct_zipf_packed", compact=2, num_tokens=300, num_max_tokens_per_rank=320),
    "hybrid_packed": WORKLOADS["hybrid_rowform"].replace(
        name="hybrid_packed", compact=2, num_tokens=300, num_max_tokens_per_rank=300),
    "dsv3_fp8_packed_rows": WORKLOADS["dsv3_fp8"].replace(
        name="dsv3_fp8_packed_rows", compact=2, num_tokens=288, num_max_tokens_per_rank=288),
    # packed power-of-two scales (fused cast, and pre-cast input carrying them)
    "dsv3_fp8_packed": WORKLOADS["dsv3_fp8"].replace(
        name="dsv3_fp8_packed", sf_pack=True, num_tokens=288, num_max_tokens_per_rank=288),
    "precast_packed_h1152": WORKLOADS["dsv3_fp8"].replace(
        name="precast_packed_h1152", x_dtype="fp8", sf_pack=True, hidden=1152, num_tokens=300,
        num_max_tokens_per_rank=300),
    # expanded blocks aligned to 128 rows with zeroed padding
    "expanded_a128_zero": WORKLOADS["expanded"].replace(
        name="expanded_a128_zero", expert_alignment=128, zero_padding=True, num_tokens=100,
        num_max_tokens_per_rank=100),
}


_HOT_BIAS: dict = {}


def _generator(seed: int, stream: int = 0, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


def _expert_bias(wl: Workload, logits: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    E, K = wl.num_experts, wl.num_topk
    if wl.routing == "gauss":
        return torch.zeros(E)
    if wl.routing == "zipf":
        # rank pi(e) of each expert in a seeded permutation; bias = -s * ln(1 + pi(e))
        pi = torch.randperm(E, generator=g).to(torch.float64)
        return (-wl.zipf_s * torch.log1p(pi)).to(torch.float32)
    if wl.routing == "hot":
        n_hot = math.ceil(wl.hot_expert_frac * E)
        hot = torch.randperm(E, generator=g)[:n_hot]
        is_hot = torch.zeros(E, dtype=torch.bool)
        is_hot[hot] = True
        # scalar bias on the hot experts, bisected on this sample until the hot
        # experts take the requested share of all routed lanes
        if wl not in _HOT_BIAS:
            lo, hi = 0.0, 16.0
            for _ in range(40):
                mid = 0.5 * (lo + hi)
                idx = torch.topk(logits + mid * is_hot, K, dim=-1).indices
                frac = is_hot[idx].float().mean().item()
                if abs(frac - wl.hot_traffic) <= 0.002:
                    break
                if frac < wl.hot_traffic:
                    lo = mid
                else:
                    hi = mid
            _HOT_BIAS[wl] = mid
        return (_HOT_BIAS[wl] * is_hot).to(torch.float32)
    raise ValueError(f"unknown routing {wl.routing!r}")


def routing(wl: Workload):
    """Return (topk_idx int64 [R,T,K], topk_weights fp32 [R,T,K]) on the CPU."""
    R, T, E, K = wl.num_ranks, wl.num_tokens, wl.num_experts, wl.num_topk
    g = _generator(wl.seed)
    logits = torch.randn(R, T, E, generator=g, dtype=torch.float32)
    bias = _expert_bias(wl, logits, g)
    scores = logits + bias
    vals, idx = torch.topk(scores, K, dim=-1)
    w = torch.softmax(vals, dim=-1).to(torch.float32)
    idx = idx.to(torch.int64)
    if wl.mask_frac > 0:
        m = torch.rand(R, T, K, generator=g) < wl.mask_frac
        idx = idx.masked_fill(m, -1)
        w = w.masked_fill(m, 0.0)
    return idx.contiguous(), w.contiguous()


def hidden(wl: Workload):
    """Return the dispatch input.

    bf16 input: (x bf16 [R,T,H], None).
    fp8 input:  (x uint8 e4m3 codes [R,T,H], x_sf fp32 [R,T,H/128]); codes are
    uniform over the finite e4m3 codes, scales uniform in [1e-3, 1.1e-2).
    Drawn after the routing on the same seeded stream.
    """
    R, T, H = wl.num_ranks, wl.num_tokens, wl.hidden
    g = _generator(wl.seed)
    # replay the routing draws so that x follows them on the same stream
    routing_draws(wl, g)
    if wl.x_dtype == "bf16":
        x = torch.empty(R, T, H, dtype=torch.bfloat16)
        for r in range(R):
            x[r] = torch.randn(T, H, generator=g).to(torch.bfloat16)
        return x, None
    codes = torch.randint(0, 256, (R, T, H), generator=g, dtype=torch.int64).to(torch.uint8)
    nan = (codes & 0x7F) == 0x7F
    codes = torch.where(nan, codes ^ 1, codes)
    G = H // 128
    if wl.sf_pack:  # exponent bytes 100..140, four per 32-bit word, zero past the last group
        b = torch.randint(100, 141, (R, T, (G + 3) // 4 * 4), generator=g, dtype=torch.int64)
        b[..., G:] = 0
        words = (b[..., 0::4] | b[..., 1::4] << 8 | b[..., 2::4] << 16 | b[..., 3::4] << 24)
        sf = words.to(torch.int64).to(torch.int32).view(torch.float32)
        return codes.contiguous(), sf.contiguous()
    sf = (torch.rand(R, T, G, generator=g) * 1e-2 + 1e-3).to(torch.float32)
    return codes.contiguous(), sf.contiguous()


def routing_draws(wl: Workload, g: torch.Generator) -> None:
    """Advance ``g`` past the routing draws (same calls as ``routing``)."""
    R, T, E, K = wl.num_ranks, wl.num_tokens, wl.num_experts, wl.num_topk
    logits = torch.randn(R, T, E, generator=g, dtype=torch.float32)
    _expert_bias(wl, logits, g)
    if wl.mask_frac > 0:
        torch.rand(R, T, K, generator=g)


def expert_outputs(wl: Workload, num_rows: int, device: str = "cpu",
                   chunk_rows: int = 1 << 16) -> torch.Tensor:
    """Random bf16(N(0,1)) expert outputs, ``num_rows`` rows of width H.

    Drawn from stream 1 of the workload seed, on ``device`` (the values depend
    on the device's generator); chunked so the fp32 staging stays small.
    """
    H = wl.hidden
    g = _generator(wl.seed, 1, device)
    y = torch.empty(num_rows, H, dtype=torch.bfloat16, device=device)
    for r0 in range(0, num_rows, chunk_rows):
        r1 = min(num_rows, r0 + chunk_rows)
        y[r0:r1] = torch.randn(r1 - r0, H, generator=g, device=device).to(torch.bfloat16)
    return y
