"""Write the stored layout fixtures of this folder.

Calls only the CPU oracle (``oracle/``) and numpy's seeded generator. Each
fixture holds a small routing and the oracle's layout of it; the slot rule
followed is PR #753 (Approach; "Direct vs hybrid dispatch"), the expanded
positions the (source rank, token) order of the per-expert blocks. The tests
re-derive every fixture from the oracle (drift check) and compare the GPU
layout with it.

usage: python tests/golden/make_golden.py
"""
import json
import os
import sys
from types import SimpleNamespace

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CASES = [
    # name, n_so, n_su, E, K, T, M, expand, align, mask_frac, seed
    ("direct_r4_e8_k3_t10", 1, 4, 8, 3, 10, 12, False, 1, 0.15, 11),
    ("hybrid_2x2_e8_k2_t9", 2, 2, 8, 2, 9, 9, False, 1, 0.1, 12),
    ("expanded_r4_e16_k3_t8_a4", 1, 4, 16, 3, 8, 8, True, 4, 0.1, 13),
]


def case_wl(c):
    name, n_so, n_su, E, K, T, M, expand, align, _, _ = c
    return SimpleNamespace(n_so=n_so, n_su=n_su, num_ranks=n_so * n_su, num_experts=E, num_topk=K,
                           num_tokens=T, num_max_tokens_per_rank=M, hidden=128, x_dtype="bf16",
                           recv_dtype="bf16", expand=expand, expert_alignment=align)


def case_idx(c):
    name, n_so, n_su, E, K, T, M, expand, align, mask, seed = c
    rng = np.random.default_rng(seed)
    R = n_so * n_su
    idx = np.stack([[rng.choice(E, K, replace=False) for _ in range(T)] for _ in range(R)]).astype(np.int64)
    idx[rng.random(idx.shape) < mask] = -1
    return idx


def main():
    for c in CASES:
        wl = case_wl(c)
        idx = case_idx(c)
        st, lay = oracle.layout(wl, idx)
        assert st == 0
        doc = {"case": c[0], "source": "written by tests/golden/make_golden.py from the CPU oracle",
               "citation": "PR #753 Approach and 'Direct vs hybrid dispatch' (slot rule, row bases)",
               "config": {k: getattr(wl, k) for k in ("n_so", "n_su", "num_experts", "num_topk", "num_tokens",
                                                      "num_max_tokens_per_rank", "expand", "expert_alignment")},
               "topk_idx": idx.tolist()}
        doc.update({k: v.tolist() for k, v in lay.items()})
        with open(os.path.join(HERE, c[0] + ".json"), "w") as f:
            json.dump(doc, f, separators=(",", ":"))
            f.write("\n")


if __name__ == "__main__":
    main()
