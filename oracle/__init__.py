"""CPU oracle for MoE token dispatch / combine: numpy front end.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the product
path never does. It shares no code with the CUDA library: the arithmetic lives
in ``ep_oracle.cpp`` (plain single-threaded C++), this file only marshals numpy
arrays (the row of every lane in the receive tensors, too, comes from the C++
side: ``lane_rows``). Which passage of the DeepEP pages each function follows is
stated in ``ep_oracle.cpp``.

A workload is any object with the attributes ``n_so, n_su, num_experts,
num_topk, num_tokens, num_max_tokens_per_rank, hidden, x_dtype, recv_dtype,
expand, expert_alignment`` (and optionally ``compact`` 0/1/2, ``zero_padding``,
``sf_pack``, ``recv_capacity``).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

OK, INVALID, UNSUPPORTED, BAD_TOPK, OVERFLOW = 0, -1, -2, -5, -6


class _Cfg(C.Structure):
    _fields_ = [(n, C.c_int32) for n in
                ("n_so", "n_su", "E", "K", "T", "M", "H", "x_fp8", "recv_fp8", "expand", "align",
                 "compact", "zero_padding", "sf_pack", "recv_capacity")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.orc_bf16_to_f32.restype = C.c_float
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_f32_to_bf16.restype = C.c_uint16
        L.orc_f32_to_bf16.argtypes = [C.c_float]
        L.orc_e4m3_to_f32.restype = C.c_float
        L.orc_e4m3_to_f32.argtypes = [C.c_uint8]
        L.orc_f32_to_e4m3.restype = C.c_uint8
        L.orc_f32_to_e4m3.argtypes = [C.c_float]
        L.orc_f32_to_bf16_n.argtypes = [P, P, C.c_int64]
        L.orc_f32_to_e4m3_n.argtypes = [P, P, C.c_int64]
        L.orc_e4m3_of_bits.argtypes = [C.c_uint32, C.c_int64, P]
        L.orc_bf16_of_bits.argtypes = [C.c_uint32, C.c_int64, P]
        L.orc_cast_row_fp8.argtypes = [P, C.c_int, P, P]
        L.orc_cast_row_fp8_ue8m0.argtypes = [P, C.c_int, P, P]
        L.orc_recv_rows.restype = C.c_int64
        L.orc_recv_rows.argtypes = [P]
        L.orc_sidecar_rows.restype = C.c_int64
        L.orc_sidecar_rows.argtypes = [P]
        L.orc_layout.restype = C.c_int
        L.orc_layout.argtypes = [P] * 13
        L.orc_dispatch_token.restype = C.c_int
        L.orc_dispatch_token.argtypes = [P, C.c_int, C.c_int] + [P] * 18
        L.orc_dispatch.restype = C.c_int
        L.orc_dispatch.argtypes = [P] * 17
        L.orc_lane_rows.restype = C.c_int
        L.orc_lane_rows.argtypes = [P] * 9
        L.orc_combine_token.restype = None
        L.orc_combine_token.argtypes = [C.c_int, C.c_int, P, P, P]
        L.orc_combine_gathered.restype = None
        L.orc_combine_gathered.argtypes = [C.c_int, C.c_int, C.c_int64, P, P, P, P]
        L.orc_combine.restype = C.c_int
        L.orc_combine.argtypes = [P] * 10
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def cfg_of(wl) -> _Cfg:
    return _Cfg(wl.n_so, wl.n_su, wl.num_experts, wl.num_topk, wl.num_tokens,
                wl.num_max_tokens_per_rank, wl.hidden, int(wl.x_dtype == "fp8"),
                int(wl.recv_dtype == "fp8"), int(bool(wl.expand)), wl.expert_alignment,
                int(getattr(wl, "compact", 0)),
                int(bool(getattr(wl, "zero_padding", False))),
                int(bool(getattr(wl, "sf_pack", False))),
                int(getattr(wl, "recv_capacity", 0)))


def _np(a, dtype):
    """C-contiguous numpy array of ``dtype`` from a CPU torch tensor or array-like.
    Integer arrays of the same width are reinterpreted (bf16 bits as uint16)."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().cpu().contiguous()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    dt = np.dtype(dtype)
    if a.dtype != dt:
        if a.dtype.kind in "iu" and dt.kind in "iu" and a.dtype.itemsize == dt.itemsize:
            a = a.view(dt)
        else:
            a = a.astype(dt)
    return a


# ---- number formats --------------------------------------------------------

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_n(_p(x), _p(out), x.size)
    return out


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().orc_f32_to_e4m3_n(_p(x), _p(out), x.size)
    return out


def e4m3_to_f32(codes: np.ndarray) -> np.ndarray:
    f = lib().orc_e4m3_to_f32
    table = np.array([f(c) for c in range(256)], dtype=np.float32)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_of_bits(first: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint8)
    lib().orc_e4m3_of_bits(first, n, _p(out))
    return out


def bf16_of_bits(first: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint16)
    lib().orc_bf16_of_bits(first, n, _p(out))
    return out


def sf_words(wl) -> int:
    """32-bit words of one row's scale sidecar: G fp32 scales, or ceil(G/4) packed words."""
    G = wl.hidden // 128
    return (G + 3) // 4 if getattr(wl, "sf_pack", False) else G


def cast_row_fp8_ue8m0(x_bits: np.ndarray):
    """Packed-exponent FP8 cast of one bf16 row: (codes uint8 [H], words uint32 [ceil(G/4)])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x.size
    q = np.empty(H, np.uint8)
    words = np.empty((H // 128 + 3) // 4, np.uint32)
    lib().orc_cast_row_fp8_ue8m0(_p(x), H, _p(q), _p(words))
    return q, words


def cast_row_fp8(x_bits: np.ndarray):
    """FP8 cast of one bf16 row (given as uint16 bits): (codes uint8 [H], sf fp32 [H/128])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x.size
    q = np.empty(H, np.uint8)
    sf = np.empty(H // 128, np.float32)
    lib().orc_cast_row_fp8(_p(x), H, _p(q), _p(sf))
    return q, sf


# ---- the path ----------------------------------------------------------------

def recv_rows(wl) -> int:
    """Rows of recv_x (and recv_sf)."""
    c = cfg_of(wl)
    return int(lib().orc_recv_rows(C.byref(c)))


def sidecar_rows(wl) -> int:
    """Rows of the sidecar tensors (recv_topk_idx, recv_topk_weights, recv_src_metadata)."""
    c = cfg_of(wl)
    return int(lib().orc_sidecar_rows(C.byref(c)))


def layout(wl, topk_idx):
    """Dispatch layout of ``topk_idx`` [R,T,K] int64. Returns (status, dict of arrays)."""
    c = cfg_of(wl)
    R, E, T, K = wl.num_ranks, wl.num_experts, wl.num_tokens, wl.num_topk
    L = E // R
    idx = _np(topk_idx, np.int64).reshape(R, T, K)
    out = dict(
        num_tokens_per_rank=np.zeros((R, R), np.int32),
        num_tokens_per_expert=np.zeros((R, E), np.int32),
        is_token_in_rank=np.zeros((R, T, R), np.uint8),
        slot_map=np.zeros((R, T, K), np.int32),
        recv_cnt=np.zeros((R, R), np.int32),
        recv_psum=np.zeros((R, R), np.int32),
        recv_region=np.zeros(R + 1, np.int32),
    )
    if wl.expand:
        out.update(exp_cnt=np.zeros((R, L), np.int32), exp_base=np.zeros((R, L + 1), np.int32),
                   exp_region=np.zeros(R + 1, np.int32), exp_pos=np.zeros((R, T, K), np.int32))
    st = lib().orc_layout(C.byref(c), _p(idx), *(_p(out[k]) for k in (
        "num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "slot_map",
        "recv_cnt", "recv_psum", "recv_region")), *(_p(out.get(k)) for k in (
        "exp_cnt", "exp_base", "exp_region", "exp_pos")))
    return st, out


def dispatch_token(wl, lay, s, t, x_row, x_sf_row, idx_tok, w_tok):
    """Receive rows of source token (s, t). Returns a dict:
    hid (received row: uint16 bf16 bits or uint8 e4m3 codes), hid_sf,
    hid_dst/hid_row (destinations of the hidden row and its rows of recv_x),
    meta_dst/meta_row (deduplicated entries: destination and row of the
    sidecar tensors) and the sidecar rows meta_idx [n,K], meta_w [n,K],
    meta_md [n,2+K]."""
    c = cfg_of(wl)
    K, H = wl.num_topk, wl.hidden
    G = H // 128
    fp8_in = wl.x_dtype == "fp8"
    fp8_out = wl.recv_dtype == "fp8"
    xr = np.ascontiguousarray(x_row, dtype=np.uint8 if fp8_in else np.uint16)
    sfr = None if x_sf_row is None else np.ascontiguousarray(x_sf_row, dtype=np.float32)
    hid = np.zeros(H * 2, np.uint8)
    hid_sf = np.zeros(max(G, 1), np.float32)
    SW = sf_words(wl)
    hid_dst = np.zeros(K, np.int32)
    hid_row = np.zeros(K, np.int64)
    meta_dst = np.zeros(K, np.int32)
    meta_row = np.zeros(K, np.int64)
    meta_idx = np.zeros((K, K), np.int64)
    meta_w = np.zeros((K, K), np.float32)
    meta_md = np.zeros((K, 2 + K), np.int32)
    slot = np.ascontiguousarray(lay["slot_map"][s, t], dtype=np.int32)
    pos = np.ascontiguousarray(lay["exp_pos"][s, t], dtype=np.int32) if wl.expand else None
    n = lib().orc_dispatch_token(
        C.byref(c), s, t, _p(slot), _p(pos), _p(lay["recv_psum"]), _p(lay["recv_region"]),
        _p(lay.get("exp_region")), _p(xr), _p(sfr),
        _p(np.ascontiguousarray(idx_tok, dtype=np.int64)),
        _p(np.ascontiguousarray(w_tok, dtype=np.float32)), _p(hid), _p(hid_sf), _p(hid_dst),
        _p(hid_row), _p(meta_dst), _p(meta_row), _p(meta_idx), _p(meta_w), _p(meta_md))
    n_hid, n_meta = n & 0xFF, n >> 8
    hid = hid[:H] if fp8_out else hid.view(np.uint16)[:H]
    return dict(hid=hid, hid_sf=hid_sf[:SW] if fp8_out else None,
                hid_dst=hid_dst[:n_hid], hid_row=hid_row[:n_hid],
                meta_dst=meta_dst[:n_meta], meta_row=meta_row[:n_meta],
                meta_idx=meta_idx[:n_meta], meta_w=meta_w[:n_meta], meta_md=meta_md[:n_meta])


def dispatch(wl, lay, x, x_sf, topk_idx, topk_weights, fill=0):
    """Full dispatch. Returns (status, dict): recv_x [rows, H] (uint16 bf16 bits or
    uint8 e4m3 codes), recv_sf [rows, G] or None, and the sidecars
    recv_topk_idx [S, K], recv_topk_weights [S, K], recv_src_metadata [S, 2+K]
    with S = sidecar_rows(wl). Rows that no entry fills keep the byte value
    `fill` in every tensor."""
    c = cfg_of(wl)
    K, H = wl.num_topk, wl.hidden
    rows = recv_rows(wl)
    S = sidecar_rows(wl)
    fp8_in = wl.x_dtype == "fp8"
    fp8_out = wl.recv_dtype == "fp8"
    xa = _np(x, np.uint8 if fp8_in else np.uint16)
    sfa = None if x_sf is None else _np(x_sf, np.float32)
    SW = sf_words(wl)
    out = dict(
        recv_x=np.full((rows, H * (1 if fp8_out else 2)), fill, np.uint8).view(np.uint8 if fp8_out else np.uint16),
        recv_sf=np.full((rows, SW * 4), fill, np.uint8).view(np.float32) if fp8_out else None,
        recv_topk_idx=np.full((S, K * 8), fill, np.uint8).view(np.int64),
        recv_topk_weights=np.full((S, K * 4), fill, np.uint8).view(np.float32),
        recv_src_metadata=np.full((S, (2 + K) * 4), fill, np.uint8).view(np.int32),
    )
    st = lib().orc_dispatch(
        C.byref(c), _p(lay["slot_map"]), _p(lay.get("exp_pos")), _p(lay.get("exp_region")),
        _p(lay.get("exp_cnt")), _p(lay.get("exp_base")), _p(lay["recv_psum"]), _p(lay["recv_region"]),
        _p(xa), _p(sfa), _p(_np(topk_idx, np.int64)), _p(_np(topk_weights, np.float32)),
        _p(out["recv_x"]), _p(out["recv_sf"]), _p(out["recv_topk_idx"]),
        _p(out["recv_topk_weights"]), _p(out["recv_src_metadata"]))
    return st, out


def combine_token(rows, w):
    """Weighted reduction of one token. ``rows``: list of K uint16 bf16 rows or None."""
    K = len(rows)
    H = next((r.size for r in rows if r is not None), 0)
    keep = [None if r is None else np.ascontiguousarray(r, dtype=np.uint16) for r in rows]
    ptrs = (C.c_void_p * K)(*[None if r is None else r.ctypes.data for r in keep])
    out = np.zeros(H, np.uint16)
    lib().orc_combine_token(K, H, ptrs, _p(np.ascontiguousarray(w, dtype=np.float32)), _p(out))
    return out


def combine_gathered(lane_rows, y, w):
    """Combine of n tokens: lane_rows [n, K] int64 rows of y (bf16 bits [rows, H]),
    -1 for masked lanes; w [n, K] fp32. Returns uint16 [n, H]."""
    lane_rows = np.ascontiguousarray(lane_rows, dtype=np.int64)
    n, K = lane_rows.shape
    ya = _np(y, np.uint16)
    H = ya.shape[-1]
    out = np.zeros((n, H), np.uint16)
    lib().orc_combine_gathered(K, H, n, _p(lane_rows), _p(ya), _p(_np(w, np.float32)), _p(out))
    return out


def lane_rows(wl, lay, topk_idx):
    """Row of every top-k lane in the receive tensors, from the C++ oracle.
    Returns (status, hid int64 [R,T,K], side int64 [R,T,K]): the recv_x row the
    lane's expert reads (its deduplicated entry's row, or its expanded row) and
    the sidecar row of its deduplicated entry; -1 for masked lanes (and, packed,
    for entries past the capacity)."""
    c = cfg_of(wl)
    R, T, K = wl.num_ranks, wl.num_tokens, wl.num_topk
    hid = np.empty((R, T, K), np.int64)
    side = np.empty((R, T, K), np.int64)
    st = lib().orc_lane_rows(C.byref(c), _p(_np(topk_idx, np.int64)), _p(lay["slot_map"]),
                             _p(lay.get("exp_pos")), _p(lay.get("exp_region")), _p(lay["recv_psum"]),
                             _p(lay["recv_region"]), _p(hid), _p(side))
    return st, hid, side


def global_rows(wl, lay, topk_idx):
    """The recv_x row of every lane (``lane_rows``' first array): int64 [R,T,K]."""
    return lane_rows(wl, lay, topk_idx)[1]


def combine(wl, lay, y, topk_idx, topk_weights):
    """Full combine of expert outputs ``y`` [rows, H] (bf16 bits, receive layout).
    Returns (status, out uint16 [R, T, H])."""
    c = cfg_of(wl)
    R, T, H = wl.num_ranks, wl.num_tokens, wl.hidden
    ya = _np(y, np.uint16)
    out = np.zeros((R, T, H), np.uint16)
    st = lib().orc_combine(C.byref(c), _p(lay["slot_map"]), _p(lay.get("exp_pos")),
                           _p(lay.get("exp_region")), _p(lay["recv_psum"]), _p(lay["recv_region"]), _p(ya),
                           _p(_np(topk_idx, np.int64)),
                           _p(_np(topk_weights, np.float32)), _p(out))
    return st, out
