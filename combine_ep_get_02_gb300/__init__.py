"""GB300-native MoE expert-parallel dispatch / combine on one GPU.

Thin ctypes binding over the C ABI of ``include/ep_get.h`` (``libep_get.so``,
built in-tree for sm_103a). Every step of the path runs in the library's CUDA
kernels; this module only marshals arguments: torch tensors supply device
memory and the current CUDA stream. There is no CPU fallback: if the library
is missing, importing the binding raises.

The entry points keep the C names (``ep_get_dispatch_layout``, ``ep_dispatch``,
``ep_combine``, ...). ``Config`` mirrors ``ep_config_t``; ``alloc_layout``,
``alloc_recv`` and ``alloc_workspace`` allocate correctly sized tensors.
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os

import torch

from . import _build

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_UNSUPPORTED, EP_ERR_WORKSPACE, EP_ERR_CUDA, EP_ERR_BAD_TOPK, \
    EP_ERR_OVERFLOW, EP_ERR_TIMEOUT, EP_ERR_BOUNDS = 0, -1, -2, -3, -4, -5, -6, -7, -8
EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3 = 0, 1

__all__ = [
    "Config", "Layout", "Recv", "EpError", "lib", "ep_workspace_bytes", "ep_recv_rows",
    "ep_workspace_init", "ep_get_dispatch_layout", "ep_get_dispatch_layout_noalloc", "ep_check_error_noalloc",
    "ep_dispatch", "ep_combine", "ep_check_error",
    "ep_dispatch_atomic", "ep_deterministic_sort",
    "ep_status_string", "ep_diag_e4m3_of_bits", "ep_diag_bf16_of_bits",
    "ep_diag_copy_fanout", "ep_diag_wait_timeout", "use_checked", "alloc_layout", "alloc_recv",
    "alloc_workspace", "config_of",
]


class EpError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {ep_status_string(status)} ({status})")
        self.status = status


class _Config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "num_scaleout_ranks", "num_scaleup_ranks", "num_experts", "num_topk", "num_tokens",
        "num_max_tokens_per_rank", "hidden", "x_dtype", "recv_dtype", "expand", "expert_alignment",
        "num_sms", "num_prologue_sms", "compact_recv", "zero_padding", "sf_pack", "copy_path",
        "recv_capacity")]


class _Layout(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "slot_map", "recv_cnt",
        "recv_psum", "exp_cnt", "exp_base", "exp_region", "exp_pos", "recv_region")]


class _Recv(C.Structure):
    _fields_ = [("recv_x", C.c_void_p), ("recv_sf", C.c_void_p), ("recv_topk_idx", C.c_void_p),
                ("recv_topk_weights", C.c_void_p), ("recv_src_metadata", C.c_void_p),
                ("recv_x_rows", C.c_int64)]


class _KeepsStruct:
    """Keeps the ctypes struct built by _c() until a field is assigned again, so
    a call reuses it instead of marshalling every field (the struct holds the
    values, and for tensors their data pointers, as of that build)."""

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        object.__setattr__(self, "_struct", None)

    def _c(self):
        st = self.__dict__.get("_struct")
        if st is None:
            st = self._build_struct()
            object.__setattr__(self, "_struct", st)
        return st


@dataclasses.dataclass
class Config(_KeepsStruct):
    num_scaleout_ranks: int
    num_scaleup_ranks: int
    num_experts: int
    num_topk: int
    num_tokens: int
    num_max_tokens_per_rank: int
    hidden: int
    x_dtype: int = EP_DTYPE_BF16
    recv_dtype: int = EP_DTYPE_BF16
    expand: int = 0
    expert_alignment: int = 1
    num_sms: int = 0
    num_prologue_sms: int = 0
    compact_recv: int = 0
    zero_padding: int = 0
    sf_pack: int = 0
    copy_path: int = 0  # unchanged rows: 0 automatic, 1 register copies, 2 bulk copies
    recv_capacity: int = 0  # packed receive rows: rows of the receive tensors (0 = R*T*min(K,R))

    @property
    def num_ranks(self) -> int:
        return self.num_scaleout_ranks * self.num_scaleup_ranks

    def _build_struct(self) -> _Config:
        return _Config(*(int(getattr(self, f[0])) for f in _Config._fields_))


def config_of(wl, **over) -> Config:
    """Config of a workload description (attributes as in ``workloads.Workload``)."""
    c = Config(wl.n_so, wl.n_su, wl.num_experts, wl.num_topk, wl.num_tokens,
               wl.num_max_tokens_per_rank, wl.hidden,
               EP_DTYPE_FP8_E4M3 if wl.x_dtype == "fp8" else EP_DTYPE_BF16,
               EP_DTYPE_FP8_E4M3 if wl.recv_dtype == "fp8" else EP_DTYPE_BF16,
               int(bool(wl.expand)), wl.expert_alignment,
               compact_recv=int(getattr(wl, "compact", 0)),
               recv_capacity=int(getattr(wl, "recv_capacity", 0)),
               zero_padding=int(bool(getattr(wl, "zero_padding", False))),
               sf_pack=int(bool(getattr(wl, "sf_pack", False))))
    return dataclasses.replace(c, **over)


_lib = None
_checked = False


def use_checked(on: bool = True) -> None:
    """Route every later call to the bounds-checked build of the library (each
    computed row index is tested against its buffer; one outside is skipped and
    reported as EP_ERR_BOUNDS by ep_check_error), or back to the normal one."""
    global _lib, _checked
    _checked, _lib = bool(on), None


def lib():
    """The loaded library. Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        path = _build.LIB_CHECKED if _checked else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(path)
        P, I = C.c_void_p, C.c_int
        L.ep_workspace_bytes.restype = C.c_size_t
        L.ep_workspace_bytes.argtypes = [P]
        L.ep_recv_rows.restype = C.c_int64
        L.ep_recv_rows.argtypes = [P]
        L.ep_workspace_init.restype = I
        L.ep_workspace_init.argtypes = [P, C.c_size_t, P]
        L.ep_get_dispatch_layout.restype = I
        L.ep_get_dispatch_layout.argtypes = [P, P, P, P, C.c_size_t, P]
        L.ep_get_dispatch_layout_noalloc.restype = I
        L.ep_get_dispatch_layout_noalloc.argtypes = [P, P, P, P]
        L.ep_check_error_noalloc.restype = I
        L.ep_check_error_noalloc.argtypes = [P]
        L.ep_dispatch.restype = I
        L.ep_dispatch.argtypes = [P, P, P, P, P, P, P, P, C.c_size_t, P]
        L.ep_dispatch_atomic.restype = I
        L.ep_dispatch_atomic.argtypes = [P, P, P, P, P, P, P, P, C.c_size_t, P]
        L.ep_deterministic_sort.restype = I
        L.ep_deterministic_sort.argtypes = [P, P, P, P, P]
        L.ep_combine.restype = I
        L.ep_combine.argtypes = [P, P, P, P, P, P, P, C.c_size_t, P]
        L.ep_check_error.restype = I
        L.ep_check_error.argtypes = [P, P]
        L.ep_status_string.restype = C.c_char_p
        L.ep_status_string.argtypes = [I]
        L.ep_diag_e4m3_of_bits.restype = I
        L.ep_diag_e4m3_of_bits.argtypes = [C.c_uint32, C.c_int64, P, P]
        L.ep_diag_bf16_of_bits.restype = I
        L.ep_diag_bf16_of_bits.argtypes = [C.c_uint32, C.c_int64, P, P]
        L.ep_diag_copy_fanout.restype = I
        L.ep_diag_copy_fanout.argtypes = [P, P, C.c_int64, I, I, I, I, I, P]
        L.ep_diag_wait_timeout.restype = I
        L.ep_diag_wait_timeout.argtypes = [P, P, I, C.c_uint32, P]
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, where: str):
    if st != EP_OK:
        raise EpError(st, where)


def ep_status_string(status: int) -> str:
    return lib().ep_status_string(int(status)).decode()


def ep_workspace_bytes(cfg: Config) -> int:
    c = cfg._c()
    return int(lib().ep_workspace_bytes(C.byref(c)))


def ep_recv_rows(cfg: Config) -> int:
    c = cfg._c()
    return int(lib().ep_recv_rows(C.byref(c)))


def ep_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().ep_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "ep_workspace_init")


@dataclasses.dataclass
class Layout(_KeepsStruct):
    num_tokens_per_rank: torch.Tensor
    num_tokens_per_expert: torch.Tensor
    is_token_in_rank: torch.Tensor
    slot_map: torch.Tensor
    recv_cnt: torch.Tensor
    recv_psum: torch.Tensor
    exp_cnt: torch.Tensor | None = None
    exp_base: torch.Tensor | None = None
    exp_region: torch.Tensor | None = None
    exp_pos: torch.Tensor | None = None
    recv_region: torch.Tensor | None = None

    def _build_struct(self) -> _Layout:
        return _Layout(*(_ptr(getattr(self, f[0])) for f in _Layout._fields_))


@dataclasses.dataclass
class Recv(_KeepsStruct):
    recv_x: torch.Tensor
    recv_sf: torch.Tensor | None
    recv_topk_idx: torch.Tensor | None
    recv_topk_weights: torch.Tensor | None
    recv_src_metadata: torch.Tensor | None

    def _build_struct(self) -> _Recv:
        return _Recv(_ptr(self.recv_x), _ptr(self.recv_sf), _ptr(self.recv_topk_idx),
                     _ptr(self.recv_topk_weights), _ptr(self.recv_src_metadata), self.recv_x.shape[0])


def alloc_workspace(cfg: Config, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of ep_workspace_bytes(cfg) bytes."""
    n = ep_workspace_bytes(cfg)
    if n == 0:
        raise EpError(EP_ERR_INVALID_ARG, "ep_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def alloc_layout(cfg: Config, device="cuda") -> Layout:
    R, E, T, K = cfg.num_ranks, cfg.num_experts, cfg.num_tokens, cfg.num_topk
    L = E // R
    i32 = dict(dtype=torch.int32, device=device)
    lay = Layout(torch.empty(R, R, **i32), torch.empty(R, E, **i32),
                 torch.empty(R, T, R, dtype=torch.uint8, device=device), torch.empty(R, T, K, **i32),
                 torch.empty(R, R, **i32), torch.empty(R, R, **i32), recv_region=torch.empty(R + 1, **i32))
    if cfg.expand:
        lay.exp_cnt = torch.empty(R, L, **i32)
        lay.exp_base = torch.empty(R, L + 1, **i32)
        lay.exp_region = torch.empty(R + 1, **i32)
        lay.exp_pos = torch.empty(R, T, K, **i32)
    return lay


def alloc_recv(cfg: Config, device="cuda", sidecars: bool = True, zero: bool = False) -> Recv:
    R, M, K, H = cfg.num_ranks, cfg.num_max_tokens_per_rank, cfg.num_topk, cfg.hidden
    rows = ep_recv_rows(cfg)
    if rows < 0:
        raise EpError(EP_ERR_INVALID_ARG, "ep_recv_rows")
    mk = torch.zeros if zero else torch.empty
    fp8 = cfg.recv_dtype == EP_DTYPE_FP8_E4M3
    recv_x = mk(rows, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=device)
    G = H // 128
    recv_sf = mk(rows, (G + 3) // 4 if cfg.sf_pack else G, dtype=torch.float32, device=device) if fp8 else None
    if not sidecars:
        return Recv(recv_x, recv_sf, None, None, None)
    # sidecar rows: one region of R*M rows per destination, or the packed rows
    side = (rows,) if cfg.compact_recv == 2 else (R, R * M)
    return Recv(recv_x, recv_sf, mk(*side, K, dtype=torch.int64, device=device),
                mk(*side, K, dtype=torch.float32, device=device),
                mk(*side, K + 2, dtype=torch.int32, device=device))


def ep_get_dispatch_layout(cfg: Config, topk_idx: torch.Tensor, layout: Layout, ws: torch.Tensor,
                           stream=None):
    c, l = cfg._c(), layout._c()
    _check(lib().ep_get_dispatch_layout(C.byref(c), _ptr(topk_idx), C.byref(l), _ptr(ws),
                                        ws.numel(), _stream(stream)), "ep_get_dispatch_layout")


def ep_get_dispatch_layout_noalloc(cfg: Config, topk_idx: torch.Tensor, layout: Layout, stream=None):
    """The layout without a caller workspace (fixed scratch inside the library)."""
    c, l = cfg._c(), layout._c()
    _check(lib().ep_get_dispatch_layout_noalloc(C.byref(c), _ptr(topk_idx), C.byref(l), _stream(stream)),
           "ep_get_dispatch_layout_noalloc")


def ep_check_error_noalloc(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the status the
    allocation-free layout latched in the library's array."""
    return int(lib().ep_check_error_noalloc(_stream(stream)))


def ep_dispatch(cfg: Config, layout: Layout, x: torch.Tensor, x_sf, topk_idx: torch.Tensor,
                topk_weights: torch.Tensor, recv: Recv, ws: torch.Tensor, stream=None):
    c, l, r = cfg._c(), layout._c(), recv._c()
    _check(lib().ep_dispatch(C.byref(c), C.byref(l), _ptr(x), _ptr(x_sf), _ptr(topk_idx),
                             _ptr(topk_weights), C.byref(r), _ptr(ws), ws.numel(), _stream(stream)),
           "ep_dispatch")


def ep_dispatch_atomic(cfg: Config, x: torch.Tensor, x_sf, topk_idx: torch.Tensor,
                       topk_weights: torch.Tensor, recv: Recv, send_counters: torch.Tensor, ws: torch.Tensor,
                       stream=None):
    """Comparison path: dispatch with racing atomicAdd slots (no layout)."""
    c, r = cfg._c(), recv._c()
    _check(lib().ep_dispatch_atomic(C.byref(c), _ptr(x), _ptr(x_sf), _ptr(topk_idx), _ptr(topk_weights),
                                    C.byref(r), _ptr(send_counters), _ptr(ws), ws.numel(), _stream(stream)),
           "ep_dispatch_atomic")


def ep_deterministic_sort(cfg: Config, recv: Recv, send_counters: torch.Tensor, sorted_recv: Recv,
                          stream=None):
    """Comparison path: sort each received segment by source token into sorted_recv."""
    c, r, o = cfg._c(), recv._c(), sorted_recv._c()
    _check(lib().ep_deterministic_sort(C.byref(c), C.byref(r), _ptr(send_counters), C.byref(o),
                                       _stream(stream)), "ep_deterministic_sort")


def ep_combine(cfg: Config, layout: Layout, y: torch.Tensor, topk_idx: torch.Tensor,
               topk_weights: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, stream=None):
    c, l = cfg._c(), layout._c()
    _check(lib().ep_combine(C.byref(c), C.byref(l), _ptr(y), _ptr(topk_idx), _ptr(topk_weights),
                            _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "ep_combine")


def ep_check_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the latched device status."""
    return int(lib().ep_check_error(_ptr(ws), _stream(stream)))


def ep_diag_e4m3_of_bits(first: int, out: torch.Tensor, stream=None):
    _check(lib().ep_diag_e4m3_of_bits(first, out.numel(), _ptr(out), _stream(stream)),
           "ep_diag_e4m3_of_bits")


def ep_diag_bf16_of_bits(first: int, out: torch.Tensor, stream=None):
    _check(lib().ep_diag_bf16_of_bits(first, out.numel(), _ptr(out), _stream(stream)),
           "ep_diag_bf16_of_bits")


def ep_diag_copy_fanout(src: torch.Tensor, dst: torch.Tensor, rows: int, row_bytes: int, fan_num: int,
                        fan_den: int, num_sms: int = 0, method: int = 0, stream=None):
    """Row r of src goes to dst rows floor(r*num/den) .. floor((r+1)*num/den)-1;
    method 0: register loads/stores, 1: bulk copies through shared memory."""
    need = rows * fan_num // fan_den * row_bytes if fan_den > 0 else 0
    if src.numel() * src.element_size() < rows * row_bytes or dst.numel() * dst.element_size() < need:
        raise EpError(EP_ERR_INVALID_ARG, "ep_diag_copy_fanout")
    _check(lib().ep_diag_copy_fanout(_ptr(src), _ptr(dst), rows, row_bytes, fan_num, fan_den, num_sms,
                                     method, _stream(stream)), "ep_diag_copy_fanout")


def ep_diag_wait_timeout(ws: torch.Tensor, src, nbytes: int, rounds: int, stream=None):
    """Run the bulk-copy dispatch's abort sequence: a wait that runs out after
    `rounds` rounds with a load of `nbytes` from `src` in flight."""
    _check(lib().ep_diag_wait_timeout(_ptr(ws), _ptr(src), nbytes, rounds,
                                      _stream(stream)), "ep_diag_wait_timeout")
