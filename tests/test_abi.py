"""The C-ABI library without a GPU: it loads, exports every entry point that
include/ep_get.h declares, sizes buffers by closed forms, and rejects bad
arguments before touching the device."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    from combine_ep_get_02_gb300 import _build
    _build.build()
    import combine_ep_get_02_gb300 as ep
    ep.lib()
    return ep


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ep_get.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(ep_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_checked_build_exports_the_same_symbols(ep):
    ep._build.build(checked=True)
    names = declared_functions()
    nm = subprocess.run(["nm", "-D", "--defined-only", ep._build.LIB_CHECKED], capture_output=True,
                        text=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)", nm))
    assert set(names) <= exported
    lib = C.CDLL(ep._build.LIB_CHECKED)
    for n in names:
        getattr(lib, n)


def test_every_declared_symbol_is_exported(ep):
    names = declared_functions()
    assert {"ep_get_dispatch_layout", "ep_dispatch", "ep_combine", "ep_workspace_bytes",
            "ep_recv_rows", "ep_check_error", "ep_status_string"} <= set(names)
    lib = C.CDLL(ep._build.LIB)
    for n in names:
        assert hasattr(lib, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", ep._build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (ep_\w+)$", nm, flags=re.M))
    assert set(names) <= exported


def cfg(ep, **kw):
    base = dict(num_scaleout_ranks=1, num_scaleup_ranks=16, num_experts=256, num_topk=8,
                num_tokens=4096, num_max_tokens_per_rank=4096, hidden=7168)
    base.update(kw)
    return ep.Config(**base)


def test_recv_rows_closed_forms(ep):
    # row form: R regions of R*M rows (the per-destination window R*M rows)
    assert ep.ep_recv_rows(cfg(ep)) == 16 * 16 * 4096
    assert ep.ep_recv_rows(cfg(ep, num_scaleout_ranks=4, num_scaleup_ranks=8, num_tokens=2048,
                                num_max_tokens_per_rank=2048)) == 32 * 32 * 2048
    # expanded: every lane plus the worst-case padding of every expert block
    assert ep.ep_recv_rows(cfg(ep, expand=1)) == 16 * 4096 * 8
    assert ep.ep_recv_rows(cfg(ep, expand=1, expert_alignment=128)) == 16 * 4096 * 8 + 256 * 127
    # compact: the same windows; packed: the most rows that can arrive, R*T*min(K, R)
    assert ep.ep_recv_rows(cfg(ep, compact_recv=1)) == 16 * 16 * 4096
    assert ep.ep_recv_rows(cfg(ep, compact_recv=2)) == 16 * 4096 * 8
    assert ep.ep_recv_rows(cfg(ep, compact_recv=2, num_topk=20)) == 16 * 4096 * 16
    assert ep.ep_recv_rows(cfg(ep, compact_recv=2, recv_capacity=1234)) == 1234


def test_workspace_bytes_closed_form(ep):
    # a 256-byte header (device error bits, the layout kernel's arrival counter)
    # plus, expanded, the per-(source, expert) cross-source offsets
    def expect(R, E, expand):
        return 256 + ((4 * R * E + 255) // 256 * 256 if expand else 0)
    assert ep.ep_workspace_bytes(cfg(ep)) == expect(16, 256, False)
    assert ep.ep_workspace_bytes(cfg(ep, expand=1)) == expect(16, 256, True)
    assert ep.ep_workspace_bytes(cfg(ep, num_scaleup_ranks=64, num_experts=512, num_tokens=513,
                                     num_max_tokens_per_rank=600, expand=1)) == expect(64, 512, True)
    assert ep.ep_workspace_bytes(cfg(ep, num_tokens=0)) == 256


@pytest.mark.parametrize("bad,code", [
    (dict(num_scaleup_ranks=0), -1),
    (dict(num_experts=250), -1),              # not a multiple of R
    (dict(num_tokens=5000), -1),              # T > M
    (dict(num_topk=0), -1),
    (dict(num_topk=33), -1),
    (dict(hidden=100), -1),                   # not a multiple of 8
    (dict(hidden=1000, recv_dtype=1), -1),    # FP8 needs a multiple of 128
    (dict(x_dtype=1, recv_dtype=0), -2),      # e4m3 in, bf16 out: not done
    (dict(num_scaleup_ranks=128, num_experts=256), -2),   # more than 64 ranks
    (dict(num_experts=8192), -2),
    (dict(expert_alignment=0), -1),
    (dict(x_dtype=7), -1),
    (dict(compact_recv=3), -1),
    (dict(compact_recv=1, expand=1), -2),     # expanded rows are packed already
    (dict(compact_recv=2, expand=1), -2),
    (dict(recv_capacity=-1, compact_recv=2), -1),
    (dict(recv_capacity=100), -2),            # a capacity only for packed rows
    (dict(zero_padding=1), -2),               # only expanded blocks have padding
    (dict(zero_padding=3, expand=1), -1),
    (dict(sf_pack=1), -2),                    # packed scales need an FP8 receive
    (dict(sf_pack=2, recv_dtype=1), -1),
    (dict(copy_path=3), -1),
    (dict(copy_path=-1), -1),
])
def test_invalid_configs_are_rejected_before_any_launch(ep, bad, code):
    c = cfg(ep, **bad)
    assert ep.ep_workspace_bytes(c) == 0
    assert ep.ep_recv_rows(c) == -1
    cc = c._c()
    lay = ep._Layout()
    st = ep.lib().ep_get_dispatch_layout(C.byref(cc), None, C.byref(lay), None, 0, None)
    assert st == code


def test_noalloc_checks_arguments_before_touching_the_device(ep):
    """The allocation-free layout refuses bad arguments before any CUDA call
    (without a GPU a call that got that far would answer EP_ERR_CUDA), so a
    refused call never writes the library's shared array."""
    L = ep.lib()
    c = cfg(ep)
    cc = c._c()
    lay = ep._Layout()
    assert L.ep_get_dispatch_layout_noalloc(C.byref(cc), C.c_void_p(0x20000), None, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_get_dispatch_layout_noalloc(C.byref(cc), C.c_void_p(0x20000), C.byref(lay), None) == \
        ep.EP_ERR_INVALID_ARG
    bad = cfg(ep, num_experts=250)._c()
    assert L.ep_get_dispatch_layout_noalloc(C.byref(bad), None, C.byref(lay), None) == ep.EP_ERR_INVALID_ARG
    big = cfg(ep, num_scaleup_ranks=64, num_experts=4096, expand=1, num_tokens=16, num_max_tokens_per_rank=16)._c()
    assert L.ep_get_dispatch_layout_noalloc(C.byref(big), None, C.byref(lay), None) == ep.EP_ERR_WORKSPACE


def test_workspace_checks(ep):
    c = cfg(ep)
    cc = c._c()
    lay = ep._Layout()
    L = ep.lib()
    assert L.ep_get_dispatch_layout(C.byref(cc), None, C.byref(lay), None, 1 << 20, None) == ep.EP_ERR_WORKSPACE
    # misaligned workspace, then one that is too small
    assert L.ep_get_dispatch_layout(C.byref(cc), None, C.byref(lay), C.c_void_p(0x1008), 1 << 20, None) == ep.EP_ERR_WORKSPACE
    assert L.ep_get_dispatch_layout(C.byref(cc), None, C.byref(lay), C.c_void_p(0x10000), 16, None) == ep.EP_ERR_WORKSPACE
    # big enough workspace but missing outputs
    n = ep.ep_workspace_bytes(c)
    assert L.ep_get_dispatch_layout(C.byref(cc), C.c_void_p(0x20000), C.byref(lay), C.c_void_p(0x10000), n, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(C.byref(cc), None, None, None, None, None, None, C.c_void_p(0x10000), n, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_combine(C.byref(cc), None, None, None, None, None, C.c_void_p(0x10000), n, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_check_error(None, None) == ep.EP_ERR_WORKSPACE


def test_misaligned_rows_are_rejected(ep):
    c = cfg(ep, num_tokens=16, num_max_tokens_per_rank=16, hidden=256)
    cc = c._c()
    n = ep.ep_workspace_bytes(c)
    ws = C.c_void_p(0x100000)
    lay = ep._Layout(*([C.c_void_p(0x200000)] * 10))
    recv = ep._Recv(C.c_void_p(0x300008), None, None, None, None, ep.ep_recv_rows(c))  # recv_x not 16-aligned
    P = C.c_void_p
    st = ep.lib().ep_dispatch(C.byref(cc), C.byref(lay), P(0x400000), None, P(0x500000), P(0x600000),
                              C.byref(recv), ws, n, None)
    assert st == ep.EP_ERR_INVALID_ARG
    recv = ep._Recv(C.c_void_p(0x300000), None, None, None, None, ep.ep_recv_rows(c) - 1)  # too small
    st = ep.lib().ep_dispatch(C.byref(cc), C.byref(lay), P(0x400000), None, P(0x500000), P(0x600000),
                              C.byref(recv), ws, n, None)
    assert st == ep.EP_ERR_INVALID_ARG
    st = ep.lib().ep_combine(C.byref(cc), C.byref(lay), P(0x400004), P(0x500000), P(0x600000),
                             P(0x700000), ws, n, None)
    assert st == ep.EP_ERR_INVALID_ARG


def test_diag_copy_rejects_bad_arguments(ep):
    L, P = ep.lib(), C.c_void_p
    a, b = P(0x100000), P(0x200000)
    for rows, rb, num, den, sms in ((1, 24, 1, 1, 0), (1, 0, 1, 1, 0), (1, 16, 1, 0, 0), (-1, 16, 1, 1, 0),
                                    (1, 16, -1, 1, 0), (1, 16, (1 << 20) + 1, 1, 0), (1 << 41, 16, 1, 1, 0),
                                    (1, 16, 1, 1, -1)):
        assert L.ep_diag_copy_fanout(a, b, rows, rb, num, den, sms, 0, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_diag_copy_fanout(P(0x100008), b, 1, 16, 1, 1, 0, 0, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_diag_copy_fanout(a, None, 1, 16, 1, 1, 0, 0, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_diag_copy_fanout(a, b, 1, 16, 1, 1, 0, 2, None) == ep.EP_ERR_INVALID_ARG
    # rows wider than one shared-memory stage: no bulk method
    assert L.ep_diag_copy_fanout(a, b, 1, 16400, 1, 1, 0, 1, None) == ep.EP_ERR_UNSUPPORTED
    # nothing to copy: accepted without a launch
    assert L.ep_diag_copy_fanout(None, None, 0, 16, 3, 1, 0, 0, None) == ep.EP_OK
    assert L.ep_diag_copy_fanout(None, None, 5, 16, 0, 1, 0, 1, None) == ep.EP_OK


def test_diag_wait_timeout_rejects_bad_arguments(ep):
    L, P = ep.lib(), C.c_void_p
    ws, src = P(0x100000), P(0x200000)
    assert L.ep_diag_wait_timeout(None, src, 16, 1, None) == ep.EP_ERR_WORKSPACE
    assert L.ep_diag_wait_timeout(P(0x100010), src, 16, 1, None) == ep.EP_ERR_WORKSPACE
    for s, n, r in ((src, 4112, 1), (src, 24, 1), (src, -16, 1), (None, 16, 1), (P(0x200008), 16, 1),
                    (src, 16, (1 << 20) + 1)):
        assert L.ep_diag_wait_timeout(ws, s, n, r, None) == ep.EP_ERR_INVALID_ARG


def test_status_strings(ep):
    assert ep.ep_status_string(0) == "EP_OK"
    assert ep.ep_status_string(-5) == "EP_ERR_BAD_TOPK"
    assert ep.ep_status_string(-7) == "EP_ERR_TIMEOUT"
    assert ep.ep_status_string(-99) == "EP_ERR_UNKNOWN"


def test_product_path_fails_loudly_without_the_library(ep, monkeypatch):
    monkeypatch.setattr(ep, "_lib", None)
    monkeypatch.setattr(ep._build, "LIB", "/nonexistent/libep_get.so")
    with pytest.raises(RuntimeError, match="missing"):
        ep.lib()


def test_kernel_hash_ignores_comments_but_not_code(ep, tmp_path, monkeypatch):
    """The ncu traffic figures are keyed by a hash of each kernel's code; a comment
    edit keeps it, a code edit changes it."""
    b = ep._build
    src = open(os.path.join(b.CSRC, "combine.cu")).read()
    assert b._code_only("int a; // note\n/* block\n comment */int b;\n\n") == "int a;\nint b;"
    base = b._code_only(src)
    assert b._code_only("// a new remark\n" + src.replace("\n", "\n/* x */", 1)) == base
    assert b._code_only(src.replace("kSteps", "kStepz", 1)) != base


def test_status_codes_agree_across_header_library_and_binding(ep):
    text = open(os.path.join(ROOT, "include", "ep_get.h")).read()
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (EP_(?:OK|ERR_\w+))\s+\(?(-?\d+)\)?", text)}
    assert codes["EP_OK"] == 0 and len(codes) >= 9
    for name, value in codes.items():
        assert getattr(ep, name) == value, name          # the binding's constant
        assert ep.ep_status_string(value) == name         # the library's name for it
    assert len(set(codes.values())) == len(codes)
